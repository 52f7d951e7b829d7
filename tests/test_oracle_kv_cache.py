"""Pins for the paged-cache append references (CPU only).

``append_logical`` is the definition (a sequence's cache grows by its new
tokens; other sequences' caches do not change).  ``BlockManagerRef`` is the
sequential copy-on-write bookkeeping; it is pinned by simulating the data
movement it prescribes on a physical pool and reading every sequence back
through its table: the result must equal the logical definition, and the
reference counts must equal the table references.
"""

import numpy as np
import pytest

import oracle


def test_append_logical_definition():
    rng = np.random.default_rng(0)
    ks = [rng.standard_normal((n, 2, 4)) for n in (3, 0, 17)]
    vs = [rng.standard_normal((n, 2, 4)) for n in (3, 0, 17)]
    kn = rng.standard_normal((3, 5, 2, 4))
    vn = rng.standard_normal((3, 5, 2, 4))
    k2, v2 = oracle.append_logical(ks, vs, kn, vn)
    for s in range(3):
        n = ks[s].shape[0]
        assert k2[s].shape == (n + 5, 2, 4)
        assert np.array_equal(k2[s][:n], ks[s]) and np.array_equal(k2[s][n:], kn[s])
        assert np.array_equal(v2[s][:n], vs[s]) and np.array_equal(v2[s][n:], vn[s])


def _forked_pool(rng, lens, share_groups, num_blocks, Hkv=2, d=4, bs=16):
    """Pool where each group of sequences shares all blocks of its first
    member's prefix (fork after the prefix), including a partial last block."""
    pool = np.full((num_blocks, Hkv, bs, d), np.nan)
    free = list(range(num_blocks))[::-1]
    tables, logical = [], []
    for group in share_groups:
        n = lens[group[0]]
        blocks = [free.pop() for _ in range((n + bs - 1) // bs)]
        data = rng.standard_normal((n, Hkv, d))
        for t in range(n):
            pool[blocks[t // bs], :, t % bs] = data[t]
        for s in group:
            assert lens[s] == n
            tables.append(list(blocks))
            logical.append(data.copy())
    return pool, tables, logical, free


def _apply(mgr, pool, k_new, T):
    """Replay the manager's decisions on a numpy pool (copies, then writes)."""
    for s in range(len(mgr.tables)):
        done = len(mgr.copies)
        slots = mgr.append(s, T)
        for src, dst in mgr.copies[done:]:
            pool[dst] = pool[src]
        for t, (blk, off) in enumerate(slots):
            pool[blk, :, off] = k_new[s, t]


@pytest.mark.parametrize("T", [1, 3, 16, 20])
def test_block_manager_matches_logical_append(T):
    rng = np.random.default_rng(T)
    lens = [21, 21, 21, 32, 32, 5]
    groups = [(0, 1, 2), (3, 4), (5,)]
    pool, tables, logical, free = _forked_pool(rng, lens, groups, 64)
    mgr = oracle.BlockManagerRef(tables, lens, 64, free)
    free_before = len(mgr.free)
    k_new = rng.standard_normal((6, T, 2, 4))
    _apply(mgr, pool, k_new, T)
    want, _ = oracle.append_logical(logical, logical, k_new, k_new)
    for s in range(6):
        n = mgr.lens[s]
        assert n == lens[s] + T
        got = np.stack([pool[mgr.tables[s][t // 16], :, t % 16] for t in range(n)])
        assert np.array_equal(got, want[s])
    # reference counts equal table references; written blocks are private
    refs = np.zeros(64, dtype=np.int64)
    for t, n in zip(mgr.tables, mgr.lens):
        for b in t[:(n + 15) // 16]:
            refs[b] += 1
    assert np.array_equal(refs, mgr.ref)
    for s in range(6):
        last = mgr.tables[s][(mgr.lens[s] - 1) // 16]
        assert mgr.ref[last] == 1
    # blocks taken = copies + blocks opened by the new tokens
    opened = sum((lens[s] + T + 15) // 16 - (lens[s] + 15) // 16 for s in range(6))
    assert free_before - len(mgr.free) == len(mgr.copies) + opened


def test_copy_on_write_counts_for_a_three_way_fork():
    # Three sequences share a partial block: the first two copy it, the last
    # one (now its only holder) writes in place.
    rng = np.random.default_rng(1)
    pool, tables, logical, free = _forked_pool(rng, [21, 21, 21], [(0, 1, 2)], 16)
    mgr = oracle.BlockManagerRef(tables, [21, 21, 21], 16, free)
    shared = tables[0][1]
    _apply(mgr, pool, rng.standard_normal((3, 1, 2, 4)), 1)
    assert [src for src, _ in mgr.copies] == [shared, shared]
    assert mgr.tables[2][1] == shared and mgr.ref[shared] == 1
    assert mgr.tables[0][0] == mgr.tables[1][0] == mgr.tables[2][0]  # full block stays shared
