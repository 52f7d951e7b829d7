"""GPU checks of kv_append (C ABI): paged-cache append with copy-on-write.

Two references from ``oracle.kv_cache``:
* the logical definition (``append_logical``): read back through the
  GPU-updated block table, every sequence's cache must equal its old cache
  followed by its new tokens, bit for bit (the kernel only moves bf16 bits);
* the sequential copy-on-write manager (``BlockManagerRef``): handling the
  sequences one by one in index order, popping the same free stack.  The
  GPU's block table, lengths, reference counts and stack top must equal it
  exactly (integer work).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa_attn_fwd_b300 import binding
from tests.parity import compare, f64

pytestmark = pytest.mark.gpu

BS = 16


def forked_state(seed, groups, lens, num_blocks, Hkv=2, d=128, max_blocks=40):
    """Sequences in `groups` share every block of their common prefix (a fork
    after lens[group[0]] tokens, partial last block included).  Returns host
    tensors: caches (NaN outside valid slots), table, lens, refs, free stack,
    and each sequence's logical K/V."""
    g = torch.Generator().manual_seed(seed)
    kc = torch.full((num_blocks, Hkv, BS, d), float("nan"), dtype=torch.bfloat16)
    vc = torch.full_like(kc, float("nan"))
    order = torch.randperm(num_blocks, generator=g).tolist()
    bt = torch.zeros(sum(len(x) for x in groups), max_blocks, dtype=torch.int32)
    S = bt.shape[0]
    seq_lens = torch.zeros(S, dtype=torch.int32)
    refs = torch.zeros(num_blocks, dtype=torch.int32)
    logical_k, logical_v = [None] * S, [None] * S
    for grp in groups:
        n = lens[grp[0]]
        nb = (n + BS - 1) // BS
        blocks = [order.pop() for _ in range(nb)]
        k = torch.randn(n, Hkv, d, generator=g).to(torch.bfloat16)
        v = torch.randn(n, Hkv, d, generator=g).to(torch.bfloat16)
        for t in range(n):
            kc[blocks[t // BS], :, t % BS] = k[t]
            vc[blocks[t // BS], :, t % BS] = v[t]
        for s in grp:
            bt[s, :nb] = torch.tensor(blocks, dtype=torch.int32)
            seq_lens[s] = n
            logical_k[s], logical_v[s] = k.clone(), v.clone()
            for b in blocks:
                refs[b] += 1
    free = torch.tensor(order, dtype=torch.int32)  # top of the stack = last entry
    return dict(kc=kc, vc=vc, bt=bt, lens=seq_lens, refs=refs, free=free,
                lk=logical_k, lv=logical_v)


def gpu_append(st, k_new, v_new):
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in st.items()
           if k in ("kc", "vc", "bt", "lens", "refs", "free")}
    top = torch.tensor([st["free"].numel()], dtype=torch.int32, device="cuda")
    binding.kv_append(k_new.cuda(), v_new.cuda(), dev["kc"], dev["vc"], dev["bt"], dev["lens"],
                      dev["refs"], dev["free"], top)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in dev.items()}, int(top.item())


def read_logical(cache, bt, lens):
    out = []
    for s in range(bt.shape[0]):
        n = int(lens[s])
        rows = [cache[int(bt[s, t // BS]), :, t % BS] for t in range(n)]
        out.append(torch.stack(rows) if rows else cache[:0, :, 0])
    return out


def bits(t):
    return t.contiguous().view(torch.int16)


GROUPS = [(0, 1, 2), (3, 4), (5,), (6, 7, 8, 9)]
LENS = {0: 21, 3: 32, 5: 5, 6: 47}


def _lens_per_seq():
    out = []
    for grp in GROUPS:
        out += [LENS[grp[0]]] * len(grp)
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 3, 16, 20])
def test_append_matches_logical_and_sequential_manager(d, T):
    lens = _lens_per_seq()
    st = forked_state(T * 7 + d, GROUPS, lens, num_blocks=96, d=d)
    S = len(lens)
    g = torch.Generator().manual_seed(T)
    k_new = torch.randn(S, T, 2, d, generator=g).to(torch.bfloat16)
    v_new = torch.randn(S, T, 2, d, generator=g).to(torch.bfloat16)
    out, top = gpu_append(st, k_new, v_new)

    mgr = oracle.BlockManagerRef(st["bt"].numpy(), st["lens"].numpy(), 96, st["free"].tolist())
    for s in range(S):
        mgr.append(s, T)
    assert top == len(mgr.free)
    assert out["lens"].tolist() == mgr.lens
    assert np.array_equal(out["refs"].numpy(), mgr.ref)
    for s in range(S):
        nb = (mgr.lens[s] + BS - 1) // BS
        assert out["bt"][s, :nb].tolist() == mgr.tables[s]

    want_k = [torch.cat([st["lk"][s], k_new[s]]) for s in range(S)]
    want_v = [torch.cat([st["lv"][s], v_new[s]]) for s in range(S)]
    got_k = read_logical(out["kc"], out["bt"], out["lens"])
    got_v = read_logical(out["vc"], out["bt"], out["lens"])
    for s in range(S):
        assert torch.equal(bits(got_k[s]), bits(want_k[s])), s
        assert torch.equal(bits(got_v[s]), bits(want_v[s])), s
    assert binding.device_status() == binding.ATTN_OK


def test_decode_steps_then_paged_decode_matches_oracle():
    # 24 decode steps of one token each, then attention over the grown caches.
    lens = _lens_per_seq()
    st = forked_state(5, GROUPS, lens, num_blocks=128)
    S = len(lens)
    dev = {k: st[k].cuda() for k in ("kc", "vc", "bt", "lens", "refs", "free")}
    top = torch.tensor([st["free"].numel()], dtype=torch.int32, device="cuda")
    g = torch.Generator().manual_seed(9)
    lk, lv = list(st["lk"]), list(st["lv"])
    for step in range(24):
        kn = torch.randn(S, 1, 2, 128, generator=g).to(torch.bfloat16)
        vn = torch.randn(S, 1, 2, 128, generator=g).to(torch.bfloat16)
        binding.kv_append(kn.cuda(), vn.cuda(), dev["kc"], dev["vc"], dev["bt"], dev["lens"],
                          dev["refs"], dev["free"], top)
        lk = [torch.cat([lk[s], kn[s]]) for s in range(S)]
        lv = [torch.cat([lv[s], vn[s]]) for s in range(S)]
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    q = torch.randn(S, 8, 128, generator=g).to(torch.bfloat16)
    o, lse = binding.paged_decode(q.cuda(), dev["kc"], dev["vc"], dev["bt"], dev["lens"])
    O, L = oracle.paged_decode_ref(f64(q), [f64(x) for x in lk], [f64(x) for x in lv],
                                   1 / math.sqrt(128))
    compare(f64(o.cpu()), f64(lse.cpu()), O, L, "decode after appends")
    # every written (last) block is private; refs match the table
    bt, ln, refs = dev["bt"].cpu(), dev["lens"].cpu(), dev["refs"].cpu()
    count = torch.zeros_like(refs)
    for s in range(S):
        for b in bt[s, :(int(ln[s]) + BS - 1) // BS].tolist():
            count[b] += 1
    assert torch.equal(count, refs)
    for s in range(S):
        assert int(refs[int(bt[s, (int(ln[s]) - 1) // BS])]) == 1


def test_empty_stack_changes_nothing_and_reports():
    lens = _lens_per_seq()
    st = forked_state(3, GROUPS, lens, num_blocks=40)
    st["free"] = st["free"][:2]  # far too few blocks for 10 sequences x 20 tokens
    S = len(lens)
    k_new = torch.zeros(S, 20, 2, 128, dtype=torch.bfloat16)
    out, top = gpu_append(st, k_new, k_new)
    assert binding.device_status() == binding.ATTN_EDEVICE
    assert top == 2
    assert torch.equal(out["bt"], st["bt"]) and torch.equal(out["lens"], st["lens"])
    assert torch.equal(out["refs"], st["refs"])
    assert torch.equal(bits(out["kc"]), bits(st["kc"]))


def test_table_overflow_reports():
    lens = _lens_per_seq()
    st = forked_state(4, GROUPS, lens, num_blocks=96, max_blocks=4)  # 64 tokens per sequence
    S = len(lens)
    k_new = torch.zeros(S, 20, 2, 128, dtype=torch.bfloat16)  # 47 + 20 > 64
    out, top = gpu_append(st, k_new, k_new)
    assert binding.device_status() == binding.ATTN_EDEVICE
    assert torch.equal(out["lens"], st["lens"]) and torch.equal(out["bt"], st["bt"])
