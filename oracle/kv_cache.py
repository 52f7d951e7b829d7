"""Reference for appending to a paged KV cache (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may use this module; the CUDA path never does.

Source: tutorial "第 3 章 进阶原理:性能模型与数值稳定性", section 3.0.6 (the
PagedAttention building blocks are the block table, sharing, and copy-on-write)
and 3.0.7 (block size 16; parallel sampling shares prefix blocks); section
3.0.2 item 3 (sharing must leave every sequence's attention unchanged).

The pages name copy-on-write but do not spell it out; the plain reading used
here (the one the kernels implement):

* A sequence's LOGICAL cache is the list of its tokens' K/V rows.  Appending T
  tokens extends that list; nothing else changes -- in particular, appending
  to one sequence never changes another sequence's logical cache, even when
  the two share physical blocks.  ``append_logical`` is that definition.
* ``BlockManagerRef`` is a sequential, one-sequence-at-a-time statement of the
  bookkeeping: a write into a block that other sequences still reference
  first copies the block into a fresh one (copy-on-write); a write into a
  block nobody else references happens in place; a write past the last block
  takes a fresh block.  Fresh blocks come off the top of a free stack, in
  sequence order.  Because that order is fixed, the resulting tables --
  physical block ids included --, reference counts and stack top are unique,
  and the GPU tests compare all of them exactly with this manager's.
"""

from __future__ import annotations

import numpy as np


def append_logical(k_seqs, v_seqs, k_new: np.ndarray, v_new: np.ndarray):
    """Logical caches after every sequence s appends k_new[s], v_new[s].

    k_seqs / v_seqs: entry s is [len_s, Hkv, d]; k_new / v_new: [S, T, Hkv, d].
    Returns the new lists (entry s is [len_s + T, Hkv, d]).
    """
    ks = [np.concatenate([np.asarray(k), np.asarray(k_new[s])], axis=0) for s, k in enumerate(k_seqs)]
    vs = [np.concatenate([np.asarray(v), np.asarray(v_new[s])], axis=0) for s, v in enumerate(v_seqs)]
    return ks, vs


class BlockManagerRef:
    """Sequential block bookkeeping with copy-on-write (plain Python).

    tables: per sequence, the list of physical block ids; lens: tokens per
    sequence; ref: reference count per physical block; free: free stack (the
    top is the end of the list).
    """

    def __init__(self, tables, lens, num_blocks, free, block_size=16):
        self.bs = block_size
        self.lens = [int(n) for n in lens]
        # only the blocks that hold tokens; entries past them are unused
        self.tables = [list(t[:(n + block_size - 1) // block_size])
                       for t, n in zip(tables, self.lens)]
        self.ref = np.zeros(num_blocks, dtype=np.int64)
        for t, n in zip(self.tables, self.lens):
            for b in t[:(n + block_size - 1) // block_size]:
                self.ref[b] += 1
        self.free = list(free)
        self.copies = []  # (src, dst) block copies performed

    def append(self, s: int, T: int):
        """Make room for T more tokens of sequence s; returns the physical
        (block, slot) of each new token."""
        out = []
        for t in range(T):
            pos = self.lens[s]
            lb, off = divmod(pos, self.bs)
            if off == 0:  # the token starts a new block
                blk = self.free.pop()
                self.ref[blk] = 1
                self.tables[s].append(blk)
            else:
                blk = self.tables[s][lb]
                if self.ref[blk] > 1:  # shared: copy before writing
                    new = self.free.pop()
                    self.ref[blk] -= 1
                    self.ref[new] = 1
                    self.copies.append((blk, new))
                    self.tables[s][lb] = new
                    blk = new
            out.append((blk, off))
            self.lens[s] = pos + 1
        return out
