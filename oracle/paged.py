"""fp64 reference for decode attention over a paged KV cache (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may use this module; the CUDA path never does.

Sources:

* Tutorial "第 3 章 进阶原理:性能模型与数值稳定性", section 3.0.6 and 3.0.7:
  PagedAttention keeps the KV cache in fixed-size blocks addressed through a
  block table; several sequences (parallel sampling, beam search) map the same
  physical blocks for a shared prefix; block size is commonly 16.  The page's
  point is that this paging must not change which attention is computed.
* "以 Transformer 为例进行分析", section 三 (decode computes one token per step)
  and 3.1.1 (PagedAttention: efficient storage and access of the KV cache).

What is computed: for every sequence s and query head h, one query row
attends all ``seq_len[s]`` keys of the sequence, with no causal mask (the
single decode query is the newest token, so every cached key precedes it):
o = softmax(scale * q k^T) v and lse, by the plain definition in
``oracle.attention``.  GQA as in that module: head h reads KV head h // G.

Two entry points:

* ``paged_decode_ref`` takes each sequence's LOGICAL contiguous K/V and never
  sees a block table.  The GPU parity tests compare against this one, so an
  indexing error on the GPU cannot be cancelled by the same error here.
* ``paged_prefill_ref`` is the chunked-prefill case: each sequence's Nq new
  queries attend its logical K/V (the cache already holds the chunk's own
  keys), with the causal mask aligned to the end of the cache.
* ``paged_decode_ref_from_pool`` first gathers the logical K/V from a
  physical pool through the block table (``gather_logical_kv``, plain loops),
  then calls the same definition.  Tests pin it to ``paged_decode_ref``
  under arbitrary block permutations and prefix sharing.
"""

from __future__ import annotations

import numpy as np

from .attention import attention_ref, scores, softmax_rows


def paged_decode_ref(q: np.ndarray, k_seqs, v_seqs, scale: float):
    """Decode attention of one query per sequence over its logical K/V.

    q: [S, H, d] float64.  k_seqs / v_seqs: sequences of arrays, entry s of
    shape [seq_len_s, Hkv, d].  Returns O [S, H, d] and lse [S, H] (float64).
    """
    q = np.asarray(q, dtype=np.float64)
    S_, H, d = q.shape
    O = np.zeros((S_, H, d))
    lse = np.zeros((S_, H))
    for s in range(S_):
        ks = np.asarray(k_seqs[s], dtype=np.float64)
        vs = np.asarray(v_seqs[s], dtype=np.float64)
        n, Hkv, dk = ks.shape
        if dk != d or vs.shape != ks.shape or H % Hkv:
            raise ValueError("bad K/V shape for sequence %d" % s)
        G = H // Hkv
        for h in range(H):
            g = h // G
            Srow = scores(q[s, h][None, :], ks[:, g, :], scale, False,
                          np.zeros(1, dtype=np.int64), 1)
            P, _, l = softmax_rows(Srow)
            O[s, h] = (P @ vs[:, g, :])[0]
            lse[s, h] = l[0]
    return O, lse


def gather_logical_kv(cache: np.ndarray, block_table: np.ndarray,
                      seq_lens: np.ndarray, block_size: int):
    """Read each sequence's logical [seq_len, Hkv, d] K (or V) from the pool.

    cache: [num_blocks, Hkv, block_size, d]; block_table: [S, max_blocks]
    (logical block -> physical block); seq_lens: [S].  Token t of sequence s
    lives in physical block block_table[s, t // block_size] at slot
    t % block_size.  Plain loops, one token at a time.
    """
    cache = np.asarray(cache)
    out = []
    for s in range(len(seq_lens)):
        n = int(seq_lens[s])
        Hkv, d = cache.shape[1], cache.shape[3]
        rows = np.empty((n, Hkv, d), dtype=cache.dtype)
        for t in range(n):
            phys = int(block_table[s, t // block_size])
            rows[t] = cache[phys, :, t % block_size, :]
        out.append(rows)
    return out


def paged_decode_ref_from_pool(q, k_cache, v_cache, block_table, seq_lens,
                               block_size: int, scale: float):
    """Gather logical K/V through the block table, then ``paged_decode_ref``."""
    ks = gather_logical_kv(k_cache, block_table, seq_lens, block_size)
    vs = gather_logical_kv(v_cache, block_table, seq_lens, block_size)
    return paged_decode_ref(q, ks, vs, scale)


def paged_prefill_ref(q: np.ndarray, k_seqs, v_seqs, scale: float, causal: bool, rows=None):
    """Chunked prefill over a paged cache, by the plain definition.

    q: [S, H, Nq, d] float64, the Nq newest tokens of every sequence (the
    chunk being prefilled).  k_seqs / v_seqs: entry s is sequence s's logical
    K / V, [seq_len_s, Hkv, d]; the chunk's own keys are its last Nq entries.
    Returns O [S, H, R, d] and lse [S, H, R] for the query rows ``rows``
    (default all Nq).

    Tutorial "第 3 章 进阶原理:性能模型与数值稳定性", section 3.0.6: FlashAttention
    and PagedAttention cooperate -- the fused kernel reads its keys through the
    block table.  Query row i of the chunk is token seq_len - Nq + i of the
    sequence, so under the causal mask it attends keys j <= i + (seq_len - Nq)
    (the bottom-right alignment of ``oracle.attention``); a row with no key
    (seq_len < Nq) gives O = 0 and lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    S_, H, Nq, d = q.shape
    R = Nq if rows is None else len(rows)
    O = np.zeros((S_, H, R, d))
    lse = np.zeros((S_, H, R))
    for s in range(S_):
        ks = np.asarray(k_seqs[s], dtype=np.float64)   # [n, Hkv, d]
        vs = np.asarray(v_seqs[s], dtype=np.float64)
        kk = ks.transpose(1, 0, 2)[None]                # [1, Hkv, n, d]
        vv = vs.transpose(1, 0, 2)[None]
        Os, Ls = attention_ref(q[s][None], kk, vv, scale, causal, rows=rows)
        O[s] = Os[0]
        lse[s] = Ls[0]
    return O, lse
