"""Seeded synthetic inputs for the attention hot path.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  It is the one module both the CUDA path's tests/bench
and the fp64 oracle consume, so both see byte-identical inputs.

Recipe (fixed so every run reproduces the same bytes):

* ``torch.Generator('cpu').manual_seed(seed)``; draws are float32 N(0, 1) via
  ``torch.randn`` in the order Q, K, V (then, for paged decode, lengths, the
  unique K blocks, the unique V blocks, the physical permutation), then rounded
  to bfloat16 (round-to-nearest-even).
* ``qk_gain`` multiplies Q and K in float32 before rounding (the long-context
  workload draws Q, K ~ N(0,1) * 1.5 for a peakier softmax).
* Paged decode: lengths are integer-uniform in [min_len, max_len]; sequences
  4g .. 4g+3 share their first ``shared_tokens // block_size`` logical blocks
  (same physical ids, parallel-sampling style); every other block is unique.
  The pool holds the unique blocks plus ``spare_frac`` spare blocks, at a
  random permutation of physical ids.  Spare blocks, slots past a sequence's
  length in its last block, and block-table entries past a sequence's last
  block (which point at a spare block) are NaN-poisoned, so a kernel that
  reads them produces NaN instead of a plausible wrong value.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch


# ---------------------------------------------------------------------------
# Workload table.  Sizes are the ones the pages' method is exercised on:
# a tiny case, a mid-size causal MHA prefill, a long-context causal GQA
# prefill, a sequence-length sweep at a fixed token count, and a batch of
# paged decode steps with shared prefixes.
# ---------------------------------------------------------------------------

PREFILL_WORKLOADS = {
    "tiny_b1h2_n128_d64": dict(B=1, H=2, Hkv=2, Nq=128, Nk=128, d=64, causal=False, qk_gain=1.0),
    "mha_b2h16_n2048_d128_causal": dict(B=2, H=16, Hkv=16, Nq=2048, Nk=2048, d=128, causal=True, qk_gain=1.0),
    "gqa_b1h32kv8_n16384_d128_causal": dict(B=1, H=32, Hkv=8, Nq=16384, Nk=16384, d=128, causal=True, qk_gain=1.5),
}


def sweep_workloads():
    """Sequence-length sweep at B*N = 16384 tokens, H = Hkv = 16."""
    out = {}
    for d in (64, 128):
        for causal in (False, True):
            for N in (512, 1024, 2048, 4096, 8192, 16384):
                name = f"sweep_n{N}_d{d}_{'causal' if causal else 'full'}"
                out[name] = dict(B=16384 // N, H=16, Hkv=16, Nq=N, Nk=N, d=d,
                                 causal=causal, qk_gain=1.0)
    return out


PAGED_WORKLOADS = {
    "paged_decode_s64_h32kv8_d128": dict(num_seqs=64, H=32, Hkv=8, d=128, block_size=16,
                                        min_len=1024, max_len=8192, group=4,
                                        shared_tokens=512, spare_frac=0.05),
}


# Chunked prefill over a paged cache: 8 sequences each append a 2048-token
# chunk to a history of U{0..14336} cached tokens (at most 16384 in all).
PAGED_PREFILL_WORKLOADS = {
    "paged_prefill_s8_h32kv8_q2048_d128": dict(num_seqs=8, H=32, Hkv=8, d=128, Nq=2048,
                                              block_size=16, min_hist=0, max_hist=14336,
                                              group=1, shared_tokens=0, spare_frac=0.05),
}


def prefill_inputs(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int,
                   seed: int = 0, qk_gain: float = 1.0, **_unused):
    """Q [B,H,Nq,d], K [B,Hkv,Nk,d], V [B,Hkv,Nk,d] bfloat16 on the CPU."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, H, Nq, d, generator=g, dtype=torch.float32)
    k = torch.randn(B, Hkv, Nk, d, generator=g, dtype=torch.float32)
    v = torch.randn(B, Hkv, Nk, d, generator=g, dtype=torch.float32)
    if qk_gain != 1.0:
        q.mul_(qk_gain)
        k.mul_(qk_gain)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def grad_output(shape, seed: int = 0) -> torch.Tensor:
    """dL/dO for the backward pass: bfloat16 N(0, 1) of ``shape`` from its own
    generator (seed + 7919), so Q, K, V of the same seed are unchanged."""
    g = torch.Generator("cpu").manual_seed(seed + 7919)
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


@dataclasses.dataclass
class PagedBatch:
    q: torch.Tensor               # [S, H, d] bf16 (decode) or [S, H, Nq, d] (chunked prefill)
    k_cache: torch.Tensor         # [num_blocks, Hkv, block_size, d] bf16 (NaN-poisoned spares)
    v_cache: torch.Tensor
    block_table: torch.Tensor     # [S, max_blocks_per_seq] int32
    seq_lens: torch.Tensor        # [S] int32
    block_size: int
    logical_ids: List[List[int]]  # per sequence: unique-block id of each logical block
    perm: torch.Tensor            # unique-block id -> physical block id (first U entries)
    k_unique: torch.Tensor        # [U, Hkv, block_size, d] bf16
    v_unique: torch.Tensor
    num_unique: int

    @property
    def num_seqs(self) -> int:
        return self.q.shape[0]

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_table.shape[1]

    def logical_kv(self, s: int):
        """Sequence s's logical K, V as [seq_len, Hkv, d] bf16 (no table lookup)."""
        ids = torch.tensor(self.logical_ids[s], dtype=torch.long)
        n = int(self.seq_lens[s])
        k = self.k_unique[ids].permute(0, 2, 1, 3).reshape(-1, self.k_unique.shape[1], self.k_unique.shape[3])
        v = self.v_unique[ids].permute(0, 2, 1, 3).reshape(-1, self.v_unique.shape[1], self.v_unique.shape[3])
        return k[:n], v[:n]

    def unique_valid_tokens(self) -> int:
        """Tokens the decode step must read once: valid slots of distinct physical blocks."""
        seen = {}
        for s, ids in enumerate(self.logical_ids):
            n = int(self.seq_lens[s])
            for lb, u in enumerate(ids):
                valid = min(self.block_size, n - lb * self.block_size)
                seen[u] = max(seen.get(u, 0), valid)
        return sum(seen.values())

    def logical_tokens(self) -> int:
        return int(self.seq_lens.sum())


def paged_decode_inputs(num_seqs: int = 64, H: int = 32, Hkv: int = 8, d: int = 128,
                        block_size: int = 16, min_len: int = 1024, max_len: int = 8192,
                        group: int = 4, shared_tokens: int = 512, spare_frac: float = 0.05,
                        max_blocks_per_seq: Optional[int] = None, seed: int = 0,
                        perm_seed: Optional[int] = None, share: bool = True,
                        index_probe: bool = False):
    """Build a paged KV cache batch for decode (see module docstring for the recipe).

    ``perm_seed``: draw the physical permutation from its own generator (all
    other draws unchanged), so tests can vary only the block placement.
    ``share=False``: give every sequence private copies of its group's prefix
    blocks with identical contents (same logical K/V, no shared ids).
    ``index_probe``: replace the random K/V by a pattern that makes one chosen
    logical position per sequence dominate (scaled score about +40 above the
    rest) and whose V rows encode the logical token index exactly in bf16
    (v[..., 0] = 1 + t // 64, v[..., 1] = 1 + t % 64, v[..., 2] = 1 + kv head;
    never 0, so the ~1e-16 weight of the other keys cannot show after rounding).
    """
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(num_seqs, H, d, generator=g, dtype=torch.float32)
    lens = torch.randint(min_len, max_len + 1, (num_seqs,), generator=g, dtype=torch.int64)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = (max_len + block_size - 1) // block_size
    return _paged_pool(g, q, lens, H, Hkv, d, block_size, group, shared_tokens, spare_frac,
                       max_blocks_per_seq, perm_seed, share, index_probe)


def paged_prefill_inputs(num_seqs: int = 8, H: int = 32, Hkv: int = 8, d: int = 128,
                         Nq: int = 2048, block_size: int = 16, min_hist: int = 0,
                         max_hist: int = 14336, group: int = 1, shared_tokens: int = 0,
                         spare_frac: float = 0.05, qk_gain: float = 1.0,
                         max_blocks_per_seq: Optional[int] = None, seed: int = 0,
                         perm_seed: Optional[int] = None, share: bool = True):
    """Paged KV cache for a chunked prefill: every sequence appends a chunk of
    ``Nq`` new tokens to a cached history of U{min_hist..max_hist} tokens.

    The cache already holds the chunk's own K/V, so sequence s has
    ``seq_lens[s] = hist_s + Nq`` cached tokens.  q is [S, H, Nq, d].  Draw
    order: Q, history lengths, then the pool exactly as for decode.
    ``qk_gain`` scales Q and every K block in float32 before rounding.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(num_seqs, H, Nq, d, generator=g, dtype=torch.float32)
    hist = torch.randint(min_hist, max_hist + 1, (num_seqs,), generator=g, dtype=torch.int64)
    lens = hist + Nq
    if max_blocks_per_seq is None:
        max_blocks_per_seq = (max_hist + Nq + block_size - 1) // block_size
    if qk_gain != 1.0:
        q.mul_(qk_gain)
    return _paged_pool(g, q, lens, H, Hkv, d, block_size, group, shared_tokens, spare_frac,
                       max_blocks_per_seq, perm_seed, share, False, k_gain=qk_gain)


def _paged_pool(g, q, lens, H, Hkv, d, block_size, group, shared_tokens, spare_frac,
                max_blocks_per_seq, perm_seed, share, index_probe, k_gain: float = 1.0):
    """Lay the logical blocks of every sequence out in a permuted, NaN-poisoned pool."""
    num_seqs = q.shape[0]
    min_len = int(lens.min())
    if group > 1 and shared_tokens % block_size:
        raise ValueError("shared_tokens must be a whole number of blocks")
    if group > 1 and min_len <= shared_tokens:
        raise ValueError("every sequence needs at least one private block")
    nblk = [(int(n) + block_size - 1) // block_size for n in lens]
    if max(nblk) > max_blocks_per_seq:
        raise ValueError("max_blocks_per_seq too small")
    shared_blocks = shared_tokens // block_size if group > 1 else 0

    # Logical -> unique block ids.  Shared prefixes: the same unique id for
    # every member of a group (share=True) or a copy-by-id per member that is
    # later filled with the same contents (share=False).
    logical_ids: List[List[int]] = []
    prefix_src = {}  # unique id of a private prefix copy -> id whose contents it copies
    nxt = 0
    for s0 in range(0, num_seqs, max(group, 1)):
        members = range(s0, min(s0 + max(group, 1), num_seqs))
        pre = list(range(nxt, nxt + shared_blocks))
        nxt += shared_blocks
        for i, s in enumerate(members):
            if share or i == 0:
                ids = list(pre)
            else:
                ids = list(range(nxt, nxt + shared_blocks))
                for a, b in zip(ids, pre):
                    prefix_src[a] = b
                nxt += shared_blocks
            priv = nblk[s] - shared_blocks
            ids += list(range(nxt, nxt + priv))
            nxt += priv
            logical_ids.append(ids)
    U = nxt
    # Draw contents for the blocks of the shared layout, so share=True and
    # share=False produce the same logical K/V from the same seed.
    U_draw = U - len(prefix_src)
    draw_of = {}
    c = 0
    for u in range(U):
        if u not in prefix_src:
            draw_of[u] = c
            c += 1
    kd = torch.randn(U_draw, Hkv, block_size, d, generator=g, dtype=torch.float32)
    vd = torch.randn(U_draw, Hkv, block_size, d, generator=g, dtype=torch.float32)
    src = torch.tensor([draw_of[prefix_src.get(u, u)] for u in range(U)], dtype=torch.long)
    k_u = kd[src]
    v_u = vd[src]
    if k_gain != 1.0:
        k_u.mul_(k_gain)
    if index_probe:
        k_u, v_u, q = _index_probe(q, k_u, v_u, logical_ids, lens, block_size, H, Hkv, d, g,
                                   shared_blocks)
    num_blocks = U + int(math.ceil(spare_frac * U))
    pg = g if perm_seed is None else torch.Generator("cpu").manual_seed(perm_seed)
    perm = torch.randperm(num_blocks, generator=pg)

    q = q.to(torch.bfloat16)
    k_u = k_u.to(torch.bfloat16)
    v_u = v_u.to(torch.bfloat16)
    nan = float("nan")
    k_cache = torch.full((num_blocks, Hkv, block_size, d), nan, dtype=torch.bfloat16)
    v_cache = torch.full((num_blocks, Hkv, block_size, d), nan, dtype=torch.bfloat16)
    k_cache[perm[:U]] = k_u
    v_cache[perm[:U]] = v_u
    # NaN-poison slots past each sequence's length (its last block is private).
    for s, ids in enumerate(logical_ids):
        valid = int(lens[s]) - block_size * (len(ids) - 1)
        if valid < block_size:
            phys = int(perm[ids[-1]])
            k_cache[phys, :, valid:, :] = nan
            v_cache[phys, :, valid:, :] = nan
    filler = int(perm[U]) if num_blocks > U else int(perm[0])
    bt = torch.full((num_seqs, max_blocks_per_seq), filler, dtype=torch.int32)
    for s, ids in enumerate(logical_ids):
        bt[s, :len(ids)] = perm[torch.tensor(ids, dtype=torch.long)].to(torch.int32)
    return PagedBatch(q=q, k_cache=k_cache, v_cache=v_cache, block_table=bt,
                      seq_lens=lens.to(torch.int32), block_size=block_size,
                      logical_ids=logical_ids, perm=perm, k_unique=k_u, v_unique=v_u,
                      num_unique=U)


def _index_probe(q, k_u, v_u, logical_ids, lens, block_size, H, Hkv, d, g, shared_blocks):
    """Dominant-key / index-encoding pattern for the exact block-table check."""
    G = H // Hkv
    # Query: every head of a KV group is the same unit-ish vector u_g.
    u = torch.zeros(Hkv, d)
    for kv in range(Hkv):
        u[kv, (2 * kv) % d] = 1.0
        u[kv, (2 * kv + 1) % d] = 1.0
    q = u.repeat_interleave(G, dim=0)[None].expand(len(logical_ids), H, d).clone()
    # Background keys: small, orthogonal-ish noise.
    k_u = 0.05 * torch.randn(k_u.shape, generator=g)
    # V rows encode the logical token index: identical for a shared prefix block
    # because its logical positions are the same in every sharing sequence.
    v_u = torch.zeros_like(v_u)
    for s, ids in enumerate(logical_ids):
        for lb, uid in enumerate(ids):
            t = torch.arange(lb * block_size, (lb + 1) * block_size, dtype=torch.float32)
            v_u[uid, :, :, 0] = (1 + t // 64)[None, :]
            v_u[uid, :, :, 1] = (1 + t % 64)[None, :]
            v_u[uid, :, :, 2] = 1 + torch.arange(Hkv, dtype=torch.float32)[:, None]
    # One target per sequence in its private part (after any shared prefix).
    for s, ids in enumerate(logical_ids):
        n = int(lens[s])
        lo = max(n // 2, shared_blocks * block_size)
        t = int(torch.randint(lo, n, (1,), generator=g))
        uid = ids[t // block_size]
        # scale = 1/sqrt(d): score = a * |u|^2 / sqrt(d) = 2a/sqrt(d); pick a for ~ +40.
        a = 20.0 * math.sqrt(d)
        k_u[uid, :, t % block_size, :] = a * u
    return k_u, v_u, q
