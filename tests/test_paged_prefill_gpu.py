"""GPU parity of paged_prefill (C ABI) against the fp64 oracle.

The oracle reads each sequence's LOGICAL K/V (never the block table), so an
indexing error on the GPU cannot be cancelled on the reference side.  A
second, exact check: with every sequence's K/V gathered into contiguous
tensors, attn_fwd runs the same tiles in the same order, so the paged result
must be bit-identical to it.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa_attn_fwd_b300 import binding, workloads
from tests.parity import compare, f64, sample_rows

pytestmark = pytest.mark.gpu


def _gpu(pb, causal=True, seq_lens=None, block_table=None):
    sl = pb.seq_lens if seq_lens is None else seq_lens
    bt = pb.block_table if block_table is None else block_table
    o, lse = binding.paged_prefill(pb.q.cuda(), pb.k_cache.cuda(), pb.v_cache.cuda(), bt.cuda(),
                                   sl.cuda(), causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def _ref(pb, causal, rows=None, seq_lens=None):
    d = pb.q.shape[-1]
    ks, vs = [], []
    for s in range(pb.num_seqs):
        k, v = pb.logical_kv(s)
        n = int(pb.seq_lens[s] if seq_lens is None else seq_lens[s])
        ks.append(f64(k[:n]))
        vs.append(f64(v[:n]))
    return oracle.paged_prefill_ref(f64(pb.q), ks, vs, 1 / math.sqrt(d), causal, rows=rows)


def _small(**kw):
    base = dict(num_seqs=4, H=8, Hkv=2, d=128, Nq=200, min_hist=0, max_hist=300)
    base.update(kw)
    seed = base.pop("seed", 0)
    return workloads.paged_prefill_inputs(**base, seed=seed)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Nq", [1, 17, 128, 200, 300])
def test_small_batches(d, causal, Nq):
    pb = _small(d=d, Nq=Nq, seed=Nq + d)
    o, lse = _gpu(pb, causal)
    O, L = _ref(pb, causal)
    compare(f64(o), f64(lse), O, L, f"paged prefill d={d} Nq={Nq} causal={causal}")


@pytest.mark.parametrize("H,Hkv", [(8, 8), (8, 1), (6, 3), (32, 8)])
def test_gqa_ratios(H, Hkv):
    pb = _small(H=H, Hkv=Hkv, Nq=256, max_hist=700, seed=H * 3 + Hkv)
    o, lse = _gpu(pb)
    O, L = _ref(pb, True)
    compare(f64(o), f64(lse), O, L, f"paged prefill H={H} Hkv={Hkv}")


def test_shared_prefix_blocks():
    pb = _small(num_seqs=8, Nq=64, min_hist=100, max_hist=600, group=4, shared_tokens=96, seed=3)
    assert pb.unique_valid_tokens() < pb.logical_tokens()
    o, lse = _gpu(pb)
    O, L = _ref(pb, True)
    compare(f64(o), f64(lse), O, L, "paged prefill shared prefix")


def test_cache_shorter_than_chunk_masks_leading_rows():
    pb = _small(Nq=160, min_hist=0, max_hist=100, seed=4)
    lens = pb.seq_lens.clone()
    lens[0] = 37    # rows 0..122 of sequence 0 see no key
    lens[1] = 0     # no key at all
    lens[2] = 160   # exactly the chunk
    o, lse = _gpu(pb, seq_lens=lens)
    assert torch.all(o[0, :, :123].float() == 0) and torch.all(torch.isneginf(lse[0, :, :123]))
    assert torch.all(o[1].float() == 0) and torch.all(torch.isneginf(lse[1]))
    O, L = _ref(pb, True, seq_lens=lens)
    compare(f64(o), f64(lse), O, L, "short caches")


def test_bit_identical_to_attn_fwd_on_gathered_kv():
    # Equal lengths, so attn_fwd over the gathered contiguous K/V runs the very
    # same tiles: any wrong block id or tail handling shows up as a bit flip.
    pb = _small(num_seqs=3, H=8, Hkv=2, Nq=384, min_hist=500, max_hist=500, seed=5)
    assert len(set(pb.seq_lens.tolist())) == 1
    n = int(pb.seq_lens[0])
    k = torch.stack([pb.logical_kv(s)[0] for s in range(3)]).permute(0, 2, 1, 3).contiguous()
    v = torch.stack([pb.logical_kv(s)[1] for s in range(3)]).permute(0, 2, 1, 3).contiguous()
    assert k.shape[2] == n
    o1, l1 = _gpu(pb)
    o2, l2 = binding.attn_fwd(pb.q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2.cpu()) and torch.equal(l1, l2.cpu())


@pytest.mark.parametrize("perm_seed", [11, 22])
def test_physical_permutation_gives_identical_bits(perm_seed):
    a = _small(seed=6)
    b = _small(seed=6, perm_seed=perm_seed)
    assert not torch.equal(a.block_table, b.block_table)
    o1, l1 = _gpu(a)
    o2, l2 = _gpu(b)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_out_of_range_block_id_reports_device_error():
    pb = _small(seed=7)
    bt = pb.block_table.clone()
    bt[1, 2] = pb.num_blocks + 3
    o, lse = binding.paged_prefill(pb.q.cuda(), pb.k_cache.cuda(), pb.v_cache.cuda(), bt.cuda(),
                                   pb.seq_lens.cuda())
    assert binding.device_status() == binding.ATTN_EDEVICE
    assert binding.device_status() == binding.ATTN_OK
    O, L = _ref(pb, True)
    good = [0, 2, 3]
    compare(f64(o.cpu()[good]), f64(lse.cpu()[good]), O[good], L[good], "other sequences")


def test_paged_prefill_workload_sampled():
    cfg = workloads.PAGED_PREFILL_WORKLOADS["paged_prefill_s8_h32kv8_q2048_d128"]
    pb = workloads.paged_prefill_inputs(**cfg, seed=0)
    o, lse = _gpu(pb)
    rows = sample_rows(cfg["Nq"], 48, seed=4)
    O, L = _ref(pb, True, rows=rows)
    compare(f64(o[:, :, rows]), f64(lse[:, :, rows]), O, L, "paged prefill workload")
    assert binding.device_status() == binding.ATTN_OK


@pytest.mark.parametrize("num_seqs,min_hist,max_hist", [
    (64, 0, 300),    # longest-first order, two candidates per lane when ranking
    (6, 120, 120),   # equal lengths: the ranking breaks ties by sequence index
    (70, 0, 90),     # more than 64 sequences: plain index order
])
def test_grid_order_by_sequence_length(num_seqs, min_hist, max_hist):
    pb = _small(num_seqs=num_seqs, H=4, Hkv=2, d=64, Nq=33, min_hist=min_hist,
                max_hist=max_hist, seed=num_seqs)
    o, lse = _gpu(pb, True)
    O, L = _ref(pb, True)
    compare(f64(o), f64(lse), O, L, f"paged prefill {num_seqs} seqs, hist {min_hist}..{max_hist}")
    assert binding.device_status() == binding.ATTN_OK
