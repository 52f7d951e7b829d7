"""GPU parity of attn_fwd (C ABI) against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa_attn_fwd_b300 import workloads
from tests.parity import check_prefill, compare, f64, run_prefill, sample_rows

pytestmark = pytest.mark.gpu


def _inputs(B, H, Hkv, Nq, Nk, d, seed=0, gain=1.0):
    return workloads.prefill_inputs(B, H, Hkv, Nq, Nk, d, seed=seed, qk_gain=gain)


def test_tiny_workload_full():
    cfg = workloads.PREFILL_WORKLOADS["tiny_b1h2_n128_d64"]
    q, k, v = workloads.prefill_inputs(**cfg)
    check_prefill(q, k, v, cfg["causal"], what="tiny")


@pytest.mark.parametrize("d", [64, 128])
def test_uniform_probabilities_give_mean_of_v(d):
    # q = 0: every score is 0, P is uniform -> O = mean(V), lse = ln Nk.
    # Checks the P V path (TMEM P operand, MN-major V) independently of Q K^T.
    q, k, v = _inputs(1, 2, 2, 128, 256, d, seed=3)
    q = torch.zeros_like(q)
    o, lse = run_prefill(q, k, v, False)
    ref = f64(v).mean(axis=2, keepdims=True)
    assert np.max(np.abs(f64(o) - ref)) < 2e-2
    assert np.max(np.abs(f64(lse) - math.log(256))) < 1e-3


@pytest.mark.parametrize("d", [64, 128])
def test_lse_only_depends_on_scores(d):
    # v = 0: O must be exactly 0; lse still checks the Q K^T path alone.
    q, k, v = _inputs(1, 2, 2, 256, 256, d, seed=4)
    v = torch.zeros_like(v)
    o, lse = run_prefill(q, k, v, True)
    assert torch.count_nonzero(o.float()) == 0
    _, L = oracle.attention_ref(f64(q), f64(k), f64(v), 1 / math.sqrt(d), True)
    assert np.max(np.abs(f64(lse) - L)) < 1e-3


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 128, 200, 383])
def test_ragged_lengths(d, causal, N):
    q, k, v = _inputs(1, 2, 1, N, N, d, seed=N)
    check_prefill(q, k, v, causal, what=f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("Nq,Nk", [(100, 300), (1, 257), (300, 100), (129, 1), (256, 640)])
@pytest.mark.parametrize("causal", [False, True])
def test_unequal_lengths_bottom_right_causal(Nq, Nk, causal):
    q, k, v = _inputs(2, 4, 2, Nq, Nk, 128, seed=Nq * 7 + Nk)
    check_prefill(q, k, v, causal, what=f"Nq={Nq} Nk={Nk} causal={causal}")


def test_fully_masked_rows_are_zero_with_neg_inf_lse():
    q, k, v = _inputs(1, 2, 2, 300, 100, 64, seed=9)
    o, lse = run_prefill(q, k, v, True)
    # rows i with i + (Nk - Nq) < 0, i.e. i < 200, attend nothing
    assert torch.all(o[:, :, :200].float() == 0)
    assert torch.all(torch.isneginf(lse[:, :, :200]))
    assert torch.all(torch.isfinite(lse[:, :, 200:]))


@pytest.mark.parametrize("H,Hkv", [(8, 1), (8, 2), (6, 3), (4, 4)])
def test_gqa_grouping(H, Hkv):
    q, k, v = _inputs(2, H, Hkv, 256, 256, 128, seed=H * 10 + Hkv)
    check_prefill(q, k, v, True, what=f"H={H} Hkv={Hkv}")


def test_peaky_softmax_triggers_rescale():
    # Large gains make the running max jump often: exercises the O rescale.
    q, k, v = _inputs(1, 2, 2, 512, 512, 128, seed=11, gain=3.0)
    check_prefill(q, k, v, True, what="gain 3")
    # increasing scores along the key axis: the max moves every tile
    qq = torch.ones(1, 1, 256, 64, dtype=torch.bfloat16)
    kk = (torch.arange(1024, dtype=torch.float32) / 64.0)[None, None, :, None].expand(1, 1, 1024, 64)
    vv = torch.randn(1, 1, 1024, 64, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    check_prefill(qq, kk.to(torch.bfloat16).contiguous(), vv, False, scale=0.125, what="ramp")


def test_non_default_scale():
    q, k, v = _inputs(1, 2, 2, 256, 256, 64, seed=12)
    check_prefill(q, k, v, True, scale=0.05, what="scale 0.05")


def test_workload_mha_b2h16_n2048_sampled():
    cfg = workloads.PREFILL_WORKLOADS["mha_b2h16_n2048_d128_causal"]
    q, k, v = workloads.prefill_inputs(**cfg)
    rows = sample_rows(cfg["Nq"], 256, seed=1)
    check_prefill(q, k, v, cfg["causal"], rows=rows, what="b2h16 n2048")


def test_workload_gqa_n16384_sampled():
    cfg = workloads.PREFILL_WORKLOADS["gqa_b1h32kv8_n16384_d128_causal"]
    q, k, v = workloads.prefill_inputs(**cfg)
    rows = sample_rows(cfg["Nq"], 512, seed=2)
    check_prefill(q, k, v, cfg["causal"], rows=rows, what="gqa n16384")


@pytest.mark.parametrize("name", sorted(workloads.sweep_workloads()))
def test_sweep_workloads_sampled(name):
    cfg = workloads.sweep_workloads()[name]
    q, k, v = workloads.prefill_inputs(**cfg)
    rows = sample_rows(cfg["Nq"], 48, seed=3)
    check_prefill(q, k, v, cfg["causal"], rows=rows, what=name)


def test_deterministic_and_lse_optional():
    from attention_fa_attn_fwd_b300 import attn_fwd
    q, k, v = (t.cuda() for t in _inputs(2, 4, 2, 700, 700, 128, seed=13))
    o1, l1 = attn_fwd(q, k, v, causal=True)
    o2, l2 = attn_fwd(q, k, v, causal=True)
    o3, l3 = attn_fwd(q, k, v, causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert l3 is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)


def test_device_status_clean():
    from attention_fa_attn_fwd_b300 import binding
    q, k, v = (t.cuda() for t in _inputs(1, 2, 2, 256, 256, 64))
    binding.attn_fwd(q, k, v, causal=True)
    assert binding.device_status() == 0


# ---- attn_fwd_ex with ATTN_FWD_EXP2_FMA (half of the exponentials on the FMA pipe)

def _run_fma(q, k, v, causal, scale=None):
    from attention_fa_attn_fwd_b300 import attn_fwd
    o, lse = attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, exp2_fma=True)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [17, 200, 383])
def test_exp2_fma_variant_ragged(d, causal, N):
    q, k, v = _inputs(1, 4, 2, N, N, d, seed=N + 7)
    o, lse = _run_fma(q, k, v, causal)
    O, L = oracle.attention_ref(f64(q), f64(k), f64(v), 1 / math.sqrt(d), causal)
    compare(f64(o), f64(lse), O, L, f"exp2-fma N={N} d={d} causal={causal}")


def test_exp2_fma_variant_masked_rows_and_peaky():
    q, k, v = _inputs(1, 2, 2, 300, 100, 128, seed=31)
    o, lse = _run_fma(q, k, v, True)
    assert torch.all(o[:, :, :200].float() == 0) and torch.all(torch.isneginf(lse[:, :, :200]))
    q, k, v = _inputs(1, 2, 2, 512, 512, 128, seed=32, gain=3.0)
    o, lse = _run_fma(q, k, v, True)
    O, L = oracle.attention_ref(f64(q), f64(k), f64(v), 1 / math.sqrt(128), True)
    compare(f64(o), f64(lse), O, L, "exp2-fma gain 3")


def test_exp2_fma_variant_workload_sampled_and_differs_from_default():
    cfg = workloads.PREFILL_WORKLOADS["gqa_b1h32kv8_n16384_d128_causal"]
    q, k, v = workloads.prefill_inputs(**cfg)
    o, lse = _run_fma(q, k, v, True)
    rows = sample_rows(cfg["Nq"], 256, seed=5)
    O, L = oracle.attention_ref(f64(q), f64(k), f64(v), 1 / math.sqrt(128), True, rows=rows)
    compare(f64(o[:, :, rows]), f64(lse[:, :, rows]), O, L, "exp2-fma gqa n16384")
    o2, _ = run_prefill(q[:, :, :512].contiguous(), k[:, :, :512].contiguous(),
                        v[:, :, :512].contiguous(), True)
    o3, _ = _run_fma(q[:, :, :512].contiguous(), k[:, :, :512].contiguous(),
                     v[:, :, :512].contiguous(), True)
    assert not torch.equal(o2, o3)  # the flag really switches the exponential


def test_long_context_64k_sampled():
    # 65536 keys: 256 K/V tiles per row block, 512 Q tiles per head
    q, k, v = _inputs(1, 4, 1, 65536, 65536, 128, seed=41)
    rows = sample_rows(65536, 24, seed=6)
    check_prefill(q, k, v, True, rows=rows, what="N=65536 causal")
