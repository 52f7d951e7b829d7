"""GPU parity of attn_bwd (C ABI) against the fp64 backward oracle.

The GPU path runs attn_fwd, then attn_bwd on its O and LSE; the oracle
differentiates the definition in float64 from the same bf16 Q, K, V, dO.
Both backward paths are checked: the default one (at d = 128 one fused
kernel, dQ through fp32 atomic adds) and ATTN_BWD_DETERMINISTIC (separate dQ
and dK/dV kernels).  Tolerances: ``tests/parity.py`` (GRAD_REL_RMS,
GRAD_MAX_REL).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa_attn_fwd_b300 import binding, workloads
from tests.parity import compare_grad, f64, sample_rows

pytestmark = pytest.mark.gpu


def _run(q, k, v, do, causal, scale=None, det=False):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = binding.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = binding.attn_bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale,
                                  deterministic=det)
    torch.cuda.synchronize()
    return dq.cpu(), dk.cpu(), dv.cpu()


def check_bwd(B, H, Hkv, Nq, Nk, d, causal, seed=0, gain=1.0, scale=None, what="",
              dets=(False, True)):
    q, k, v = workloads.prefill_inputs(B, H, Hkv, Nq, Nk, d, seed=seed, qk_gain=gain)
    do = workloads.grad_output(q.shape, seed=seed)
    sc = (1.0 / math.sqrt(d)) if scale is None else scale
    rq, rk, rv, _ = oracle.attention_bwd_ref(f64(q), f64(k), f64(v), f64(do), sc, causal)
    for det in dets:
        tag = f"{what} {'deterministic' if det else 'default'}"
        dq, dk, dv = _run(q, k, v, do, causal, scale, det)
        compare_grad(f64(dq), rq, f"dq {tag}")
        compare_grad(f64(dk), rk, f"dk {tag}")
        compare_grad(f64(dv), rv, f"dv {tag}")


@pytest.mark.parametrize("causal", [False, True])
def test_tiny(causal):
    check_bwd(1, 2, 2, 128, 128, 64, causal, what="tiny")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 200, 383])
def test_ragged_lengths(d, causal, N):
    check_bwd(1, 2, 1, N, N, d, causal, seed=N + d, what=f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 100), (1, 257), (256, 640), (64, 64),
                                   (65, 1000), (1000, 65)])
@pytest.mark.parametrize("causal", [False, True])
def test_unequal_lengths(Nq, Nk, causal):
    check_bwd(2, 4, 2, Nq, Nk, 128, causal, seed=Nq + 3 * Nk, what=f"Nq={Nq} Nk={Nk}")


@pytest.mark.parametrize("H,Hkv", [(8, 1), (8, 2), (6, 3), (16, 1)])
def test_gqa(H, Hkv):
    check_bwd(1, H, Hkv, 384, 384, 128, True, seed=H + Hkv, what=f"H={H} Hkv={Hkv}")


def test_peaky_and_nondefault_scale():
    check_bwd(1, 2, 2, 512, 512, 128, True, seed=21, gain=2.0, what="gain 2")
    check_bwd(1, 2, 2, 256, 256, 64, False, seed=22, scale=0.05, what="scale 0.05")


def test_mid_size_causal_gqa():
    check_bwd(1, 8, 2, 1024, 1024, 128, True, seed=23, what="B1 H8 Hkv2 N1024")


def test_multi_batch_many_tiles():
    # several batches and KV heads, more CTAs than SMs, non-causal and causal
    check_bwd(3, 8, 4, 640, 640, 128, False, seed=31, what="B3 H8 Hkv4 N640 full")
    check_bwd(3, 8, 4, 640, 640, 128, True, seed=32, what="B3 H8 Hkv4 N640 causal")


@pytest.mark.parametrize("d", [64, 128])
def test_fully_masked_rows_give_zero_dq(d):
    q, k, v = workloads.prefill_inputs(1, 2, 2, 300, 100, d, seed=9)
    do = workloads.grad_output(q.shape, seed=9)
    rq, rk, rv, _ = oracle.attention_bwd_ref(f64(q), f64(k), f64(v), f64(do), 1 / math.sqrt(d),
                                             True)
    for det in (False, True):
        dq, dk, dv = _run(q, k, v, do, True, det=det)
        assert torch.all(dq[:, :, :200].float() == 0)
        compare_grad(f64(dq), rq, f"dq masked rows d={d} det={det}")
        compare_grad(f64(dk), rk, f"dk masked rows d={d} det={det}")
        compare_grad(f64(dv), rv, f"dv masked rows d={d} det={det}")


def test_deterministic_and_status_clean():
    q, k, v = (t.cuda() for t in workloads.prefill_inputs(2, 4, 2, 700, 700, 128, seed=13))
    do = workloads.grad_output(q.shape, seed=13).cuda()
    o, lse = binding.attn_fwd(q, k, v, causal=True)
    # ATTN_BWD_DETERMINISTIC: identical bits on repeat
    a = binding.attn_bwd(q, k, v, o, do, lse, causal=True, deterministic=True)
    b = binding.attn_bwd(q, k, v, o, do, lse, causal=True, deterministic=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    # default path: dk and dv accumulate in a fixed order (identical bits);
    # dq sums key tiles' shares in arrival order, so only fp32 rounding differs
    c = binding.attn_bwd(q, k, v, o, do, lse, causal=True)
    e = binding.attn_bwd(q, k, v, o, do, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(c[1], e[1]) and torch.equal(c[2], e[2])
    rel = ((c[0].float() - e[0].float()).norm() / e[0].float().norm()).item()
    assert rel < 1e-3, rel
    assert binding.device_status() == binding.ATTN_OK


def test_long_context_gqa_sampled():
    """The long-context causal GQA workload the backward is timed on
    (B1 H32 Hkv8 N16384 d128, Q and K x1.5): dQ on 64 seeded query rows of
    every head, dK and dV on 64 seeded key rows of two seeded KV groups.
    Every key row's gradient sums over all 16384 queries of the 4 heads of its
    group, so this covers the long accumulation in dK/dV, the multi-wave grids
    and the long key loop of dQ."""
    cfg = workloads.PREFILL_WORKLOADS["gqa_b1h32kv8_n16384_d128_causal"]
    q, k, v = workloads.prefill_inputs(**cfg)
    do = workloads.grad_output(q.shape, seed=0)
    N, d = cfg["Nq"], cfg["d"]
    qr = sample_rows(N, 64, seed=101)
    kr = sample_rows(N, 64, seed=102)
    groups = sorted(np.random.default_rng(103).choice(cfg["Hkv"], size=2, replace=False).tolist())
    pairs = [(0, g) for g in groups]
    rq, rk, rv = oracle.attention_bwd_rows(f64(q), f64(k), f64(v), f64(do), 1 / math.sqrt(d),
                                           True, qr, kr, pairs)
    for det in (False, True):
        tag = "deterministic" if det else "default"
        dq, dk, dv = _run(q, k, v, do, True, det=det)
        compare_grad(f64(dq[:, :, qr]), rq, f"dq long-context {tag} (64 rows x 32 heads)")
        for n, (b, g) in enumerate(pairs):
            compare_grad(f64(dk[b, g, kr]), rk[n], f"dk long-context {tag} group {g} (64 rows)")
            compare_grad(f64(dv[b, g, kr]), rv[n], f"dv long-context {tag} group {g} (64 rows)")
