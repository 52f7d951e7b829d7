"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding, run the fp64 oracle on the same seeded inputs, compare.

Tolerances (fixed for the bf16-in / fp32-accumulate path):
  O:   max |o - o_ref| <= 2e-2  and  ||o - o_ref||_2 / ||o_ref||_2 <= 5e-3
  LSE: max |lse - lse_ref| <= 1e-3 (natural log, fp32); -inf exactly where the
       oracle has no unmasked key (and o = 0 there).
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle

O_MAX_ABS = 2e-2
O_REL_RMS = 5e-3
LSE_MAX_ABS = 1e-3

# Gradients (attn_bwd): P and dS are rounded to bf16 before their matrix
# products and dq/dk/dv are rounded to bf16 on output -- three rounding stages
# of relative RMS about 2^-7/sqrt(12) ~ 2.3e-3 each, plus the forward's
# rounded O (through D) and its LSE error (<= 1e-3 relative in P).  Bounds:
#   ||g - g_ref||_2 / ||g_ref||_2 <= 1e-2
#   max |g - g_ref| <= 2e-2 * max(max |g_ref|, 1e-2)
# The 1e-2 floor covers gradients that vanish in exact arithmetic (a single
# key: dS = P (dP - D) = 0), where only rounding residue of order
# |dO| |V| 2^-8 * 1e-4 remains; with N(0,1) inputs real gradients are O(0.1-1).
GRAD_REL_RMS = 1e-2
GRAD_MAX_REL = 2e-2
GRAD_FLOOR = 1e-2


# (label, statistics) of every comparison made in this process; printed at the
# end of a pytest run by conftest.py (and written to $PARITY_STATS_OUT if set).
RECORDED = []


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact bf16 -> float64 through the oracle's own decoder."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(t.view(torch.int16).numpy())
    return t.double().numpy()


def sample_rows(Nq: int, n: int, seed: int) -> np.ndarray:
    """n seeded query rows, always including the first and the last row."""
    if n >= Nq:
        return np.arange(Nq)
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(Nq, size=n - 2, replace=False).tolist()) | {0, Nq - 1}
    return np.array(sorted(rows))


def compare(o_gpu: np.ndarray, lse_gpu, O_ref: np.ndarray, L_ref, what: str = ""):
    """Assert the tolerances; return a dict of error statistics."""
    assert o_gpu.shape == O_ref.shape, (o_gpu.shape, O_ref.shape)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    diff = o_gpu - O_ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.sqrt(np.sum(O_ref ** 2)))
    rel_rms = float(np.sqrt(np.sum(diff ** 2)) / den) if den > 0 else float(np.sqrt(np.sum(diff ** 2)))
    stats = {"o_max_abs": max_abs, "o_rel_rms": rel_rms}
    if L_ref is not None:
        fin = np.isfinite(L_ref)
        assert np.array_equal(np.isfinite(lse_gpu), fin), f"{what}: -inf pattern differs"
        assert np.all(np.isneginf(lse_gpu[~fin])), f"{what}: masked rows must have lse = -inf"
        lse_err = float(np.max(np.abs(lse_gpu[fin] - L_ref[fin]))) if fin.any() else 0.0
        stats["lse_max_abs"] = lse_err
        assert lse_err <= LSE_MAX_ABS, f"{what}: lse max abs {lse_err}"
    RECORDED.append((what, stats))
    assert max_abs <= O_MAX_ABS, f"{what}: O max abs {max_abs} ({stats})"
    assert rel_rms <= O_REL_RMS, f"{what}: O rel rms {rel_rms} ({stats})"
    return stats


def run_prefill(q, k, v, causal, scale=None):
    """Run attn_fwd on the GPU; returns (o, lse) as CPU tensors."""
    from attention_fa_attn_fwd_b300 import attn_fwd
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def check_prefill(q, k, v, causal, rows=None, scale=None, what=""):
    """GPU attn_fwd vs the oracle on all rows, or on the given query rows."""
    d = q.shape[-1]
    scale = (1.0 / math.sqrt(d)) if scale is None else scale
    o, lse = run_prefill(q, k, v, causal, scale)
    rr = np.arange(q.shape[2]) if rows is None else np.asarray(rows)
    O_ref, L_ref = oracle.attention_ref(f64(q), f64(k), f64(v), scale, causal, rows=rr)
    return compare(f64(o[:, :, rr]), f64(lse[:, :, rr]), O_ref, L_ref, what)


def compare_grad(g: np.ndarray, g_ref: np.ndarray, what: str = ""):
    """Assert the gradient tolerances; return error statistics."""
    assert g.shape == g_ref.shape, (g.shape, g_ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite gradient"
    diff = g - g_ref
    ref_max = float(np.max(np.abs(g_ref))) if g_ref.size else 0.0
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.sqrt(np.sum(g_ref ** 2)))
    floor = GRAD_FLOOR * np.sqrt(g_ref.size)
    rel_rms = float(np.sqrt(np.sum(diff ** 2)) / max(den, floor))
    stats = {"max_abs": max_abs, "ref_max": ref_max, "rel_rms": rel_rms}
    RECORDED.append((what, stats))
    assert rel_rms <= GRAD_REL_RMS, f"{what}: rel rms {rel_rms} ({stats})"
    assert max_abs <= GRAD_MAX_REL * max(ref_max, GRAD_FLOOR), f"{what}: max abs {max_abs} ({stats})"
    return stats
