"""The FMA-pipe exp2 of attn_fwd_ex (CPU only).

The kernel's constants are the least-squares cubic written by
``csrc/fit_exp2_poly.py``.  Here the header is parsed, the kernel's steps
(clamp, round to the nearest integer by adding 1.5 * 2^23, reduced argument
f, Horner in float32, exponent-field add, zero below -126) are replayed in
numpy float32, and the result is compared with 2^x in float64.
"""

import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_fa_attn_fwd_b300", "csrc")


def header_coeffs():
    text = open(os.path.join(CSRC, "exp2_poly.h")).read()
    vals = dict(re.findall(r"kExp2Poly(\d) = ([-0-9.e]+)f;", text))
    return np.array([float(vals[str(j)]) for j in range(4)], dtype=np.float32)


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fma32(a, b, c):
    # a*b is exact in float64 for float32 inputs; one rounding to float32
    return f32(a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64))


def exp2_fma_replay(x):
    c = header_coeffs()
    x = np.maximum(f32(x), np.float32(-127.0))
    magic = np.float32(12582912.0)
    j = f32(x.astype(np.float64) + magic)
    n = f32(j.astype(np.float64) - magic)
    f = fma32(n, np.full_like(n, -1.0), x)
    p = fma32(np.full_like(f, c[3]), f, np.full_like(f, c[2]))
    p = fma32(p, f, np.full_like(f, c[1]))
    p = fma32(p, f, np.full_like(f, c[0]))
    bits = (p.view(np.int32).astype(np.int64) + (j.view(np.int32).astype(np.int64) << 23)) \
        & 0xFFFFFFFF
    r = bits.astype(np.uint32).view(np.float32)
    return np.where(x < -126.0, np.float32(0.0), r)


def test_relative_error_over_the_softmax_range():
    # normal results (x >= -125): relative error of the cubic only
    x = np.linspace(-125.0, 10.0, 2_000_001)
    got = exp2_fma_replay(x).astype(np.float64)
    want = np.exp2(f32(x).astype(np.float64))
    rel = np.abs(got / want - 1)
    assert rel.max() < 1e-4, rel.max()
    # [-126, -125): results near the bottom of the float range, absolute error tiny
    x = np.linspace(-126.0, -125.0, 10_001)
    err = np.abs(exp2_fma_replay(x).astype(np.float64) - np.exp2(f32(x).astype(np.float64)))
    assert err.max() < 2.0 ** -137


def test_exact_integers_and_zero_below_range():
    x = np.arange(-125, 11, dtype=np.float64)
    got = exp2_fma_replay(x).astype(np.float64)
    assert np.max(np.abs(got / np.exp2(x) - 1)) < 1e-4
    assert np.all(exp2_fma_replay(np.array([-126.5, -200.0, -np.inf])) == 0)


def test_header_matches_a_fresh_fit():
    spec = importlib.util.spec_from_file_location("fit", os.path.join(CSRC, "fit_exp2_poly.py"))
    fit = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fit)
    c = fit.fit().astype(np.float32)
    assert np.array_equal(c, header_coeffs())
    assert fit.check(c) < fit.MAX_REL
