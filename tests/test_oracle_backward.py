"""Pins for the fp64 backward oracle (CPU only).

``oracle.attention_bwd_ref`` writes out the chain rule of the forward
definition.  It is tied here to facts that do not come from it: central finite
differences of the forward oracle (itself pinned by brute force), torch
autograd through float64 scaled_dot_product_attention (a library special
case), and identities that follow from softmax rows summing to one.  Planted
mistakes (a dropped softmax-Jacobian term, a sign, a scale, a transposed dS, a
GQA head that overwrites instead of accumulating) must each fail a pin.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle.attention import scores, softmax_rows


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _case(seed, B=1, H=2, Hkv=1, Nq=4, Nk=5, d=3):
    return (_rand((B, H, Nq, d), seed), _rand((B, Hkv, Nk, d), seed + 1),
            _rand((B, Hkv, Nk, d), seed + 2), _rand((B, H, Nq, d), seed + 3))


def pin_finite_differences(fn):
    for seed, shape, causal in [(0, dict(), False), (4, dict(), True),
                                (8, dict(H=4, Hkv=2, Nq=5, Nk=3, d=2), True),
                                (12, dict(Nq=3, Nk=3, d=4), True)]:
        q, k, v, do = _case(seed, **shape)
        scale = 0.7
        dq, dk, dv, _ = fn(q, k, v, do, scale, causal)

        def loss(q_, k_, v_):
            O, _ = oracle.attention_ref(q_, k_, v_, scale, causal)
            return float(np.sum(O * do))

        eps = 1e-6
        for x, g in ((q, dq), (k, dk), (v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + eps
                lp = loss(q, k, v)
                x[idx] = old - eps
                lm = loss(q, k, v)
                x[idx] = old
                num[idx] = (lp - lm) / (2 * eps)
            assert np.max(np.abs(num - g)) <= 1e-7, (seed, np.max(np.abs(num - g)))


def pin_torch_autograd(fn):
    for seed, (H, Hkv, N, d), causal in [(20, (2, 2, 6, 4), True), (24, (4, 2, 7, 3), False),
                                         (28, (4, 1, 5, 8), True)]:
        q, k, v, do = _case(seed, H=H, Hkv=Hkv, Nq=N, Nk=N, d=d)
        scale = 1.0 / math.sqrt(d)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        G = H // Hkv
        o = torch.nn.functional.scaled_dot_product_attention(
            tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1),
            is_causal=causal, scale=scale)
        o.backward(torch.tensor(do))
        dq, dk, dv, _ = fn(q, k, v, do, scale, causal)
        assert np.max(np.abs(tq.grad.numpy() - dq)) <= 1e-10
        assert np.max(np.abs(tk.grad.numpy() - dk)) <= 1e-10
        assert np.max(np.abs(tv.grad.numpy() - dv)) <= 1e-10


def pin_row_sum_identities(fn):
    # Rows of P sum to 1, so rows of dS sum to 0: sum over keys of dK is 0,
    # and sum over keys of dV is the sum of dO over the rows that see a key.
    q, k, v, do = _case(40, B=2, H=4, Hkv=2, Nq=9, Nk=6, d=5)
    dq, dk, dv, D = fn(q, k, v, do, 0.5, True)
    assert np.max(np.abs(dk.sum(axis=2))) <= 1e-12
    G = 2
    for b in range(2):
        for g in range(2):
            seen = np.arange(9) + (6 - 9) >= 0  # bottom-right: rows 0..2 see no key
            want = sum(do[b, h][seen].sum(axis=0) for h in range(g * G, (g + 1) * G))
            assert np.allclose(dv[b, g].sum(axis=0), want, atol=1e-12)
    # D_i = rowsum(dO_i * O_i)
    O, _ = oracle.attention_ref(q, k, v, 0.5, True)
    assert np.allclose(D, np.sum(O * do, axis=-1), atol=1e-12)
    # dQ of a row that sees no key is 0
    assert np.all(dq[:, :, :3] == 0)


BACKWARD_PINS = [pin_finite_differences, pin_torch_autograd, pin_row_sum_identities]


@pytest.mark.parametrize("pin", BACKWARD_PINS, ids=lambda p: p.__name__)
def test_backward_ref_pins(pin):
    pin(oracle.attention_bwd_ref)


def _mutant(kind):
    def fn(q, k, v, do, scale, causal):
        B, H, Nq, d = q.shape
        Hkv, Nk = k.shape[1], k.shape[2]
        G = H // Hkv
        dq = np.zeros_like(q)
        dk = np.zeros_like(k)
        dv = np.zeros_like(v)
        D = np.zeros((B, H, Nq))
        for b in range(B):
            for h in range(H):
                g = h // G
                S = scores(q[b, h], k[b, g], scale, causal, np.arange(Nq), Nq)
                P, _, _ = softmax_rows(S)
                pv = P.T @ do[b, h]
                if kind == "gqa_overwrite":
                    dv[b, g] = pv
                else:
                    dv[b, g] += pv
                dP = do[b, h] @ v[b, g].T
                Dh = np.sum(P * dP, axis=1)
                if kind == "drop_D":
                    Dh = 0 * Dh
                dS = P * (dP - Dh[:, None])
                if kind == "sign":
                    dS = -dS
                if kind == "transposed_dS" and Nq == Nk:
                    dS = dS.T
                dq[b, h] = scale * (dS @ k[b, g])
                dk[b, g] += (1.0 if kind == "dk_no_scale" else scale) * (dS.T @ q[b, h])
                D[b, h] = Dh
        return dq, dk, dv, D
    return fn


@pytest.mark.parametrize("kind", ["gqa_overwrite", "drop_D", "sign", "transposed_dS",
                                  "dk_no_scale"])
def test_pins_catch_backward_mutant(kind):
    caught = []
    for pin in BACKWARD_PINS:
        try:
            pin(_mutant(kind))
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, kind


def test_mutant_harness_passes_when_correct():
    for pin in BACKWARD_PINS:
        pin(_mutant("none"))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,row_slice", [(1, 4, 2, 9, 9, 4, 4), (2, 6, 3, 7, 11, 3, 3),
                                                      (1, 2, 1, 12, 5, 5, 5), (1, 4, 1, 6, 6, 8, 100)])
def test_rows_variant_equals_autograd_rows(causal, B, H, Hkv, Nq, Nk, d, row_slice):
    """attention_bwd_rows on chosen rows equals float64 torch autograd through
    scaled_dot_product_attention (a library special case, independent of the
    oracle) on the same rows, and the full chain-rule oracle."""
    rng = np.random.default_rng(Nq * 31 + Nk + d)
    q = rng.standard_normal((B, H, Nq, d))
    k = rng.standard_normal((B, Hkv, Nk, d))
    v = rng.standard_normal((B, Hkv, Nk, d))
    do = rng.standard_normal((B, H, Nq, d))
    scale = 0.6
    qr = np.array(sorted(rng.choice(Nq, size=min(Nq, 4), replace=False)))
    kr = np.array(sorted(rng.choice(Nk, size=min(Nk, 3), replace=False)))
    pairs = [(b, g) for b in range(B) for g in range(Hkv)][::-1]
    dq, dk, dv = oracle.attention_bwd_rows(q, k, v, do, scale, causal, qr, kr, pairs,
                                           row_slice=row_slice)
    # torch's is_causal is top-left aligned; build the bottom-right mask explicitly
    G = H // Hkv
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    mask = None
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        allowed = j <= i + (Nk - Nq)
        mask = torch.where(allowed, 0.0, float("-inf")).double()
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1), attn_mask=mask,
        scale=scale)
    # rows with no key give NaN in torch; their gradient is 0 by the reading
    o = torch.nan_to_num(o)
    o.backward(torch.tensor(do))
    gq, gk, gv = (torch.nan_to_num(t.grad).numpy() for t in (tq, tk, tv))
    assert np.max(np.abs(dq - gq[:, :, qr])) <= 1e-10
    for n, (b, g) in enumerate(pairs):
        assert np.max(np.abs(dk[n] - gk[b, g, kr])) <= 1e-10
        assert np.max(np.abs(dv[n] - gv[b, g, kr])) <= 1e-10
    fq, fk, fv, _ = oracle.attention_bwd_ref(q, k, v, do, scale, causal)
    assert np.max(np.abs(dq - fq[:, :, qr])) <= 1e-12
    for n, (b, g) in enumerate(pairs):
        assert np.max(np.abs(dk[n] - fk[b, g, kr])) <= 1e-12
        assert np.max(np.abs(dv[n] - fv[b, g, kr])) <= 1e-12
