"""Pins for the chunked paged-prefill oracle (CPU only).

``oracle.paged_prefill_ref`` applies the definition per sequence with the
causal mask aligned to the end of the cache.  It is tied here to facts that do
not come from it: pure-Python brute force, the equivalence of a chunk with the
last rows of one causal pass over the whole sequence, decode as the
one-token special case, and the block-table gather under any permutation.
A planted mistake (the other causal alignment, a dropped history) must fail a
pin.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa_attn_fwd_b300 import workloads
from tests.test_oracle import brute_force


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _case(seed, S=3, H=4, Hkv=2, Nq=5, d=4, lens=(5, 9, 12)):
    q = _rand((S, H, Nq, d), seed)
    ks = [_rand((n, Hkv, d), seed + 10 + s) for s, n in enumerate(lens)]
    vs = [_rand((n, Hkv, d), seed + 20 + s) for s, n in enumerate(lens)]
    return q, ks, vs


def pin_brute_force(fn):
    for seed, lens, causal in [(0, (5, 9, 12), True), (1, (5, 6, 7), False),
                               (2, (2, 5, 11), True), (3, (1, 3, 8), True)]:
        q, ks, vs = _case(seed, lens=lens)
        scale = 1.0 / math.sqrt(q.shape[-1])
        O, L = fn(q, ks, vs, scale, causal)
        for s in range(q.shape[0]):
            kk = ks[s].transpose(1, 0, 2)[None]
            vv = vs[s].transpose(1, 0, 2)[None]
            Ob, Lb = brute_force(q[s][None], kk, vv, scale, causal)
            fin = np.isfinite(Lb[0])
            assert np.array_equal(np.isfinite(L[s]), fin)
            assert np.max(np.abs(O[s] - Ob[0])) <= 1e-12
            assert np.max(np.abs(L[s][fin] - Lb[0][fin])) <= 1e-12


def pin_chunk_equals_last_rows_of_full_pass(fn):
    # One causal pass over n tokens, then the last Nq rows: a chunked prefill
    # of those Nq tokens over the same cache must give the same rows.
    rng = np.random.default_rng(7)
    H, Hkv, d, n, Nq = 4, 2, 8, 37, 11
    qf = rng.standard_normal((1, H, n, d))
    k = rng.standard_normal((n, Hkv, d))
    v = rng.standard_normal((n, Hkv, d))
    scale = 0.3
    Of, Lf = oracle.attention_ref(qf, k.transpose(1, 0, 2)[None], v.transpose(1, 0, 2)[None],
                                  scale, True, rows=np.arange(n - Nq, n))
    O, L = fn(qf[:, :, n - Nq:], [k], [v], scale, True)
    assert np.max(np.abs(O[0] - Of[0])) <= 1e-12
    assert np.max(np.abs(L[0] - Lf[0])) <= 1e-12


def pin_one_token_chunk_is_decode(fn):
    q, ks, vs = _case(4, Nq=1, lens=(3, 17, 40))
    scale = 0.5
    O, L = fn(q, ks, vs, scale, True)
    Od, Ld = oracle.paged_decode_ref(q[:, :, 0], ks, vs, scale)
    assert np.max(np.abs(O[:, :, 0] - Od)) <= 1e-12
    assert np.max(np.abs(L[:, :, 0] - Ld)) <= 1e-12


def pin_short_cache_masks_leading_rows(fn):
    # seq_len < Nq: row i sees keys j <= i + seq_len - Nq; rows with none are 0 / -inf.
    q, ks, vs = _case(5, Nq=6, lens=(4, 6, 6))
    O, L = fn(q, ks, vs, 0.4, True)
    assert np.all(O[0, :, :2] == 0) and np.all(np.isneginf(L[0, :, :2]))
    assert np.all(np.isfinite(L[0, :, 2:]))
    # row 2 of sequence 0 sees only key 0: O = v_0, lse = score
    G = q.shape[1] // ks[0].shape[1]
    for h in range(q.shape[1]):
        assert np.allclose(O[0, h, 2], vs[0][0, h // G], atol=1e-14)
        assert np.isclose(L[0, h, 2], 0.4 * q[0, h, 2] @ ks[0][0, h // G], atol=1e-14)


PAGED_PREFILL_PINS = [pin_brute_force, pin_chunk_equals_last_rows_of_full_pass,
                      pin_one_token_chunk_is_decode, pin_short_cache_masks_leading_rows]


@pytest.mark.parametrize("pin", PAGED_PREFILL_PINS, ids=lambda p: p.__name__)
def test_paged_prefill_ref_pins(pin):
    pin(oracle.paged_prefill_ref)


def _f64(t):
    return oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy())


@pytest.mark.parametrize("perm_seed", [None, 5, 6])
def test_gather_through_pool_matches_logical(perm_seed):
    pb = workloads.paged_prefill_inputs(num_seqs=3, H=4, Hkv=2, d=16, Nq=20, min_hist=0,
                                        max_hist=50, seed=1, perm_seed=perm_seed)
    scale = 0.25
    ks = oracle.gather_logical_kv(_f64(pb.k_cache), pb.block_table.numpy(), pb.seq_lens.numpy(), 16)
    vs = oracle.gather_logical_kv(_f64(pb.v_cache), pb.block_table.numpy(), pb.seq_lens.numpy(), 16)
    O, L = oracle.paged_prefill_ref(_f64(pb.q), ks, vs, scale, True)
    lk = [_f64(pb.logical_kv(s)[0]) for s in range(3)]
    lv = [_f64(pb.logical_kv(s)[1]) for s in range(3)]
    O2, L2 = oracle.paged_prefill_ref(_f64(pb.q), lk, lv, scale, True)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    assert np.all(np.isfinite(O))  # the NaN-poisoned slots are never read


def _mutant(kind):
    def fn(q, ks, vs, scale, causal, rows=None):
        S_, H, Nq, d = q.shape
        O = np.zeros((S_, H, Nq, d))
        L = np.zeros((S_, H, Nq))
        for s in range(S_):
            k = ks[s][-Nq:] if kind == "drop_history" else ks[s]
            v = vs[s][-Nq:] if kind == "drop_history" else vs[s]
            n, Hkv, _ = k.shape
            G = H // Hkv
            for h in range(H):
                Sm = scale * q[s, h] @ k[:, h // G].T
                if causal:
                    i = np.arange(Nq)[:, None]
                    j = np.arange(n)[None, :]
                    lim = i if kind == "top_left" else i + n - Nq
                    Sm = np.where(j > lim, -np.inf, Sm)
                P, _, lse = oracle.softmax_rows(Sm)
                O[s, h] = P @ v[:, h // G]
                L[s, h] = lse
        return O, L
    return fn


@pytest.mark.parametrize("kind", ["top_left", "drop_history"])
def test_pins_catch_paged_prefill_mutant(kind):
    caught = []
    for pin in PAGED_PREFILL_PINS:
        try:
            pin(_mutant(kind))
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, kind


def test_mutant_harness_itself_passes_when_correct():
    for pin in PAGED_PREFILL_PINS:
        pin(_mutant("none"))
