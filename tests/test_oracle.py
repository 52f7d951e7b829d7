"""Pins for the fp64 oracle (CPU only).

The oracle is the plain definition of attention; these tests tie it to facts
that do not come from the oracle itself: pure-Python brute force, closed
forms, invariants of softmax, a library routine in a special case, and the
single-pass recurrence restated independently.  ``test_oracle_mutants.py``
plants plausible mistakes in copies of the oracle and checks that these pins
catch each one.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_ref, attention_online, softmax_rows, scores
from attention_fa_attn_fwd_b300 import workloads


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- pin helpers
# Each pin takes the attention function under test, so the mutant tests can
# run the same pins against deliberately broken copies.

def brute_force(q, k, v, scale, causal):
    """Pure-Python double loop with math.fsum / math.exp (no numpy arithmetic)."""
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    G = H // Hkv
    O = [[[[0.0] * d for _ in range(Nq)] for _ in range(H)] for _ in range(B)]
    L = [[[0.0] * Nq for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            g = h // G
            for i in range(Nq):
                s = []
                for j in range(Nk):
                    if causal and j > i + (Nk - Nq):
                        continue
                    s.append((j, scale * math.fsum(float(q[b, h, i, t]) * float(k[b, g, j, t])
                                                   for t in range(d))))
                if not s:
                    O[b][h][i] = [0.0] * d
                    L[b][h][i] = -math.inf
                    continue
                m = max(x for _, x in s)
                e = [(j, math.exp(x - m)) for j, x in s]
                den = math.fsum(w for _, w in e)
                for t in range(d):
                    O[b][h][i][t] = math.fsum(w * float(v[b, g, j, t]) for j, w in e) / den
                L[b][h][i] = m + math.log(den)
    return np.array(O), np.array(L)


def pin_brute_force(fn, seed=0):
    for trial, (B, H, Hkv, Nq, Nk, d, causal) in enumerate([
            (1, 1, 1, 3, 5, 4, False), (1, 2, 1, 5, 5, 3, True), (2, 4, 2, 4, 7, 8, True),
            (1, 2, 2, 8, 8, 8, False), (1, 3, 1, 6, 4, 2, True), (1, 1, 1, 1, 8, 5, True)]):
        q = _rand((B, H, Nq, d), seed + 3 * trial)
        k = _rand((B, Hkv, Nk, d), seed + 3 * trial + 1)
        v = _rand((B, Hkv, Nk, d), seed + 3 * trial + 2)
        scale = 1.0 / math.sqrt(d)
        O, L = fn(q, k, v, scale, causal)
        Ob, Lb = brute_force(q, k, v, scale, causal)
        fin = np.isfinite(Lb)
        assert np.array_equal(np.isfinite(L), fin)
        assert np.max(np.abs(O - Ob)) <= 1e-12
        assert np.max(np.abs(L[fin] - Lb[fin])) <= 1e-12


def pin_closed_forms(fn):
    rng = np.random.default_rng(5)
    d = 6
    scale = 0.37
    # Nk == 1: the single key gets all the weight.
    q = rng.standard_normal((1, 2, 4, d)); k = rng.standard_normal((1, 2, 1, d))
    v = rng.standard_normal((1, 2, 1, d))
    O, L = fn(q, k, v, scale, False)
    assert np.allclose(O, np.broadcast_to(v, O.shape), atol=1e-14)
    assert np.allclose(L, scale * np.einsum("bhid,bhjd->bhi", q, k), atol=1e-14)
    # Causal row 0 (Nq == Nk): sees only key 0.
    q = rng.standard_normal((1, 1, 5, d)); k = rng.standard_normal((1, 1, 5, d))
    v = rng.standard_normal((1, 1, 5, d))
    O, L = fn(q, k, v, scale, True)
    assert np.allclose(O[0, 0, 0], v[0, 0, 0], atol=1e-14)
    assert abs(L[0, 0, 0] - scale * q[0, 0, 0] @ k[0, 0, 0]) < 1e-14
    # q == 0: uniform weights over the unmasked keys.
    q = np.zeros((1, 1, 5, d))
    O, L = fn(q, k, v, scale, True)
    for i in range(5):
        assert np.allclose(O[0, 0, i], v[0, 0, :i + 1].mean(axis=0), atol=1e-14)
        assert abs(L[0, 0, i] - math.log(i + 1)) < 1e-14


def pin_identical_keys(fn):
    rng = np.random.default_rng(7)
    d, Nk = 8, 9
    q = rng.standard_normal((1, 1, 3, d))
    k = np.broadcast_to(rng.standard_normal(d), (1, 1, Nk, d)).copy()
    v = rng.standard_normal((1, 1, Nk, d))
    O, L = fn(q, k, v, 0.5, False)
    for i in range(3):
        assert np.allclose(O[0, 0, i], v[0, 0].mean(axis=0), atol=1e-13)
        assert abs(L[0, 0, i] - (0.5 * q[0, 0, i] @ k[0, 0, 0] + math.log(Nk))) < 1e-13


def pin_dominant_key(fn):
    rng = np.random.default_rng(11)
    d, Nk = 8, 12
    q = rng.standard_normal((1, 1, 1, d))
    k = 0.1 * rng.standard_normal((1, 1, Nk, d))
    j = 7
    k[0, 0, j] = 60.0 * q[0, 0, 0] / (q[0, 0, 0] @ q[0, 0, 0])   # score 60 * scale above 0
    v = rng.standard_normal((1, 1, Nk, d))
    O, _ = fn(q, k, v, 1.0, False)
    assert np.allclose(O[0, 0, 0], v[0, 0, j], atol=1e-12)


def pin_causal_prefix(fn):
    rng = np.random.default_rng(13)
    for Nq, Nk in [(6, 6), (3, 7)]:
        d = 5
        q = rng.standard_normal((1, 1, Nq, d)); k = rng.standard_normal((1, 1, Nk, d))
        v = rng.standard_normal((1, 1, Nk, d))
        O, L = fn(q, k, v, 0.4, True)
        for i in range(Nq):
            n = i + 1 + (Nk - Nq)
            Oi, Li = fn(q[:, :, i:i + 1], k[:, :, :n], v[:, :, :n], 0.4, False)
            assert np.allclose(O[0, 0, i], Oi[0, 0, 0], atol=1e-13)
            assert abs(L[0, 0, i] - Li[0, 0, 0]) < 1e-13


def pin_gqa_equals_repeated_mha(fn):
    rng = np.random.default_rng(17)
    B, H, Hkv, N, d = 2, 6, 2, 5, 4
    q = rng.standard_normal((B, H, N, d)); k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    O, L = fn(q, k, v, 0.5, True)
    kr = np.repeat(k, H // Hkv, axis=1); vr = np.repeat(v, H // Hkv, axis=1)
    O2, L2 = fn(q, kr, vr, 0.5, True)
    assert np.allclose(O, O2, atol=1e-14) and np.allclose(L, L2, atol=1e-14)


def pin_torch_sdpa(fn):
    """Library special case: torch SDPA in float64 (Nq == Nk, so its top-left
    causal alignment coincides with the bottom-right reading)."""
    g = torch.Generator().manual_seed(3)
    for causal in (False, True):
        q = torch.randn(2, 4, 33, 16, generator=g, dtype=torch.float64)
        k = torch.randn(2, 2, 33, 16, generator=g, dtype=torch.float64)
        v = torch.randn(2, 2, 33, 16, generator=g, dtype=torch.float64)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k.repeat_interleave(2, 1), v.repeat_interleave(2, 1), is_causal=causal, scale=0.3)
        O, _ = fn(q.numpy(), k.numpy(), v.numpy(), 0.3, causal)
        assert np.max(np.abs(O - ref.numpy())) < 1e-12


def pin_lse_matches_logsumexp(fn):
    """lse equals scipy's logsumexp of the masked scaled scores."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(19)
    q = rng.standard_normal((1, 2, 6, 4)) * 3; k = rng.standard_normal((1, 1, 9, 4)) * 3
    v = rng.standard_normal((1, 1, 9, 4))
    _, L = fn(q, k, v, 0.7, True)
    for h in range(2):
        for i in range(6):
            n = i + 1 + 3
            ref = logsumexp(0.7 * (k[0, 0, :n] @ q[0, h, i]))
            assert abs(L[0, h, i] - ref) < 1e-12


ALL_PINS = [pin_brute_force, pin_closed_forms, pin_identical_keys, pin_dominant_key,
            pin_causal_prefix, pin_gqa_equals_repeated_mha, pin_torch_sdpa,
            pin_lse_matches_logsumexp]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_attention_ref_pins(pin):
    pin(attention_ref)


# ------------------------------------------------------------- stage pins

def test_softmax_rows_sum_to_one_and_shift_invariance():
    rng = np.random.default_rng(23)
    S = rng.standard_normal((7, 11)) * 5
    S[2, 3:] = -np.inf
    P, m, L = softmax_rows(S)
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(P >= 0) and np.all(P[2, 3:] == 0)
    c = np.array([0.0, 3.0, -7.5, 100.0, -100.0, 1e-3, 42.0])
    P2, m2, L2 = softmax_rows(S + c[:, None])
    assert np.allclose(P2, P, atol=1e-14)
    assert np.allclose(L2, L + c, atol=1e-12)
    assert np.allclose(m2, m + c, atol=1e-12)


def test_softmax_rows_all_masked_row():
    S = np.array([[-np.inf, -np.inf], [0.0, 1.0]])
    P, m, L = softmax_rows(S)
    assert np.all(P[0] == 0) and L[0] == -np.inf and m[0] == -np.inf
    assert abs(P[1, 1] - math.e / (1 + math.e)) < 1e-15


def test_no_keys_is_a_fully_masked_row():
    P, m, L = softmax_rows(np.zeros((3, 0)))
    assert P.shape == (3, 0) and np.all(np.isneginf(m)) and np.all(np.isneginf(L))
    O, L = oracle.paged_decode_ref(np.ones((1, 2, 4)), [np.zeros((0, 1, 4))],
                                   [np.zeros((0, 1, 4))], 0.5)
    assert np.all(O == 0) and np.all(np.isneginf(L))


def test_scores_mask_bottom_right():
    q = np.ones((3, 2)); k = np.ones((5, 2))
    S = scores(q, k, 1.0, True, np.arange(3), 3)
    # Nq=3, Nk=5: row i sees keys 0..i+2
    expect = np.array([[2, 2, 2, -np.inf, -np.inf], [2, 2, 2, 2, -np.inf], [2, 2, 2, 2, 2]])
    assert np.array_equal(S, expect)


def test_fully_masked_rows_when_nq_exceeds_nk():
    rng = np.random.default_rng(29)
    q = rng.standard_normal((1, 1, 6, 4)); k = rng.standard_normal((1, 1, 3, 4))
    v = rng.standard_normal((1, 1, 3, 4))
    O, L = attention_ref(q, k, v, 0.5, True)
    # rows 0..2 have limit i - 3 < 0: no keys
    assert np.all(O[0, 0, :3] == 0) and np.all(np.isneginf(L[0, 0, :3]))
    assert np.all(np.isfinite(L[0, 0, 3:]))
    Ob, Lb = brute_force(q, k, v, 0.5, True)
    assert np.max(np.abs(O - Ob)) < 1e-12


def test_rows_subset_matches_full():
    rng = np.random.default_rng(31)
    q = rng.standard_normal((2, 4, 40, 8)); k = rng.standard_normal((2, 2, 40, 8))
    v = rng.standard_normal((2, 2, 40, 8))
    O, L = attention_ref(q, k, v, 0.35, True)
    rows = np.array([0, 5, 17, 39])
    Os, Ls = attention_ref(q, k, v, 0.35, True, rows=rows)
    assert np.array_equal(Os, O[:, :, rows]) and np.array_equal(Ls, L[:, :, rows])


@pytest.mark.parametrize("chunk", [1, 3, 16, 64, 1000])
@pytest.mark.parametrize("tau", [None, 0.0, 8.0 * math.log(2.0)])
def test_online_recurrence_equals_definition(chunk, tau):
    rng = np.random.default_rng(37)
    q = rng.standard_normal((1, 4, 50, 16)) * 2; k = rng.standard_normal((1, 2, 70, 16)) * 2
    v = rng.standard_normal((1, 2, 70, 16))
    for causal in (False, True):
        O, L = attention_ref(q, k, v, 0.25, causal)
        O2, L2 = attention_online(q, k, v, 0.25, causal, chunk, tau=tau)
        assert np.max(np.abs(O - O2)) < 1e-12
        assert np.max(np.abs(L - L2)) < 1e-12


def test_online_recurrence_fully_masked_rows():
    rng = np.random.default_rng(41)
    q = rng.standard_normal((1, 1, 9, 4)); k = rng.standard_normal((1, 1, 4, 4))
    v = rng.standard_normal((1, 1, 4, 4))
    O, L = attention_ref(q, k, v, 0.5, True)
    O2, L2 = attention_online(q, k, v, 0.5, True, 2, tau=5.0)
    assert np.array_equal(np.isneginf(L), np.isneginf(L2))
    fin = np.isfinite(L)
    assert np.max(np.abs(O - O2)) < 1e-12 and np.max(np.abs(L[fin] - L2[fin])) < 1e-12


# ----------------------------------------------------------------- bf16 pins

def test_bf16_decode_known_patterns():
    bits = np.array([0x3F80, 0x4000, 0xC040, 0x3F81, 0x0001, 0x8000, 0x7F80, 0xFF80, 0x7F7F],
                    dtype=np.uint16)
    want = [1.0, 2.0, -3.0, 1.0 + 2.0 ** -7, 2.0 ** -133, -0.0, math.inf, -math.inf,
            (2 - 2.0 ** -7) * 2.0 ** 127]
    got = oracle.bf16_bits_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w
    assert math.copysign(1.0, got[5]) == -1.0
    assert np.isnan(oracle.bf16_bits_to_f64(np.array([0x7FC0], dtype=np.uint16))[0])


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(0)
    x = (torch.randn(10000, generator=g) * 100).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy()
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), x.double().numpy())


# ------------------------------------------------------------- paged pins

def _small_paged(**kw):
    base = dict(num_seqs=8, H=4, Hkv=2, d=16, block_size=16, min_len=40, max_len=100,
                group=4, shared_tokens=32, spare_frac=0.25)
    base.update(kw)
    return workloads.paged_decode_inputs(**base)


def _f64(t):
    return oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy())


def _logical_ref(pb, scale):
    ks, vs = zip(*(pb.logical_kv(s) for s in range(pb.num_seqs)))
    return oracle.paged_decode_ref(_f64(pb.q), [_f64(k) for k in ks], [_f64(v) for v in vs], scale)


def test_paged_matches_contiguous_attention():
    pb = _small_paged()
    scale = 0.25
    O, L = _logical_ref(pb, scale)
    for s in range(pb.num_seqs):
        k, v = pb.logical_kv(s)
        qq = _f64(pb.q[s])[None, :, None, :]                     # [1,H,1,d]
        kk = _f64(k).transpose(1, 0, 2)[None]                    # [1,Hkv,n,d]
        vv = _f64(v).transpose(1, 0, 2)[None]
        O2, L2 = attention_ref(qq, kk, vv, scale, False)
        assert np.allclose(O[s], O2[0, :, 0], atol=1e-14)
        assert np.allclose(L[s], L2[0, :, 0], atol=1e-14)


@pytest.mark.parametrize("perm_seed", [101, 202, 303])
def test_paged_pool_gather_independent_of_permutation(perm_seed):
    pb = _small_paged(perm_seed=perm_seed)
    scale = 0.25
    O, L = _logical_ref(pb, scale)
    O2, L2 = oracle.paged_decode_ref_from_pool(
        _f64(pb.q), _f64(pb.k_cache), _f64(pb.v_cache), pb.block_table.numpy(),
        pb.seq_lens.numpy(), pb.block_size, scale)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    assert np.all(np.isfinite(O2))      # NaN poison never read


def test_paged_sharing_does_not_change_results():
    shared = _small_paged(share=True)
    private = _small_paged(share=False)
    assert shared.num_blocks < private.num_blocks
    scale = 0.25
    Os, Ls = oracle.paged_decode_ref_from_pool(
        _f64(shared.q), _f64(shared.k_cache), _f64(shared.v_cache), shared.block_table.numpy(),
        shared.seq_lens.numpy(), 16, scale)
    Op, Lp = oracle.paged_decode_ref_from_pool(
        _f64(private.q), _f64(private.k_cache), _f64(private.v_cache), private.block_table.numpy(),
        private.seq_lens.numpy(), 16, scale)
    assert np.array_equal(Os, Op) and np.array_equal(Ls, Lp)
    # shared prefix really is shared: same physical ids across a group
    bt = shared.block_table.numpy()
    assert np.array_equal(bt[0, :2], bt[3, :2]) and not np.array_equal(bt[0, :2], bt[4, :2])


def test_paged_nan_poison_present_and_unused():
    pb = _small_paged()
    kc = _f64(pb.k_cache)
    assert np.isnan(kc).any()            # spares / tails are poisoned
    valid = 0
    for s in range(pb.num_seqs):
        n = int(pb.seq_lens[s])
        for t in range(n):
            phys = int(pb.block_table[s, t // 16])
            assert not np.isnan(kc[phys, :, t % 16]).any()
            valid += 1
    assert valid == pb.logical_tokens()


def test_paged_index_probe_exact_in_oracle():
    pb = _small_paged(index_probe=True, min_len=70, max_len=100)
    O, _ = _logical_ref(pb, 1.0 / math.sqrt(16))
    # bf16 rounding of the oracle output recovers the encoded index exactly
    Ob = torch.from_numpy(O).to(torch.bfloat16).double().numpy()
    for s in range(pb.num_seqs):
        t = (Ob[s, :, 0] - 1) * 64 + (Ob[s, :, 1] - 1)
        assert np.all(t == t[0])
        k, _ = pb.logical_kv(s)
        tgt = int(torch.argmax(k[:, 0, 0].float().abs()))
        assert t[0] == tgt
        assert np.array_equal(Ob[s, :, 2], 1 + np.arange(4) // 2)


def test_unique_token_count():
    pb = _small_paged()
    lens = pb.seq_lens.numpy()
    # every group of 4 shares 32 tokens: 3 * 32 logical tokens per group are not unique
    assert pb.unique_valid_tokens() == lens.sum() - 3 * 32 * (pb.num_seqs // 4)
