"""fp64 reference for exact scaled dot-product attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may use this module; the CUDA path never does.

Sources (page title, then the part of the page):

* Interview notes "他人面经整理", answer "介绍你理解的flashattention", part 1:
  self-attention is Softmax(Q K^T / sqrt(d_k)) V, and the naive implementation
  materialises S = Q K^T (N x N) and P = softmax(S) before multiplying by V.
* Same answer, part 2, "Online Softmax": per query row keep the running maximum
  m_i and the running sum l_i of exp(x - m_i); on each new block of scores
  rescale l and the partial output by exp(m_old - m_new), add the block's
  exp-sum and P_ij V_j; the single pass reaches the exact softmax.
* FAQ page "Wie unterscheidet sich die Implementierung von FlashAttention-2 ...
  von der Standard-Attention-Berechnung ...", comparison table: the standard
  computation builds the full N x N matrix; FlashAttention-2 reaches the same
  result incrementally (online softmax) without storing it.

Readings where the pages are silent (the same readings hold for the kernels):

* ``scale`` is an argument; the definition's value is 1/sqrt(d).
* Causal masking is bottom-right aligned: query row i (0-based) may attend key
  j iff j <= i + (Nk - Nq).  For Nq == Nk this is the usual j <= i.
* GQA: query head h reads key/value head h // (H / Hkv).
* The log-sum-exp output is lse_i = m_i + ln(sum_j exp(S_ij - m_i)) over the
  scaled, masked scores, natural logarithm.
* A row whose keys are all masked has no softmax; its output row is 0 and its
  lse is -inf.

The oracle is the plain definition, written out with numpy in float64; S and P
are materialised, nothing is blocked, fused or reordered.
"""

from __future__ import annotations

import numpy as np


def causal_limit(i, Nq: int, Nk: int):
    """Largest key index query row ``i`` may attend under the causal mask.

    Bottom-right alignment (reading stated in the module docstring): the last
    query row sees every key, row i sees keys 0 .. i + (Nk - Nq).
    """
    return np.asarray(i) + (Nk - Nq)


def scores(q_rows: np.ndarray, k: np.ndarray, scale: float, causal: bool,
           row_idx: np.ndarray, Nq: int) -> np.ndarray:
    """S = scale * Q K^T with the causal mask applied as -inf.

    q_rows: [R, d] float64, the query rows numbered ``row_idx`` (length R) in a
    sequence of Nq queries.  k: [Nk, d] float64.  Returns S: [R, Nk].
    Interview notes "他人面经整理", flashattention answer part 1 (S = QK^T,
    scaled by 1/sqrt(d_k)).
    """
    S = scale * (q_rows @ k.T)
    if causal:
        Nk = k.shape[0]
        lim = causal_limit(np.asarray(row_idx), Nq, Nk)
        j = np.arange(Nk)
        S = np.where(j[None, :] > lim[:, None], -np.inf, S)
    return S


def softmax_rows(S: np.ndarray):
    """Row softmax of S with its row maximum and natural log-sum-exp.

    Returns (P, m, lse) where m_i = max_j S_ij, P_ij = exp(S_ij - m_i) /
    sum_j exp(S_ij - m_i) and lse_i = m_i + ln sum_j exp(S_ij - m_i).
    Rows that are entirely -inf, and rows of a zero-width S (no keys), give
    P = 0, m = -inf, lse = -inf.
    Interview notes "他人面经整理", flashattention answer part 2 (m_i is the row
    maximum, l_i the sum of exp(x - m_i)).
    """
    if S.shape[1] == 0:  # no keys at all: same as a fully masked row
        R = S.shape[0]
        return np.zeros((R, 0)), np.full(R, -np.inf), np.full(R, -np.inf)
    m = S.max(axis=1)
    dead = ~np.isfinite(m)
    m_safe = np.where(dead, 0.0, m)
    E = np.exp(S - m_safe[:, None])
    l = E.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(dead[:, None], 0.0, E / np.where(dead, 1.0, l)[:, None])
        lse = np.where(dead, -np.inf, m_safe + np.log(np.where(dead, 1.0, l)))
    return P, m, lse


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d] / [B, Hkv, N, d]")
    B, H, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    if Hkv <= 0 or H % Hkv:
        raise ValueError(f"H={H} is not a multiple of Hkv={Hkv}")
    return B, H, Hkv, Nq, Nk, d


def attention_ref(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                  causal: bool, rows=None):
    """Plain attention O = softmax(scale Q K^T [masked]) V and per-row lse.

    q: [B, H, Nq, d]; k, v: [B, Hkv, Nk, d] (float64; bf16 inputs decode
    exactly).  rows: optional 1-D array of query-row indices evaluated for
    every (b, h); default all Nq rows.  Returns O [B, H, R, d] and lse
    [B, H, R] in float64.

    Steps, in the order of the definition (Interview notes "他人面经整理",
    flashattention answer part 1): S = scale Q K^T, mask, P = softmax(S),
    O = P V; lse from the same row statistics.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Hkv, Nq, Nk, d = _check_shapes(q, k, v)
    G = H // Hkv
    row_idx = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    R = row_idx.shape[0]
    O = np.zeros((B, H, R, d), dtype=np.float64)
    lse = np.zeros((B, H, R), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            g = h // G
            S = scores(q[b, h, row_idx], k[b, g], scale, causal, row_idx, Nq)
            P, _, lse_bh = softmax_rows(S)
            O[b, h] = P @ v[b, g]
            lse[b, h] = lse_bh
    return O, lse


def attention_online(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                     causal: bool, chunk: int, tau=None):
    """Chunked single-pass online-softmax restatement, in float64.

    Follows the recurrence of Interview notes "他人面经整理", flashattention
    answer part 2 ("Online Softmax"): per row keep m (running max) and l
    (running sum of exp(s - m)); for each block of ``chunk`` keys find the
    block maximum, set m_new = max(m_old, block max), rescale l and the
    accumulated output by exp(m_old - m_new), then add the block's exp-sum and
    P_block V_block.  The output is divided by l once at the end (the
    deferred normalisation of FlashAttention-2, FAQ page table: fewer
    non-matmul operations).

    ``tau``: if given, the reference maximum is only moved when the new
    maximum exceeds it by more than ``tau`` (natural-log units); otherwise the
    stale maximum is kept.  Exact in real arithmetic because numerator and
    denominator share the reference; exp(s - m) then stays <= exp(tau).

    This exists only to pin ``attention_ref``; it is not the oracle the GPU is
    compared with.  Returns (O [B,H,Nq,d], lse [B,H,Nq]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Hkv, Nq, Nk, d = _check_shapes(q, k, v)
    G = H // Hkv
    rows = np.arange(Nq)
    O = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            g = h // G
            m = np.full(Nq, -np.inf)
            l = np.zeros(Nq)
            acc = np.zeros((Nq, d))
            for j0 in range(0, Nk, chunk):
                kj = k[b, g, j0:j0 + chunk]
                vj = v[b, g, j0:j0 + chunk]
                s = scale * (q[b, h] @ kj.T)
                if causal:
                    jj = np.arange(j0, j0 + kj.shape[0])
                    s = np.where(jj[None, :] > causal_limit(rows, Nq, Nk)[:, None],
                                 -np.inf, s)
                m_blk = s.max(axis=1)
                m_cand = np.maximum(m, m_blk)
                if tau is None:
                    move = m_cand > m
                else:
                    move = (m_cand > m + tau) | (~np.isfinite(m) & np.isfinite(m_cand))
                m_new = np.where(move, m_cand, m)
                # alpha = exp(m_old - m_new); 1 where the reference did not move
                with np.errstate(invalid="ignore"):
                    alpha = np.where(move & np.isfinite(m), np.exp(m - m_new), 1.0)
                alpha = np.where(~np.isfinite(m) & move, 0.0, alpha)
                m_use = np.where(np.isfinite(m_new), m_new, 0.0)
                p = np.exp(s - m_use[:, None])
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ vj
                m = m_new
            dead = l == 0.0
            O[b, h] = np.where(dead[:, None], 0.0, acc / np.where(dead, 1.0, l)[:, None])
            with np.errstate(divide="ignore"):
                lse[b, h] = np.where(dead, -np.inf, np.where(np.isfinite(m), m, 0.0)
                                     + np.log(np.where(dead, 1.0, l)))
    return O, lse
