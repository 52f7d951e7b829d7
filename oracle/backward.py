"""fp64 reference for the attention backward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may use this module; the CUDA path never does.

Sources:

* Interview notes "他人面经整理", answer "介绍你理解的flashattention", part 3
  ("为反向传播进行的重计算"): the backward pass needs P, and instead of storing
  the N x N matrix it is recomputed from Q, K, V and the softmax statistics the
  forward pass kept.
* FAQ page "Wie unterscheidet sich die Implementierung von FlashAttention-2
  ...", comparison table, row on the backward pass: recomputation instead of a
  stored attention matrix.

The pages state that P is recomputed but print no gradient formulas, so this
module writes out the derivative of the forward definition (the plain chain
rule, which the recomputing kernels must reach up to rounding):

    S = scale Q K^T (masked),  P = softmax_rows(S),  O = P V
    dV = P^T dO
    dP = dO V^T
    dS_ij = P_ij (dP_ij - D_i),   D_i = sum_j P_ij dP_ij   (softmax Jacobian)
    dQ = scale dS K
    dK = scale dS^T Q

With grouped-query attention the gradient of a key/value head is the sum over
the query heads that read it (head h reads KV head h // (H / Hkv)).  Rows with
no unmasked key have P = 0 and contribute nothing.  P is materialised; nothing
is blocked or fused.
"""

from __future__ import annotations

import numpy as np

from .attention import _check_shapes, scores, softmax_rows


def attention_bwd_ref(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray,
                      scale: float, causal: bool):
    """Gradients (dQ, dK, dV) of sum(O * dO) for O = attention(q, k, v).

    q, do: [B, H, Nq, d]; k, v: [B, Hkv, Nk, d] (float64).  Returns dq
    [B, H, Nq, d], dk and dv [B, Hkv, Nk, d], and D [B, H, Nq] (the row sums
    of P * dP, which the kernels also need).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, Hkv, Nq, Nk, d = _check_shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("do must have q's shape")
    G = H // Hkv
    rows = np.arange(Nq)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            g = h // G
            S = scores(q[b, h], k[b, g], scale, causal, rows, Nq)
            P, _, _ = softmax_rows(S)
            dv[b, g] += P.T @ do[b, h]
            dP = do[b, h] @ v[b, g].T
            Dh = np.sum(P * dP, axis=1)
            dS = P * (dP - Dh[:, None])
            dq[b, h] = scale * (dS @ k[b, g])
            dk[b, g] += scale * (dS.T @ q[b, h])
            D[b, h] = Dh
    return dq, dk, dv, D


def attention_bwd_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray,
                       scale: float, causal: bool, q_rows, key_rows, kv_heads,
                       row_slice: int = 1024):
    """The same gradients as ``attention_bwd_ref``, evaluated only where asked.

    For sizes where the full N x N matrices do not fit (a 16k-token context),
    this returns
      dq  [B, H, len(q_rows), d]        the rows ``q_rows`` of dQ, every head;
      dk, dv [len(kv_heads), len(key_rows), d]
                                        the rows ``key_rows`` of dK and dV for
                                        each (b, kv head) pair in ``kv_heads``.
    The arithmetic is the chain rule written out in ``attention_bwd_ref``:

    * a dQ row i needs the full row i of P (the softmax over all its keys),
      the full row of dP = dO_i V^T, D_i = sum_j P_ij dP_ij, and then
      dQ_i = scale sum_j P_ij (dP_ij - D_i) K_j;
    * a dK / dV row j needs column j of P and dP for every query of every
      head that reads the KV head, and each query's D_i, which needs that
      query's whole row: dV_j = sum_i P_ij dO_i, dK_j = scale sum_i
      P_ij (dP_ij - D_i) Q_i, summed over the heads of the group.

    Query rows are evaluated ``row_slice`` at a time only to bound memory;
    every row's softmax and D are taken over the full row, as in the
    definition.  q, k, v, do float64 as for ``attention_bwd_ref``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, Hkv, Nq, Nk, d = _check_shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("do must have q's shape")
    G = H // Hkv
    qr = np.asarray(q_rows, dtype=np.int64)
    kr = np.asarray(key_rows, dtype=np.int64)
    dq = np.zeros((B, H, qr.shape[0], d))
    for b in range(B):
        for h in range(H):
            g = h // G
            S = scores(q[b, h, qr], k[b, g], scale, causal, qr, Nq)
            P, _, _ = softmax_rows(S)
            dP = do[b, h, qr] @ v[b, g].T
            Dh = np.sum(P * dP, axis=1)
            dq[b, h] = scale * ((P * (dP - Dh[:, None])) @ k[b, g])
    pairs = [(int(b), int(g)) for b, g in kv_heads]
    dk = np.zeros((len(pairs), kr.shape[0], d))
    dv = np.zeros((len(pairs), kr.shape[0], d))
    for n, (b, g) in enumerate(pairs):
        for h in range(g * G, (g + 1) * G):
            for i0 in range(0, Nq, row_slice):
                rows = np.arange(i0, min(Nq, i0 + row_slice))
                S = scores(q[b, h, rows], k[b, g], scale, causal, rows, Nq)
                P, _, _ = softmax_rows(S)
                dP = do[b, h, rows] @ v[b, g].T
                Dh = np.sum(P * dP, axis=1)
                Pc = P[:, kr]
                dSc = Pc * (dP[:, kr] - Dh[:, None])
                dv[n] += Pc.T @ do[b, h, rows]
                dk[n] += scale * (dSc.T @ q[b, h, rows])
    return dq, dk, dv
