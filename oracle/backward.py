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
