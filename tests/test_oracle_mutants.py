"""Plant plausible mistakes in copies of the oracle; the pins must catch each.

Every mutant below is the plain definition with one deliberate error of the
kind a reader could miss: a wrong head index, the other causal alignment, a
dropped scale, a sign flip, a swapped operand, a dropped mask, a wrong lse.
Each must fail at least one pin of ``test_oracle.py``.  (Mistakes are only
ever planted here, in CPU copies of the oracle.)
"""

import numpy as np
import pytest

from oracle.attention import softmax_rows
from tests.test_oracle import ALL_PINS


def _mutant(kind):
    def fn(q, k, v, scale, causal, rows=None):
        q = np.asarray(q, float); k = np.asarray(k, float); v = np.asarray(v, float)
        B, H, Nq, d = q.shape
        Hkv, Nk = k.shape[1], k.shape[2]
        G = H // Hkv
        O = np.zeros((B, H, Nq, d)); L = np.zeros((B, H, Nq))
        for b in range(B):
            for h in range(H):
                g = h % Hkv if kind == "gqa_modulo" else h // G
                sc = 1.0 if kind == "no_scale" else scale
                S = sc * (q[b, h] @ k[b, g].T)
                if causal and kind != "no_mask":
                    i = np.arange(Nq)[:, None]; j = np.arange(Nk)[None, :]
                    lim = i if kind == "top_left" else i + (Nk - Nq)
                    S = np.where(j > lim, -np.inf, S)
                if kind == "exp_sign":
                    S = -S
                P, m, lse = softmax_rows(S)
                if kind == "lse_no_max":
                    lse = lse - np.where(np.isfinite(m), m, 0.0)
                vv = k[b, g] if kind == "k_for_v" else v[b, g]
                O[b, h] = P @ vv
                if kind == "transposed_p" and Nq == Nk:
                    O[b, h] = P.T @ vv
                L[b, h] = lse
        return O, L
    return fn


MUTANTS = ["gqa_modulo", "top_left", "no_scale", "exp_sign", "lse_no_max", "k_for_v",
           "no_mask", "transposed_p"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_mutant(kind):
    fn = _mutant(kind)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(fn)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {kind}"
