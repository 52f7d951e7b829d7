"""The oracle still reproduces its stored outputs on the tiny seeded workload."""

import json
import math
import os

import numpy as np
import torch

import oracle
from attention_fa_attn_fwd_b300 import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_golden_fixture():
    with open(os.path.join(HERE, "golden", "tiny_b1h2_n128_d64.json")) as fh:
        gold = json.load(fh)
    cfg = workloads.PREFILL_WORKLOADS[gold["workload"]]
    q, k, v = workloads.prefill_inputs(**cfg, seed=gold["seed"])
    f = lambda t: oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy())
    O, L = oracle.attention_ref(f(q), f(k), f(v), gold["scale"], cfg["causal"])
    for b, h, i, c, val in gold["o_samples"]:
        assert abs(O[b, h, i, c] - val) < 1e-12
    assert np.max(np.abs(L[0] - np.array(gold["lse"]))) < 1e-12
