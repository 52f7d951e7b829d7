"""Write ``tiny_b1h2_n128_d64.json``: oracle outputs for the tiny seeded workload.

The pages print no worked numeric example for attention, so the only stored
expected values in this repository are written by this script, which calls
nothing but ``oracle/`` (and the seeded input generator).  The fixture guards
the oracle against silent drift; the oracle itself is pinned by
``tests/test_oracle.py``.

Run:  python tests/golden/make_golden.py
"""

import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from attention_fa_attn_fwd_b300 import workloads  # noqa: E402


def main():
    cfg = workloads.PREFILL_WORKLOADS["tiny_b1h2_n128_d64"]
    q, k, v = workloads.prefill_inputs(**cfg, seed=0)
    f = lambda t: oracle.bf16_bits_to_f64(t.contiguous().view(__import__("torch").int16).numpy())
    O, L = oracle.attention_ref(f(q), f(k), f(v), 1.0 / math.sqrt(cfg["d"]), cfg["causal"])
    rng = np.random.default_rng(1234)
    idx = [(0, int(rng.integers(2)), int(rng.integers(128)), int(rng.integers(64)))
           for _ in range(64)]
    out = {
        "source": "written by tests/golden/make_golden.py from oracle.attention_ref",
        "workload": "tiny_b1h2_n128_d64", "seed": 0, "scale": 1.0 / math.sqrt(cfg["d"]),
        "o_samples": [[b, h, i, c, float(O[b, h, i, c])] for b, h, i, c in idx],
        "lse": L[0].tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_b1h2_n128_d64.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
