"""Failure detection on the GPU without a GPU fault.

Every wait in the kernels is bounded.  attn_selftest_wait_timeout makes one
such wait run out (a barrier that nothing signals, 20 ms limit) and checks
that the expiry is recorded; afterwards the context must still run the
normal kernels correctly.  Nothing here traps, asserts on the device or
touches a bad address.
"""

import math
import time

import pytest
import torch

import oracle
from attention_fa_attn_fwd_b300 import binding, workloads
from tests.parity import compare, f64

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_survives():
    t0 = time.perf_counter()
    assert binding.selftest_wait_timeout(20000) == binding.ATTN_OK
    assert time.perf_counter() - t0 < 5.0
    # twice in a row: the word is cleared and set again
    assert binding.selftest_wait_timeout(5000) == binding.ATTN_OK
    # the library's own error words are untouched, and kernels still work
    assert binding.device_status() == binding.ATTN_OK
    q, k, v = workloads.prefill_inputs(1, 2, 2, 200, 200, 128, seed=3)
    o, lse = binding.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    O, L = oracle.attention_ref(f64(q), f64(k), f64(v), 1 / math.sqrt(128), True)
    compare(f64(o.cpu()), f64(lse.cpu()), O, L, "after the self-test")
