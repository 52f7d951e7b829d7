"""Failure detection on the GPU without a GPU fault.

Every wait in the kernels is bounded.  attn_selftest_wait_timeout makes one
such wait run out (a barrier that nothing signals, 20 ms limit) and checks
that the expiry is recorded; afterwards the context must still run the
normal kernels correctly.  ATTN_FWD_DIAG_WAIT_EXPIRES does the same inside a
real prefill launch (1 ms limit), to check that the expiry only affects the
launch it happened in; ATTN_BWD_DIAG_WAIT_EXPIRES makes one expire in the
middle of a backward CTA's work, so that its warps must drain copies and
products in flight.  Nothing here traps, asserts on the device or touches a
bad address.
"""

import math
import time

import pytest
import torch

import oracle
from attention_fa_attn_fwd_b300 import binding, workloads
from tests.parity import compare, compare_grad, f64

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


def _case(seed):
    q, k, v = workloads.prefill_inputs(1, 4, 2, 700, 700, 128, seed=seed)
    O, L = oracle.attention_ref(f64(q), f64(k), f64(v), 1 / math.sqrt(128), True)
    return (q.cuda(), k.cuda(), v.cuda()), (O, L)


def test_a_timeout_stays_inside_its_launch():
    """attn_fwd_ex(ATTN_FWD_DIAG_WAIT_EXPIRES) lets one bounded wait of a real
    prefill launch expire (CTA 0, in the producer two key tiles in, with
    copies and products of the CTA in flight, which its warps drain).
    The next launch, with no attn_device_status in between, must compute the
    right result: the timeout skips work only in the launch that recorded
    it.  attn_device_status then reports the code once."""
    (q, k, v), (O, L) = _case(5)
    assert binding.device_status() == binding.ATTN_OK
    binding.attn_fwd(q, k, v, causal=True, diag_wait_expires=True)
    o, lse = binding.attn_fwd(q, k, v, causal=True)
    o2, lse2 = binding.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    compare(f64(o.cpu()), f64(lse.cpu()), O, L, "launch after a timed-out launch")
    compare(f64(o2.cpu()), f64(lse2.cpu()), O, L, "second launch after a timed-out launch")
    assert binding.device_status() == binding.ATTN_EDEVICE
    assert "0x105" in binding.load_library().attn_last_error().decode()
    assert binding.device_status() == binding.ATTN_OK


def test_a_timeout_does_not_void_another_streams_launch():
    """A launch whose wait expires on one stream, and a normal launch queued
    right behind it on a second stream (they can run at the same time): the
    second one computes the right result."""
    (q, k, v), (O, L) = _case(6)
    assert binding.device_status() == binding.ATTN_OK
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        binding.attn_fwd(q, k, v, causal=True, diag_wait_expires=True, stream=s1)
    with torch.cuda.stream(s2):
        o, lse = binding.attn_fwd(q, k, v, causal=True, stream=s2)
    torch.cuda.synchronize()
    compare(f64(o.cpu()), f64(lse.cpu()), O, L, "other stream during a timed-out launch")
    assert binding.device_status() == binding.ATTN_EDEVICE
    assert binding.device_status() == binding.ATTN_OK


@pytest.mark.parametrize("det", [False, True])
def test_a_backward_timeout_drains_and_stays_inside_its_launch(det):
    """attn_bwd_ex(ATTN_BWD_DIAG_WAIT_EXPIRES) lets the dV/dK-issuing warp of
    the first key-stationary CTA give up on a barrier nothing signals a few
    query halves in, while that CTA's copies and products are in flight: its
    warps drain what they issued and exit.  The next call, with no
    attn_device_status in between, must give the oracle's gradients, and the
    code is reported once."""
    q, k, v = workloads.prefill_inputs(1, 4, 2, 1000, 1000, 128, seed=7)
    do = workloads.grad_output(q.shape, seed=7)
    sc = 1 / math.sqrt(128)
    rq, rk, rv, _ = oracle.attention_bwd_ref(f64(q), f64(k), f64(v), f64(do), sc, True)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = binding.attn_fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    t0 = time.perf_counter()
    binding.attn_bwd(qd, kd, vd, o, dod, lse, causal=True, deterministic=det,
                     diag_wait_expires=True)
    dq, dk, dv = binding.attn_bwd(qd, kd, vd, o, dod, lse, causal=True, deterministic=det)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    tag = "deterministic" if det else "default"
    compare_grad(f64(dq.cpu()), rq, f"dq after a timed-out backward ({tag})")
    compare_grad(f64(dk.cpu()), rk, f"dk after a timed-out backward ({tag})")
    compare_grad(f64(dv.cpu()), rv, f"dv after a timed-out backward ({tag})")
    assert binding.device_status() == binding.ATTN_EDEVICE
    assert "0x105" in binding.load_library().attn_last_error().decode()
    assert binding.device_status() == binding.ATTN_OK
