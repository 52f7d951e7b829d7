"""GPU checks of attn_fwd_host (C ABI): the forward on host buffers with the
transfers overlapped.

Each (batch, KV head) range runs the same kernel on the same rows as one
attn_fwd call over device buffers, so the results must be bit-identical to
it for every split of the units, pinned or pageable host memory; one case is
also checked against the fp64 oracle directly.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa_attn_fwd_b300 import binding, workloads
from tests.parity import compare, f64

pytestmark = pytest.mark.gpu


def _device_reference(q, k, v, causal):
    o, lse = binding.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def _bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


@pytest.mark.parametrize("chunks", [0, 1, 3, 5, 16])
@pytest.mark.parametrize("pinned", [True, False])
def test_bit_identical_to_device_path(chunks, pinned):
    B, H, Hkv, N, d = 2, 8, 2, 700, 128   # 4 (batch, KV head) units, ragged tail tile
    q, k, v = workloads.prefill_inputs(B, H, Hkv, N, N, d, seed=11, qk_gain=1.5)
    o_ref, lse_ref = _device_reference(q, k, v, True)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
        o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    else:
        o = torch.empty(q.shape, dtype=torch.bfloat16)
        lse = torch.empty((B, H, N), dtype=torch.float32)
    o, lse = binding.attn_fwd_host(q, k, v, causal=True, o=o, lse=lse, chunks=chunks)
    torch.cuda.synchronize()
    assert torch.equal(_bits(o), _bits(o_ref))
    assert torch.equal(_bits(lse), _bits(lse_ref))
    assert binding.device_status() == binding.ATTN_OK


@pytest.mark.parametrize("d", [64, 128])
def test_against_oracle_unequal_lengths_no_lse(d):
    B, H, Hkv, Nq, Nk = 1, 6, 3, 200, 333
    q, k, v = workloads.prefill_inputs(B, H, Hkv, Nq, Nk, d, seed=5)
    o, lse = binding.attn_fwd_host(q, k, v, causal=True, want_lse=False, chunks=2)
    torch.cuda.synchronize()
    assert lse is None
    O, L = oracle.attention_ref(f64(q), f64(k), f64(v), 1 / math.sqrt(d), True)
    compare(f64(o), None, O, None, f"attn_fwd_host d={d}")


def test_stream_ordered_back_to_back_calls_share_a_workspace():
    # Two calls on one side stream reuse one workspace: the second call's
    # input copies must wait for the first call's output copies.
    B, H, Hkv, N, d = 1, 16, 4, 1024, 128
    ins = [workloads.prefill_inputs(B, H, Hkv, N, N, d, seed=s) for s in (21, 22)]
    refs = [_device_reference(q, k, v, False) for q, k, v in ins]
    ws = torch.empty(binding.attn_fwd_host_workspace_size(B, H, Hkv, N, N, d), dtype=torch.uint8,
                     device="cuda")
    side = torch.cuda.Stream()
    # The host tensors must outlive the asynchronous calls: keep the pinned
    # copies referenced until the stream has finished.
    pinned = [tuple(t.pin_memory() for t in x) for x in ins]
    outs = []
    for q, k, v in pinned:
        outs.append(binding.attn_fwd_host(q, k, v, workspace=ws, chunks=4, stream=side))
    side.synchronize()
    for (o, lse), (o_ref, lse_ref) in zip(outs, refs):
        assert torch.equal(_bits(o), _bits(o_ref))
        assert torch.equal(_bits(lse), _bits(lse_ref))


def test_workspace_too_small_is_rejected():
    q, k, v = workloads.prefill_inputs(1, 2, 1, 128, 128, 64)
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.AttnError) as e:
        binding.attn_fwd_host(q, k, v, workspace=ws)
    assert e.value.status == binding.ATTN_EINVAL


def test_captured_in_a_cuda_graph_and_replayed():
    # The copy streams fork from and join back to the capturing stream, so the
    # whole call (copies in, kernels, copies out) becomes one graph.
    B, H, Hkv, N, d = 1, 8, 2, 512, 128
    q, k, v = workloads.prefill_inputs(B, H, Hkv, N, N, d, seed=31)
    o_ref, lse_ref = _device_reference(q, k, v, True)
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(binding.attn_fwd_host_workspace_size(B, H, Hkv, N, N, d), dtype=torch.uint8,
                     device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        binding.attn_fwd_host(qp, kp, vp, causal=True, o=o, lse=lse, workspace=ws, chunks=2,
                              stream=side)  # first call creates the copy streams
    side.synchronize()
    o.zero_()
    lse.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        binding.attn_fwd_host(qp, kp, vp, causal=True, o=o, lse=lse, workspace=ws, chunks=2,
                              stream=side)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(o), _bits(o_ref))
    assert torch.equal(_bits(lse), _bits(lse_ref))
