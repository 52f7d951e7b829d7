"""paged_decode_noalloc: paged decode for callers that may not allocate device
memory (e.g. a plugin given only its input/output buffers, or a server that
reserved all device memory for its KV pool at start-up).  It must give the
same results as paged_decode with a caller workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes
import math

import pytest
import torch

from attention_fa_attn_fwd_b300 import binding, workloads
from tests.parity import compare, f64


def _noalloc(lib, pb, o, lse):
    qd = pb["q"]
    S, H, d = qd.shape
    nb, Hkv, bs, _ = pb["kc"].shape
    return lib.paged_decode_noalloc(
        qd.data_ptr(), pb["kc"].data_ptr(), pb["vc"].data_ptr(), pb["bt"].data_ptr(),
        pb["sl"].data_ptr(), S, H, Hkv, d, nb, pb["bt"].shape[1], bs, 1.0 / math.sqrt(d),
        o.data_ptr(), lse.data_ptr(), int(torch.cuda.current_stream().cuda_stream))


def _device_batch(**kw):
    b = workloads.paged_decode_inputs(**kw)
    return {"q": b.q.cuda(), "kc": b.k_cache.cuda(), "vc": b.v_cache.cuda(),
            "bt": b.block_table.cuda(), "sl": b.seq_lens.cuda()}


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = binding.load_library()
    batches = [
        _device_batch(**workloads.PAGED_WORKLOADS["paged_decode_s64_h32kv8_d128"], seed=0),
        _device_batch(num_seqs=8, H=8, Hkv=2, d=128, min_len=40, max_len=700, group=4,
                      shared_tokens=32, spare_frac=0.1, seed=9),
    ]
    for call, pb in enumerate(batches):  # two calls in a row, sharing the scratch
        o_ref, l_ref = binding.paged_decode(pb["q"], pb["kc"], pb["vc"], pb["bt"], pb["sl"])
        o = torch.full_like(pb["q"], float("nan"))
        lse = torch.full(o.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(lib, pb, o, lse)
        assert st == binding.ATTN_OK, lib.attn_last_error()
        torch.cuda.synchronize()
        compare(f64(o), f64(lse), f64(o_ref), f64(l_ref), f"no-alloc call {call}")
    assert binding.device_status() == binding.ATTN_OK


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = binding.load_library()
    fake = ctypes.c_void_p(0x10000)
    # 4096 sequences x 64 heads x 512 blocks needs far more than 32 MiB of partials
    st = lib.paged_decode_noalloc(fake, fake, fake, fake, fake, 4096, 64, 8, 128, 100000, 512,
                                  16, 0.088, fake, None, None)
    assert st == binding.ATTN_EINVAL
    assert b"static scratch" in lib.attn_last_error()
