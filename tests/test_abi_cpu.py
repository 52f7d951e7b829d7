"""The C-ABI library loads without a GPU, exports every declared symbol, and
rejects invalid arguments before touching the device (CPU only)."""

import ctypes
import os
import re

import pytest

from attention_fa_attn_fwd_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_b300.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from attention_fa_attn_fwd_b300 import build
    build.build()
    return binding.load_library()


def test_header_declares_expected_api():
    assert declared_functions() == sorted(["attn_fwd", "attn_fwd_ex", "attn_fwd_host",
                                           "attn_fwd_host_workspace_size",
                                           "paged_decode", "paged_decode_workspace_size",
                                           "paged_decode_noalloc", "paged_prefill", "attn_bwd",
                                           "attn_bwd_ex", "attn_bwd_workspace_size", "kv_append",
                                           "kv_append_workspace_size", "attn_selftest_wait_timeout",
                                           "attn_last_error",
                                           "attn_device_status"])


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(binding.SIGNATURES)


def _fake(n=0):
    return ctypes.c_void_p(0x10000 + 256 * n)  # aligned, never dereferenced


def _fwd(lib, **kw):
    a = dict(q=_fake(1), k=_fake(2), v=_fake(3), o=_fake(4), lse=None, B=1, H=2, Hkv=2, Nq=128,
             Nk=128, d=64, scale=0.125, causal=0, stream=None)
    a.update(kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"],
                        a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), binding.ATTN_EINVAL),
    (dict(o=None), binding.ATTN_EINVAL),
    (dict(B=0), binding.ATTN_EINVAL),
    (dict(Nk=0), binding.ATTN_EINVAL),
    (dict(H=3, Hkv=2), binding.ATTN_EINVAL),
    (dict(scale=0.0), binding.ATTN_EINVAL),
    (dict(scale=-1.0), binding.ATTN_EINVAL),
    (dict(scale=float("nan")), binding.ATTN_EINVAL),
    (dict(scale=float("inf")), binding.ATTN_EINVAL),
    (dict(causal=2), binding.ATTN_EINVAL),
    (dict(d=96), binding.ATTN_EUNSUPPORTED),
    (dict(d=256), binding.ATTN_EUNSUPPORTED),
    (dict(q=ctypes.c_void_p(0x10008)), binding.ATTN_EINVAL),
    (dict(lse=ctypes.c_void_p(0x10002)), binding.ATTN_EINVAL),
])
def test_attn_fwd_rejects_bad_arguments(lib, kw, status):
    assert _fwd(lib, **kw) == status
    assert lib.attn_last_error()


def _dec(lib, **kw):
    a = dict(q=_fake(1), kc=_fake(2), vc=_fake(3), bt=_fake(4), sl=_fake(5), S=4, H=32, Hkv=8,
             d=128, nb=100, mb=64, bs=16, scale=0.088, o=_fake(6), lse=None, ws=_fake(7),
             wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.paged_decode(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["S"], a["H"], a["Hkv"],
                            a["d"], a["nb"], a["mb"], a["bs"], a["scale"], a["o"], a["lse"],
                            a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(bt=None), binding.ATTN_EINVAL),
    (dict(ws=None), binding.ATTN_EINVAL),
    (dict(S=0), binding.ATTN_EINVAL),
    (dict(bs=32), binding.ATTN_EINVAL),
    (dict(H=30), binding.ATTN_EINVAL),
    (dict(H=68, Hkv=4), binding.ATTN_EUNSUPPORTED),
    (dict(d=80), binding.ATTN_EUNSUPPORTED),
    (dict(wsb=16), binding.ATTN_EINVAL),
    (dict(scale=0.0), binding.ATTN_EINVAL),
    (dict(nb=1 << 30), binding.ATTN_EINVAL),
    (dict(kc=ctypes.c_void_p(0x10004)), binding.ATTN_EINVAL),
])
def test_paged_decode_rejects_bad_arguments(lib, kw, status):
    assert _dec(lib, **kw) == status


def test_workspace_size(lib):
    n = lib.paged_decode_workspace_size(64, 32, 8, 128, 512)
    # 64 seqs x 32 heads x splits x (d + 2) fp32
    assert n > 0 and n % (64 * 32 * 130 * 4) == 0
    assert lib.paged_decode_workspace_size(0, 32, 8, 128, 512) == 0
    assert lib.paged_decode_workspace_size(64, 30, 8, 128, 512) == 0


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(lib) in (binding.ATTN_ECUDA, binding.ATTN_EUNSUPPORTED)


def _pp(lib, **kw):
    a = dict(q=_fake(1), kc=_fake(2), vc=_fake(3), bt=_fake(4), sl=_fake(5), S=4, H=32, Hkv=8,
             Nq=256, d=128, nb=100, mb=64, bs=16, scale=0.088, causal=1, o=_fake(6), lse=None,
             stream=None)
    a.update(kw)
    return lib.paged_prefill(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["S"], a["H"], a["Hkv"],
                             a["Nq"], a["d"], a["nb"], a["mb"], a["bs"], a["scale"], a["causal"],
                             a["o"], a["lse"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), binding.ATTN_EINVAL),
    (dict(sl=None), binding.ATTN_EINVAL),
    (dict(S=0), binding.ATTN_EINVAL),
    (dict(Nq=0), binding.ATTN_EINVAL),
    (dict(bs=8), binding.ATTN_EINVAL),
    (dict(H=30), binding.ATTN_EINVAL),
    (dict(d=96), binding.ATTN_EUNSUPPORTED),
    (dict(causal=3), binding.ATTN_EINVAL),
    (dict(scale=float("nan")), binding.ATTN_EINVAL),
    (dict(nb=1 << 30), binding.ATTN_EINVAL),
    (dict(o=ctypes.c_void_p(0x10008)), binding.ATTN_EINVAL),
    (dict(bt=ctypes.c_void_p(0x10002)), binding.ATTN_EINVAL),
])
def test_paged_prefill_rejects_bad_arguments(lib, kw, status):
    assert _pp(lib, **kw) == status
    assert lib.attn_last_error()


def _bwd(lib, **kw):
    a = dict(q=_fake(1), k=_fake(2), v=_fake(3), o=_fake(4), do=_fake(5), lse=_fake(6),
             dq=_fake(7), dk=_fake(8), dv=_fake(9), B=1, H=4, Hkv=2, Nq=256, Nk=256, d=128,
             scale=0.088, causal=1, ws=_fake(10), wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"],
                        a["dv"], a["B"], a["H"], a["Hkv"], a["Nq"], a["Nk"], a["d"], a["scale"],
                        a["causal"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(do=None), binding.ATTN_EINVAL),
    (dict(lse=None), binding.ATTN_EINVAL),
    (dict(ws=None), binding.ATTN_EINVAL),
    (dict(wsb=16), binding.ATTN_EINVAL),
    (dict(Nk=0), binding.ATTN_EINVAL),
    (dict(H=3), binding.ATTN_EINVAL),
    (dict(d=32), binding.ATTN_EUNSUPPORTED),
    (dict(causal=-1), binding.ATTN_EINVAL),
    (dict(scale=0.0), binding.ATTN_EINVAL),
    (dict(dk=ctypes.c_void_p(0x10004)), binding.ATTN_EINVAL),
])
def test_attn_bwd_rejects_bad_arguments(lib, kw, status):
    assert _bwd(lib, **kw) == status
    assert lib.attn_last_error()


def test_bwd_workspace_size(lib):
    # D (rounded up to 256 bytes), plus the fp32 dQ accumulator at d = 128
    assert lib.attn_bwd_workspace_size(2, 16, 2048, 64) == 2 * 16 * 2048 * 4
    assert lib.attn_bwd_workspace_size(1, 1, 1, 64) == 256
    assert lib.attn_bwd_workspace_size(2, 16, 2048, 128) == 2 * 16 * 2048 * 4 * 129
    assert lib.attn_bwd_workspace_size(1, 1, 1, 128) == 256 + 512
    assert lib.attn_bwd_workspace_size(0, 1, 1, 128) == 0
    assert lib.attn_bwd_workspace_size(1, 1, 1, 96) == 0


def test_attn_bwd_ex_flags(lib):
    a = [_fake(i) for i in range(1, 10)]
    common = (1, 4, 2, 256, 256, 128, 0.088, 1, _fake(10), 1 << 20)
    # unknown flag bits are rejected before anything else happens
    for bad in (0x4, 0x8, 0x80000000):
        assert lib.attn_bwd_ex(*a, *common, bad, None) == binding.ATTN_EINVAL
        assert "flags" in lib.attn_last_error().decode()
    # the known flags pass the flag check (and fail later, on the fake
    # workspace size, not on the flags)
    for good in (binding.ATTN_BWD_DETERMINISTIC, binding.ATTN_BWD_DIAG_WAIT_EXPIRES):
        tiny = (1, 4, 2, 256, 256, 128, 0.088, 1, _fake(10), 16)
        assert lib.attn_bwd_ex(*a, *tiny, good, None) == binding.ATTN_EINVAL
        assert "flags" not in lib.attn_last_error().decode()
    # the deterministic path needs only the D part of the workspace; the
    # default path at d = 128 needs the accumulator too
    small = (1, 4, 2, 256, 256, 128, 0.088, 1, _fake(10), 4096)
    assert lib.attn_bwd_ex(*a, *small, 0, None) == binding.ATTN_EINVAL
    assert "workspace" in lib.attn_last_error().decode()


def _app(lib, **kw):
    a = dict(kn=_fake(1), vn=_fake(2), kc=_fake(3), vc=_fake(4), bt=_fake(5), sl=_fake(6),
             rf=_fake(7), fi=_fake(8), ft=_fake(9), S=4, T=1, Hkv=8, d=128, nb=100, mb=64, bs=16,
             ws=_fake(10), wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.kv_append(a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["sl"], a["rf"], a["fi"],
                         a["ft"], a["S"], a["T"], a["Hkv"], a["d"], a["nb"], a["mb"], a["bs"],
                         a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(rf=None), binding.ATTN_EINVAL),
    (dict(ft=None), binding.ATTN_EINVAL),
    (dict(T=0), binding.ATTN_EINVAL),
    (dict(bs=32), binding.ATTN_EINVAL),
    (dict(d=256), binding.ATTN_EUNSUPPORTED),
    (dict(S=70000), binding.ATTN_EINVAL),
    (dict(wsb=64), binding.ATTN_EINVAL),
    (dict(kn=ctypes.c_void_p(0x10008)), binding.ATTN_EINVAL),
])
def test_kv_append_rejects_bad_arguments(lib, kw, status):
    assert _app(lib, **kw) == status
    assert lib.attn_last_error()


def test_selftest_rejects_bad_limit(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == binding.ATTN_EINVAL
    assert lib.attn_selftest_wait_timeout(2_000_000, None) == binding.ATTN_EINVAL


def test_attn_fwd_ex_flags(lib):
    a = dict(q=_fake(1), k=_fake(2), v=_fake(3), o=_fake(4))
    # unknown flag bits are rejected before anything else runs
    for bad in (0x4, 0x8, 0x80000000):
        st = lib.attn_fwd_ex(a["q"], a["k"], a["v"], a["o"], None, 1, 2, 2, 128, 128, 64,
                             0.125, 0, bad, None)
        assert st == binding.ATTN_EINVAL
        assert b"flags" in lib.attn_last_error()


def _fwd_host(lib, **kw):
    a = dict(q=_fake(1), k=_fake(2), v=_fake(3), o=_fake(4), lse=None, B=1, H=4, Hkv=2, Nq=128,
             Nk=256, d=128, scale=0.088, causal=1, ws=_fake(5), wsb=1 << 30, chunks=0,
             stream=None)
    a.update(kw)
    return lib.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"],
                             a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], a["ws"], a["wsb"],
                             a["chunks"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), binding.ATTN_EINVAL),
    (dict(ws=None), binding.ATTN_EINVAL),
    (dict(ws=ctypes.c_void_p(0x10010)), binding.ATTN_EINVAL),   # not 256-byte aligned
    (dict(wsb=1024), binding.ATTN_EINVAL),                       # too small
    (dict(chunks=-1), binding.ATTN_EINVAL),
    (dict(chunks=17), binding.ATTN_EINVAL),
    (dict(H=3), binding.ATTN_EINVAL),
    (dict(Nq=0), binding.ATTN_EINVAL),
    (dict(causal=2), binding.ATTN_EINVAL),
    (dict(scale=float("nan")), binding.ATTN_EINVAL),
    (dict(d=80), binding.ATTN_EUNSUPPORTED),
])
def test_attn_fwd_host_rejects_bad_arguments(lib, kw, status):
    assert _fwd_host(lib, **kw) == status
    assert lib.attn_last_error()


def test_fwd_host_workspace_size(lib):
    # Q + K + V + O + LSE, each rounded up to 256 bytes
    B, H, Hkv, Nq, Nk, d = 2, 8, 2, 300, 500, 64
    r = lambda n: (n + 255) // 256 * 256
    want = (r(B * H * Nq * d * 2) + 2 * r(B * Hkv * Nk * d * 2) + r(B * H * Nq * d * 2)
            + r(B * H * Nq * 4))
    assert lib.attn_fwd_host_workspace_size(B, H, Hkv, Nq, Nk, d) == want
    assert lib.attn_fwd_host_workspace_size(B, 7, Hkv, Nq, Nk, d) == 0
    assert lib.attn_fwd_host_workspace_size(B, H, Hkv, Nq, Nk, 96) == 0
    assert lib.attn_fwd_host_workspace_size(0, H, Hkv, Nq, Nk, d) == 0
