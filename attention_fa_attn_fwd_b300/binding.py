"""ctypes binding for ``libattn_b300.so`` (argument marshalling only).

Every entry point here checks that the torch tensors it is handed have the
dtype, device and contiguity the C ABI expects, then passes raw device
pointers, sizes and the current CUDA stream to the library.  All arithmetic
runs in the library's kernels; there is no fallback of any kind.  If the
library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

# Status codes of include/attn_b300.h
ATTN_OK = 0
ATTN_EINVAL = 1
ATTN_EUNSUPPORTED = 2
ATTN_ECUDA = 3
ATTN_EDEVICE = 4
ATTN_FWD_EXP2_FMA = 1  # attn_fwd_ex flags
ATTN_FWD_DIAG_WAIT_EXPIRES = 2
ATTN_BWD_DETERMINISTIC = 1  # attn_bwd_ex flag
ATTN_BWD_DIAG_WAIT_EXPIRES = 2  # attn_bwd_ex flag: failure-detection test only
_STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_EINVAL", 2: "ATTN_EUNSUPPORTED",
                 3: "ATTN_ECUDA", 4: "ATTN_EDEVICE"}

# Every symbol the header declares, with (restype, argtypes).
_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, ctypes.c_uint,
                         _vp]),
    "attn_fwd_host_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "attn_fwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _i,
                           _vp]),
    "paged_decode_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "paged_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f,
                          _vp, _vp, _vp, _sz, _vp]),
    "paged_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f,
                                  _vp, _vp, _vp]),
    "paged_prefill": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i,
                           _vp, _vp, _vp]),
    "attn_bwd_workspace_size": (_sz, [_i, _i, _i, _i]),
    "attn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i,
                      _vp, _sz, _vp]),
    "attn_bwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f,
                         _i, _vp, _sz, ctypes.c_uint, _vp]),
    "kv_append_workspace_size": (_sz, [_i, _i]),
    "kv_append": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                       _vp, _sz, _vp]),
    "attn_selftest_wait_timeout": (_i, [ctypes.c_uint, _vp]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_device_status": (_i, [_vp]),
}


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, "libattn_b300.so")


def load_library():
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m attention_fa_attn_fwd_b300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(status: int):
    if status != ATTN_OK:
        msg = load_library().attn_last_error()
        raise AttnError(status, msg.decode() if msg else "")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
             causal: bool = False, scale: Optional[float] = None,
             o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             want_lse: bool = True, stream=None,
             exp2_fma: bool = False,
             diag_wait_expires: bool = False) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """O = softmax(scale Q K^T [causal]) V and per-row LSE via ``attn_fwd``.

    q [B,H,Nq,d], k/v [B,Hkv,Nk,d], bf16, contiguous, on one CUDA device.
    Returns (o [B,H,Nq,d] bf16, lse [B,H,Nq] fp32 or None).
    ``exp2_fma=True`` calls ``attn_fwd_ex`` with ATTN_FWD_EXP2_FMA;
    ``diag_wait_expires=True`` adds ATTN_FWD_DIAG_WAIT_EXPIRES (a
    failure-detection test: the outputs are then undefined).
    """
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    B, H, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    else:
        _need(o, "o", torch.bfloat16, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    if lse is None and want_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    elif lse is not None:
        _need(lse, "lse", torch.float32, 3)
        if tuple(lse.shape) != (B, H, Nq):
            raise ValueError("lse must be [B, H, Nq]")
    flags = (ATTN_FWD_EXP2_FMA if exp2_fma else 0) | \
        (ATTN_FWD_DIAG_WAIT_EXPIRES if diag_wait_expires else 0)
    if flags:
        st = lib.attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr() if lse is not None else None,
                             B, H, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                             flags, _stream_handle(stream))
    else:
        st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          lse.data_ptr() if lse is not None else None,
                          B, H, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                          _stream_handle(stream))
    _check(st)
    return o, lse


def _need_host(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_fwd_host_workspace_size(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    return int(load_library().attn_fwd_host_workspace_size(B, H, Hkv, Nq, Nk, d))


def attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  causal: bool = False, scale: Optional[float] = None,
                  o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  want_lse: bool = True, workspace: Optional[torch.Tensor] = None,
                  chunks: int = 0, device=None,
                  stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """``attn_fwd_host``: the forward on HOST tensors (pinned for overlap).

    q [B,H,Nq,d], k/v [B,Hkv,Nk,d] bf16 CPU tensors; o / lse are CPU outputs
    (allocated pinned if not given).  ``workspace`` is a uint8 CUDA tensor of
    at least ``attn_fwd_host_workspace_size`` bytes (allocated on ``device``,
    default the current one, if not given).  Asynchronous on ``stream``: the
    outputs are valid once the stream has reached this call's end, and every
    host tensor passed in must stay alive and unchanged until then (a
    temporary such as ``q.pin_memory()`` may be freed and its pinned block
    reused before the copies run).
    """
    lib = load_library()
    _need_host(q, "q", torch.bfloat16, 4)
    _need_host(k, "k", torch.bfloat16, 4)
    _need_host(v, "v", torch.bfloat16, 4)
    B, H, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    else:
        _need_host(o, "o", torch.bfloat16, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    if lse is None and want_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    elif lse is not None:
        _need_host(lse, "lse", torch.float32, 3)
        if tuple(lse.shape) != (B, H, Nq):
            raise ValueError("lse must be [B, H, Nq]")
    need = int(lib.attn_fwd_host_workspace_size(B, H, Hkv, Nq, Nk, d))
    if workspace is None:
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif not workspace.is_cuda or workspace.dtype != torch.uint8:
        raise TypeError("workspace must be a uint8 CUDA tensor")
    st = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr() if lse is not None else None,
                           B, H, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                           workspace.data_ptr(), workspace.numel(), int(chunks),
                           _stream_handle(stream))
    _check(st)
    return o, lse


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             do: torch.Tensor, lse: torch.Tensor, causal: bool = False,
             scale: Optional[float] = None, dq: Optional[torch.Tensor] = None,
             dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, stream=None,
             deterministic: bool = False, diag_wait_expires: bool = False):
    """Gradients (dq, dk, dv) of ``attn_fwd`` via ``attn_bwd_ex``.

    q, o, do [B,H,Nq,d] bf16; k, v [B,Hkv,Nk,d] bf16; lse [B,H,Nq] fp32 from
    ``attn_fwd``.  ``workspace``: uint8 CUDA tensor of at least
    ``attn_bwd_workspace_size`` bytes (allocated here if omitted).
    ``deterministic`` sets ATTN_BWD_DETERMINISTIC (bit-reproducible dq).
    ``diag_wait_expires`` adds ATTN_BWD_DIAG_WAIT_EXPIRES (a failure test:
    one bounded wait of the call expires; its outputs are undefined).
    """
    lib = load_library()
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _need(t, name, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    B, H, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if k.shape != v.shape or o.shape != q.shape or do.shape != q.shape or k.shape[0] != B \
            or k.shape[3] != d or tuple(lse.shape) != (B, H, Nq):
        raise ValueError("attn_bwd: shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, name, ref in ((dq, "dq", q), (dk, "dk", k), (dv, "dv", v)):
        _need(t, name, torch.bfloat16, 4)
        if t.shape != ref.shape:
            raise ValueError(f"{name} has the wrong shape")
    need = int(lib.attn_bwd_workspace_size(B, H, Nq, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    elif workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a uint8 CUDA tensor")
    flags = (ATTN_BWD_DETERMINISTIC if deterministic else 0) | \
        (ATTN_BWD_DIAG_WAIT_EXPIRES if diag_wait_expires else 0)
    st = lib.attn_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                         lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         B, H, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                         workspace.data_ptr(), workspace.numel(), flags, _stream_handle(stream))
    _check(st)
    return dq, dk, dv


def attn_bwd_workspace_size(B: int, H: int, Nq: int, d: int) -> int:
    return int(load_library().attn_bwd_workspace_size(B, H, Nq, d))


def paged_decode_workspace_size(num_seqs: int, H: int, Hkv: int, d: int,
                                max_blocks_per_seq: int) -> int:
    return int(load_library().paged_decode_workspace_size(num_seqs, H, Hkv, d, max_blocks_per_seq))


def paged_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_table: torch.Tensor, seq_lens: torch.Tensor,
                 scale: Optional[float] = None, o: Optional[torch.Tensor] = None,
                 lse: Optional[torch.Tensor] = None, want_lse: bool = True,
                 workspace: Optional[torch.Tensor] = None,
                 stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Decode attention over a paged KV cache via ``paged_decode``.

    q [S,H,d] bf16; k_cache/v_cache [num_blocks,Hkv,block_size,d] bf16;
    block_table [S,max_blocks] int32; seq_lens [S] int32.  ``workspace`` is a
    uint8 CUDA tensor of at least ``paged_decode_workspace_size`` bytes
    (allocated here if omitted).  Returns (o [S,H,d] bf16, lse [S,H] fp32).
    """
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    S, H, d = q.shape
    num_blocks, Hkv, block_size, dk = k_cache.shape
    if v_cache.shape != k_cache.shape or dk != d:
        raise ValueError("k_cache / v_cache / q shapes disagree")
    if block_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_table / seq_lens must have num_seqs rows")
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    else:
        _need(o, "o", torch.bfloat16, 3)
    if lse is None and want_lse:
        lse = torch.empty((S, H), dtype=torch.float32, device=q.device)
    elif lse is not None:
        _need(lse, "lse", torch.float32, 2)
    ws_bytes = paged_decode_workspace_size(S, H, Hkv, d, max_blocks)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    elif workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a uint8 CUDA tensor")
    st = lib.paged_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                          block_table.data_ptr(), seq_lens.data_ptr(),
                          S, H, Hkv, d, num_blocks, max_blocks, block_size, float(scale),
                          o.data_ptr(), lse.data_ptr() if lse is not None else None,
                          workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(st)
    return o, lse


def paged_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_table: torch.Tensor, seq_lens: torch.Tensor,
                         scale: Optional[float] = None, o: Optional[torch.Tensor] = None,
                         lse: Optional[torch.Tensor] = None,
                         stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """``paged_decode`` through the entry point that allocates nothing: the
    library's fixed 32 MiB scratch array replaces the workspace.  Calls that
    may overlap on the GPU race on that array; keep them on one stream."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    S, H, d = q.shape
    num_blocks, Hkv, block_size, dk = k_cache.shape
    if v_cache.shape != k_cache.shape or dk != d:
        raise ValueError("k_cache / v_cache / q shapes disagree")
    if block_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_table / seq_lens must have num_seqs rows")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    else:
        _need(o, "o", torch.bfloat16, 3)
    if lse is None:
        lse = torch.empty((S, H), dtype=torch.float32, device=q.device)
    else:
        _need(lse, "lse", torch.float32, 2)
    st = lib.paged_decode_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                  block_table.data_ptr(), seq_lens.data_ptr(), S, H, Hkv, d,
                                  num_blocks, block_table.shape[1], block_size, float(scale),
                                  o.data_ptr(), lse.data_ptr(), _stream_handle(stream))
    _check(st)
    return o, lse


def paged_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                  block_table: torch.Tensor, seq_lens: torch.Tensor, causal: bool = True,
                  scale: Optional[float] = None, o: Optional[torch.Tensor] = None,
                  lse: Optional[torch.Tensor] = None, want_lse: bool = True,
                  stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked prefill over a paged KV cache via ``paged_prefill``.

    q [S,H,Nq,d] bf16 (each sequence's newest Nq tokens); k_cache/v_cache
    [num_blocks,Hkv,16,d] bf16; block_table [S,max_blocks] int32; seq_lens
    [S] int32 (cached tokens, the chunk included).  Returns
    (o [S,H,Nq,d] bf16, lse [S,H,Nq] fp32 or None).
    """
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    S, H, Nq, d = q.shape
    num_blocks, Hkv, block_size, dk = k_cache.shape
    if v_cache.shape != k_cache.shape or dk != d:
        raise ValueError("k_cache / v_cache / q shapes disagree")
    if block_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_table / seq_lens must have num_seqs rows")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    else:
        _need(o, "o", torch.bfloat16, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    if lse is None and want_lse:
        lse = torch.empty((S, H, Nq), dtype=torch.float32, device=q.device)
    elif lse is not None:
        _need(lse, "lse", torch.float32, 3)
    st = lib.paged_prefill(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                           block_table.data_ptr(), seq_lens.data_ptr(), S, H, Hkv, Nq, d,
                           num_blocks, block_table.shape[1], block_size, float(scale),
                           int(bool(causal)), o.data_ptr(),
                           lse.data_ptr() if lse is not None else None, _stream_handle(stream))
    _check(st)
    return o, lse


def kv_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
              ref_counts: torch.Tensor, free_ids: torch.Tensor, free_top: torch.Tensor,
              workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Append T tokens per sequence to a paged cache via ``kv_append`` (in place).

    k_new/v_new [S,T,Hkv,d] bf16; caches [num_blocks,Hkv,16,d] bf16;
    block_table [S,max_blocks], seq_lens [S], ref_counts [num_blocks],
    free_ids [n], free_top [1] int32 -- all updated on the device.
    """
    lib = load_library()
    _need(k_new, "k_new", torch.bfloat16, 4)
    _need(v_new, "v_new", torch.bfloat16, 4)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(ref_counts, "ref_counts", torch.int32, 1)
    _need(free_ids, "free_ids", torch.int32, 1)
    _need(free_top, "free_top", torch.int32, 1)
    S, T, Hkv, d = k_new.shape
    num_blocks, hk, block_size, dk = k_cache.shape
    if v_new.shape != k_new.shape or v_cache.shape != k_cache.shape or hk != Hkv or dk != d:
        raise ValueError("kv_append: shape mismatch")
    if block_table.shape[0] != S or seq_lens.shape[0] != S or ref_counts.shape[0] != num_blocks:
        raise ValueError("kv_append: table sizes disagree")
    need = int(lib.kv_append_workspace_size(S, num_blocks))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=k_new.device)
    st = lib.kv_append(k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                       block_table.data_ptr(), seq_lens.data_ptr(), ref_counts.data_ptr(),
                       free_ids.data_ptr(), free_top.data_ptr(), S, T, Hkv, d, num_blocks,
                       block_table.shape[1], block_size, workspace.data_ptr(), workspace.numel(),
                       _stream_handle(stream))
    _check(st)


def kv_append_workspace_size(num_seqs: int, num_blocks: int) -> int:
    return int(load_library().kv_append_workspace_size(num_seqs, num_blocks))


def selftest_wait_timeout(limit_us: int = 20000, stream=None) -> int:
    """Run the bounded-wait self-test (see ``attn_selftest_wait_timeout``);
    returns the status code (ATTN_OK when the expired wait was reported)."""
    return int(load_library().attn_selftest_wait_timeout(int(limit_us), _stream_handle(stream)))


def device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the kernels' device error word."""
    return int(load_library().attn_device_status(_stream_handle(stream)))
