"""Exact attention forward (FlashAttention-2-style prefill) and paged decode for B300 (sm_103a).

The compute lives in ``libattn_b300.so`` (CUDA, built from ``csrc/``); the C
ABI is declared in ``include/attn_b300.h``.  ``binding`` marshals torch
tensors to that ABI.  ``workloads`` draws the seeded synthetic inputs.
"""

from .binding import (  # noqa: F401
    AttnError,
    attn_bwd,
    attn_fwd,
    kv_append,
    paged_decode,
    paged_prefill,
    paged_decode_workspace_size,
    library_path,
    load_library,
)
