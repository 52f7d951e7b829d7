"""fp64 CPU oracle for exact scaled dot-product attention and paged decode.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain, obviously
correct statement of what the attention hot path computes.  Only the test
suite (``tests/``), ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py`` may import or call it.  The product path --
the CUDA library behind ``include/attn_b300.h`` and its Python binding --
never imports, links or calls anything here, and nothing here imports the
product path.  The only code both sides share is the seeded input generator
(``attention_fa_attn_fwd_b300.workloads``), which holds none of the method's
arithmetic.

Modules
-------
``attention``  the definition softmax(scale * Q K^T [+ causal mask]) V with S
               and P materialised, plus the per-row log-sum-exp; and a
               chunked online-softmax restatement of the single-pass
               recurrence, used only to pin the definition.
``paged``      paged-decode and chunked paged-prefill references: gather
               each sequence's logical K/V through the block table, then
               apply the definition.
``backward``   gradients of the definition (dQ, dK, dV) by the chain rule,
               with P materialised.
``kv_cache``   appending tokens to a paged cache: the logical definition and
               a sequential copy-on-write block manager.
``bf16``       exact decoding of bfloat16 bit patterns to float64.

Every function states the passage of the source pages it follows.  Every
function is pinned by tests in ``tests/test_oracle.py`` against closed forms,
invariants, brute force and a library special case; none is "parity
unpinned".
"""

from .bf16 import bf16_bits_to_f64
from .attention import (
    causal_limit,
    scores,
    softmax_rows,
    attention_ref,
    attention_online,
)
from .backward import attention_bwd_ref, attention_bwd_rows
from .kv_cache import BlockManagerRef, append_logical
from .paged import gather_logical_kv, paged_decode_ref, paged_decode_ref_from_pool, paged_prefill_ref

__all__ = [
    "bf16_bits_to_f64",
    "causal_limit",
    "scores",
    "softmax_rows",
    "attention_ref",
    "attention_online",
    "gather_logical_kv",
    "paged_decode_ref",
    "paged_decode_ref_from_pool",
    "paged_prefill_ref",
    "attention_bwd_ref",
    "attention_bwd_rows",
    "append_logical",
    "BlockManagerRef",
]
