"""Exact bfloat16 -> float64 decoding (oracle test infrastructure only).

bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
bits, 7 fraction bits.  Placing the 16-bit pattern in the high half of a
32-bit word therefore yields the binary32 with the same value, and binary32
-> binary64 conversion is exact.  The pages fix 16-bit inputs with fp32
accumulation ("FSA" page, section 2.2 item 3, mixed-precision fp16 in / fp32
accumulate; tutorial chapter 3, section 3.0.7 on fp32 accumulation being the
default); the kernels read bf16, so the oracle decodes the same bits exactly.
"""

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode an array of raw bfloat16 bit patterns (uint16/int16) to float64.

    Exact for every finite value, both infinities and NaN.
    """
    b = np.asarray(bits)
    if b.dtype not in (np.uint16, np.int16):
        raise TypeError(f"expected 16-bit integer bit patterns, got {b.dtype}")
    u32 = b.view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)
