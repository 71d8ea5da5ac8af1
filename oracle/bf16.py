"""bf16 bit patterns (uint16) to wider floats.  Oracle-side helper.

A bf16 value is the upper half of an IEEE binary32 value, so widening is a
16-bit left shift of the bit pattern; it is exact.
"""
import numpy as np


def to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(bits) -> np.ndarray:
    return to_f32(bits).astype(np.float64)


NEG_ZERO = np.uint16(0x8000)
POS_ZERO = np.uint16(0x0000)
