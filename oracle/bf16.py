"""bfloat16 as 16-bit patterns, for the oracle (numpy has no bf16 type).

A bf16 value is the upper half of an IEEE-754 binary32 word. Widening is exact;
narrowing rounds to nearest, ties to even, done here in integer arithmetic on
the binary32 bits. NaN inputs stay NaN (quiet bit forced).
"""
import numpy as np


def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    r = np.where(nan, (u >> 16) | 0x40, r)
    return (r & 0xFFFF).astype(np.uint16)


def bf16_bits_to_f64(b):
    """Exact value of bf16 bit patterns, as float64."""
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(b):
    """Exact value of bf16 bit patterns, as float32."""
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)
