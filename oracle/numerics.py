"""Storage-format conversions of the oracle, in float64.

Test infrastructure: see the package docstring.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned
    as float64.  bf16 keeps 8 significant bits; frexp gives m in [0.5, 1), so
    m * 2**8 rounded to an integer keeps exactly those bits."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def dequant_int4(packed, scale_bits) -> np.ndarray:
    """Symmetric int4, groups of 64 along K: w[r, k] = q[r, k] * s[r, k // 64].

    `packed` [R, K/2] uint8 holds two's-complement nibbles, even k in the low
    nibble; `scale_bits` [R, K/64] are bf16 bit patterns."""
    packed = np.asarray(packed, dtype=np.uint8)
    R, half = packed.shape
    K = 2 * half
    lo = (packed & 0x0F).astype(np.int16)
    hi = (packed >> 4).astype(np.int16)
    q = np.empty((R, K), dtype=np.int16)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    q = np.where(q >= 8, q - 16, q).astype(np.float64)
    s = bf16_bits_to_f64(scale_bits)
    return (q.reshape(R, K // 64, 64) * s[:, :, None]).reshape(R, K)


def dequant_int3(packed, scale_bits) -> np.ndarray:
    """Symmetric int3, groups of 64 along K: w[r, k] = q[r, k] * s[r, k // 64].

    `packed` [R, 3K/8] uint8: each 3 bytes b0, b1, b2 are one little-endian
    24-bit word b0 + 256 b1 + 65536 b2 holding 8 consecutive codes, code j of
    the word at bits 3j .. 3j + 2, as 3-bit two's complement (4..7 stand for
    -4..-1); `scale_bits` [R, K/64] are bf16 bit patterns."""
    packed = np.asarray(packed, dtype=np.uint8)
    R, nb = packed.shape
    K = nb // 3 * 8
    b = packed.reshape(R, K // 8, 3).astype(np.int64)
    word = b[:, :, 0] + 256 * b[:, :, 1] + 65536 * b[:, :, 2]
    q = np.empty((R, K // 8, 8), dtype=np.int64)
    for j in range(8):
        q[:, :, j] = (word // (8 ** j)) % 8
    q = np.where(q >= 4, q - 8, q).reshape(R, K).astype(np.float64)
    s = bf16_bits_to_f64(scale_bits)
    return (q.reshape(R, K // 64, 64) * s[:, :, None]).reshape(R, K)


def to_f64(raw, dtype: str) -> np.ndarray:
    """A stored tensor in its format ('f32' values, 'bf16' bits, 'int4' or
    'int3' pair) -> float64."""
    if dtype == "int4":
        return dequant_int4(*raw)
    if dtype == "int3":
        return dequant_int3(*raw)
    if dtype == "bf16":
        return bf16_bits_to_f64(raw)
    return np.asarray(raw, dtype=np.float64)
