"""Counter-based 32-bit hash used for every random draw.

The mixer is the public-domain integer hash "hash32" (two rounds of
xor-shift-16 and a multiply by 0x45d9f3b, then a final xor-shift-16).  Its
multiplier is below 2**27, so the same arithmetic runs bit-identically in
NumPy (uint64) and in PyTorch (int64, CPU or CUDA) without overflow.
A value is keyed by (seed, stream, index): the same key always gives the same
value, independently of how many other values are drawn or in what order.
"""
from __future__ import annotations

import numpy as np

MASK32 = 0xFFFFFFFF
_M = 0x45D9F3B
_STREAM_MUL = 0x2545F49


def _mix_np(x: np.ndarray) -> np.ndarray:
    x = (((x >> np.uint64(16)) ^ x) * np.uint64(_M)) & np.uint64(MASK32)
    x = (((x >> np.uint64(16)) ^ x) * np.uint64(_M)) & np.uint64(MASK32)
    return (x >> np.uint64(16)) ^ x


def _mix_int(x: int) -> int:
    x &= MASK32
    x = (((x >> 16) ^ x) * _M) & MASK32
    x = (((x >> 16) ^ x) * _M) & MASK32
    return (x >> 16) ^ x


def stream_key(seed: int, stream: int) -> int:
    """32-bit key of one stream (one tensor, one prompt, ...)."""
    return _mix_int(_mix_int(seed & MASK32) ^ ((stream * _STREAM_MUL) & MASK32))


def hash_np(key: int, idx: np.ndarray) -> np.ndarray:
    """uint64 array of 32-bit hashes of element indices `idx` under `key`."""
    k = np.uint64(key)
    x = (idx.astype(np.uint64) & np.uint64(MASK32)) ^ k
    x = _mix_np(x)
    x = (x + k) & np.uint64(MASK32)
    return _mix_np(x)


def hash_torch(key: int, idx):
    """Same as hash_np on an int64 torch tensor (any device)."""
    x = (idx & MASK32) ^ key
    for _ in range(2):
        x = (((x >> 16) ^ x) * _M) & MASK32
    x = (x >> 16) ^ x
    x = (x + key) & MASK32
    for _ in range(2):
        x = (((x >> 16) ^ x) * _M) & MASK32
    return (x >> 16) ^ x


def hash_int(key: int, idx: int) -> int:
    x = ((idx & MASK32) ^ key)
    x = _mix_int(x)
    x = (x + key) & MASK32
    return _mix_int(x)
