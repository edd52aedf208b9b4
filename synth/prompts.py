"""Seeded prompts and the continuous-batching schedule.

Prompt tokens are uniform over [0, vocab) with seed `model_seed + 1000`
(stream = sequence index).  Config 5's prompt lengths are uniform in
[256, 8192] and arrival offsets uniform in [0, 64] steps, both from seed 4.
A uniform integer in [0, n) is `(h * n) >> 32` of a 32-bit hash h.
"""
from __future__ import annotations

import numpy as np

from .configs import Workload
from .hashing import hash_np, hash_int, stream_key

_PROMPT_SEED_OFFSET = 1000
_LEN_STREAM = 70001
_ARRIVAL_STREAM = 70002


def uniform_ints(seed: int, stream: int, count: int, n: int, start: int = 0) -> np.ndarray:
    idx = np.arange(start, start + count, dtype=np.uint64)
    h = hash_np(stream_key(seed, stream), idx)
    return ((h * np.uint64(n)) >> np.uint64(32)).astype(np.int64)


def prompt_tokens(model_seed: int, vocab: int, length: int, seq: int = 0) -> np.ndarray:
    """int32 tokens of prompt number `seq`."""
    return uniform_ints(model_seed + _PROMPT_SEED_OFFSET, seq, length, vocab).astype(np.int32)


def schedule(w: Workload):
    """[(arrival_step, prompt_len)] for each sequence of a workload."""
    if w.n_seqs == 1 or w.len_range is None:
        return [(0, w.prompt_len)]
    lo, hi = w.len_range
    alo, ahi = w.arrival_range
    out = []
    for i in range(w.n_seqs):
        L = lo + ((hash_int(stream_key(w.sched_seed, _LEN_STREAM), i) * (hi - lo + 1)) >> 32)
        a = alo + ((hash_int(stream_key(w.sched_seed, _ARRIVAL_STREAM), i) * (ahi - alo + 1)) >> 32)
        out.append((int(a), int(L)))
    return out
