"""Seeded synthetic inputs for the Flint-shaped MoE decode step.

This package is the ONE source of inputs shared by the CPU oracle and the CUDA
path.  It holds no arithmetic of the decode step itself: it only draws
weights, prompts and batching schedules from counter-based hashes, and
quantises the seeded bf16 weights into the symmetric int4 (group 64) storage
format that defines the int4 model.  Both sides consume what it produces; the
oracle dequantises and computes on its own, the CUDA library on its own.
"""
from .configs import CONFIGS, EXTRA, FLINT_INT4_E3, ModelShape, get_config  # noqa: F401
from . import weights, prompts  # noqa: F401
