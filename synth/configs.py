"""The five decode workloads, as data.

Model shape: the Flint MoE transformer described on "rec Megakernel and
Tempo9 Compared", §2 (49 layers, a 2048-wide residual, top-6 experts, dense
MLP in layers 0 and 1).  The pages do not give the remaining dimensions; the
ones here (16 query / 4 key-value heads of 128, 64 experts of FFN 768, dense
FFN 6144, vocabulary 151936, RoPE theta 1e6) complete the shape, and the tiny
shape is a scaled-down model of the same family for fast end-to-end checks.
"""
from __future__ import annotations

import dataclasses
from typing import Optional


@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    n_dense: int          # layers [0, n_dense) use a dense SwiGLU MLP
    dense_ffn: int
    n_experts: int
    top_k: int
    expert_ffn: int
    rope_theta: float
    rms_eps: float
    wdtype: str           # "f32" | "bf16" | "int4": dtype of the linear layers
    seed: int             # weight seed
    expert_dtype: Optional[str] = None  # "int3": the experts' format; None: wdtype

    @property
    def xdtype(self) -> str:
        """Storage dtype of the expert matrices (gate, up, down of every expert)."""
        return self.expert_dtype or self.wdtype

    @property
    def aux_dtype(self) -> str:
        """dtype of embedding, norms and router: fp32 for the fp32 model, else bf16."""
        return "f32" if self.wdtype == "f32" else "bf16"

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def with_(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)


TINY = ModelShape(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64,
                  vocab=1024, n_dense=1, dense_ffn=512, n_experts=8, top_k=2,
                  expert_ffn=128, rope_theta=1e4, rms_eps=1e-6, wdtype="f32",
                  seed=0)

FLINT_BF16 = ModelShape(n_layers=49, hidden=2048, n_heads=16, n_kv_heads=4,
                        head_dim=128, vocab=151936, n_dense=2, dense_ffn=6144,
                        n_experts=64, top_k=6, expert_ffn=768, rope_theta=1e6,
                        rms_eps=1e-6, wdtype="bf16", seed=1)

FLINT_INT4 = FLINT_BF16.with_(wdtype="int4")

# The lower-bit expert variant ("rec Megakernel and Tempo9 Compared", §5 Method:
# rec serves the Flint model with INT3 experts): the same seeded weights, the
# expert matrices in symmetric int3 (group 64), everything else in int4.
FLINT_INT4_E3 = FLINT_INT4.with_(expert_dtype="int3")


@dataclasses.dataclass(frozen=True)
class Workload:
    id: int
    name: str
    model: ModelShape
    prompt_len: int                 # per sequence (configs 1-4)
    decode_tokens: int              # generated tokens per sequence
    batch: int = 1
    prefill_chunk: int = 4096
    n_seqs: int = 1                 # config 5: concurrent sequences
    len_range: Optional[tuple] = None     # config 5: prompt lengths U[lo, hi]
    arrival_range: Optional[tuple] = None  # config 5: arrival offsets U[lo, hi] steps
    sched_seed: int = 0


CONFIGS = {
    1: Workload(1, "tiny-f32", TINY, prompt_len=64, decode_tokens=16),
    2: Workload(2, "flint-bf16-ctx2048", FLINT_BF16, prompt_len=2048, decode_tokens=256),
    3: Workload(3, "flint-int4-ctx2048", FLINT_INT4, prompt_len=2048, decode_tokens=256),
    4: Workload(4, "flint-int4-ctx8022", FLINT_INT4, prompt_len=8022, decode_tokens=256),
    5: Workload(5, "flint-int4-cb16", FLINT_INT4, prompt_len=0, decode_tokens=256,
                batch=16, n_seqs=16, len_range=(256, 8192), arrival_range=(0, 64),
                sched_seed=4),
}


# Workloads beyond the five configurations: the int3-expert model on the
# shape and context of configuration 3.
EXTRA = {
    "flint-int4e3-ctx2048": Workload(6, "flint-int4e3-ctx2048", FLINT_INT4_E3, prompt_len=2048,
                                     decode_tokens=256),
}


def get_config(i: int) -> Workload:
    return CONFIGS[int(i)]
