"""Helpers wiring seeded or hand-made weights into the oracle's fetch API."""
from __future__ import annotations

import dataclasses

import numpy as np

from synth import weights as SW
from synth.configs import ModelShape


def weights_struct(m: ModelShape, w: dict):
    """The C ABI's mk_weights over a dict of device tensors (the Engine's
    weight dict format); returns (weights, layers), the second to be kept
    alive with the first."""
    from moe_decode_megakernel_persistent_gb300 import _lib as L
    from moe_decode_megakernel_persistent_gb300.engine import _lin, _ptr
    layers = (L.mk_layer_weights * m.n_layers)()
    for l in range(m.n_layers):
        lw = layers[l]
        lw.attn_norm = _ptr(w[("attn_norm", l)])
        lw.ffn_norm = _ptr(w[("ffn_norm", l)])
        for name in ("wq", "wk", "wv", "wo"):
            setattr(lw, name, _lin(w[(name, l)]))
        if l < m.n_dense:
            for name in ("gate", "up", "down"):
                setattr(lw, name, _lin(w[(name, l)]))
        else:
            lw.router = _ptr(w[("router", l)])
            for name in ("exp_gate", "exp_up", "exp_down"):
                setattr(lw, name, _lin(w[(name, l)]))
    return L.mk_weights(embed=_ptr(w[("embed",)]), final_norm=_ptr(w[("final_norm",)]),
                        lm_head=_lin(w[("lm_head",)]), layers=layers), layers


def synth_fetch(m: ModelShape):
    """fetch(name, layer, expert) -> (raw, dtype) from the seeded generator,
    keeping the storage-format tensors it has produced."""
    cache = {}

    def fetch(name, layer, expert):
        key = (name, layer, expert)
        if key not in cache:
            if name in ("embed", "attn_norm", "ffn_norm", "final_norm", "router"):
                cache[key] = (SW.raw_np(m, name, layer, expert), m.aux_dtype)
            else:
                cache[key] = (SW.linear_np(m, name, layer, expert), SW.storage_dtype(m, name))
        return cache[key]
    return fetch


@dataclasses.dataclass
class Dims:
    n_layers: int = 2
    hidden: int = 24
    n_heads: int = 4
    n_kv_heads: int = 2
    head_dim: int = 6
    vocab: int = 37
    n_dense: int = 1
    dense_ffn: int = 20
    n_experts: int = 5
    top_k: int = 2
    expert_ffn: int = 14
    rope_theta: float = 100.0
    rms_eps: float = 1e-6

    @property
    def q_dim(self):
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim


def random_tensors(d: Dims, seed: int = 0, scale: float = 0.3):
    """float64 weights with every dimension distinct (q_dim != hidden, ...),
    so that a transposed operand fails on shape."""
    rng = np.random.default_rng(seed)
    H = d.hidden
    t = {("embed", -1, None): rng.normal(0, 1, (d.vocab, H)),
         ("final_norm", -1, None): rng.uniform(0.5, 1.5, H),
         ("lm_head", -1, None): rng.normal(0, scale, (d.vocab, H))}
    for l in range(d.n_layers):
        t[("attn_norm", l, None)] = rng.uniform(0.5, 1.5, H)
        t[("ffn_norm", l, None)] = rng.uniform(0.5, 1.5, H)
        t[("wq", l, None)] = rng.normal(0, scale, (d.q_dim, H))
        t[("wk", l, None)] = rng.normal(0, scale, (d.kv_dim, H))
        t[("wv", l, None)] = rng.normal(0, scale, (d.kv_dim, H))
        t[("wo", l, None)] = rng.normal(0, scale, (H, d.q_dim))
        if l < d.n_dense:
            t[("gate", l, None)] = rng.normal(0, scale, (d.dense_ffn, H))
            t[("up", l, None)] = rng.normal(0, scale, (d.dense_ffn, H))
            t[("down", l, None)] = rng.normal(0, scale, (H, d.dense_ffn))
        else:
            t[("router", l, None)] = rng.normal(0, 1.0, (d.n_experts, H))
            for e in range(d.n_experts):
                t[("exp_gate", l, e)] = rng.normal(0, scale, (d.expert_ffn, H))
                t[("exp_up", l, e)] = rng.normal(0, scale, (d.expert_ffn, H))
                t[("exp_down", l, e)] = rng.normal(0, scale, (H, d.expert_ffn))
    return t


def dict_fetch(t: dict):
    def fetch(name, layer, expert):
        return t[(name, layer, expert)], "f64"
    return fetch
