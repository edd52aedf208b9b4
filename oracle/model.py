"""Plain float64 CPU oracle of one Flint-shaped MoE decode step.

Test infrastructure: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline may use it.  It shares no code with the CUDA library.

What it computes follows the operator list of "rec Megakernel and Tempo9
Compared", §2 ("Where Does rec's Single-Stream Advantage Come From?"): input
RMSNorm, QKV projection, RoPE, KV write, attention, output projection and
residual, post-attention RMSNorm, MoE router with top-k selection, expert
gate/up -> SiLU -> down (dense SwiGLU MLP in the first layers), residual, and
after the last layer final norm, lm_head and argmax.  The page names these
steps but not their formulas; the readings taken here are:

  RMSNorm   y = x / sqrt(mean(x^2) + eps) * w
  RoPE      rotate-half pairs (i, i + d/2); inv_freq_i = theta^(-2i/d);
            angle = pos * inv_freq_i; positions 0-based
  attention scale 1/sqrt(d); grouped-query with contiguous groups
            (q head h uses kv head h // (n_heads / n_kv_heads)); the new
            token's K/V are stored (rounded to bf16, the cache's storage
            format) before it attends, so it attends to itself
  router    p = softmax(z . Wr^T); top-k by p, ties to the lower expert id;
            weights p_j / sum over the selected p
  expert    Wd (silu(Wg z) * (Wu z)); dense layers the same with weight 1
  argmax    ties to the lowest token id

All arithmetic is float64; bf16 appears only where the model stores values in
bf16 (weights as given, and the KV cache).

Pins (tests/test_oracle_pins.py) — every function here is pinned by at least
one check against a closed form, a brute-force computation or an invariant:
  rmsnorm      closed form on constant vectors; scale invariance
  rope         identity at pos 0; pair norms kept; relative-position property;
               equals the complex-multiplication form
  attention    float64 brute-force loops; ctx 1 -> V_0; equal keys -> mean(V)
  router_topk  top-k == all experts gives the dense softmax mixture;
               brute-force enumeration on tiny inputs
  swiglu       one expert with top-1 equals a dense SwiGLU MLP
  decode       incremental decode == full causal recompute (prefill)
  PagedKV      any page permutation == contiguous KV, bit-exact
"""
from __future__ import annotations

import math
from collections import OrderedDict
from typing import Callable

import numpy as np

from .numerics import round_bf16, to_f64


# ------------------------------------------------------------- primitives

def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Root-mean-square norm over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotary embedding, rotate-half convention, on the last axis of x.

    x: [..., d]; pos: scalar or array broadcastable to x.shape[:-1]."""
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Softmax attention of one position over T cached positions.

    q: [n_heads, d]; K, V: [T, n_kv, d] -> [n_heads, d]."""
    nh, d = q.shape
    nkv = K.shape[1]
    grp = nh // nkv
    out = np.empty((nh, d))
    for h in range(nh):
        g = h // grp
        s = K[:, g, :] @ q[h] / math.sqrt(d)
        p = np.exp(s - s.max())
        out[h] = (p / p.sum()) @ V[:, g, :]
    return out


def causal_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, start: int = 0) -> np.ndarray:
    """Attention of T0 new positions (absolute positions start..start+T0-1)
    over all T positions stored so far, each seeing positions <= its own.

    Q: [T0, n_heads, d]; K, V: [T, n_kv, d] -> [T0, n_heads, d]."""
    T0, nh, d = Q.shape
    T = K.shape[0]
    nkv = K.shape[1]
    grp = nh // nkv
    qpos = start + np.arange(T0)
    mask = np.arange(T)[None, :] <= qpos[:, None]            # [T0, T]
    out = np.empty((T0, nh, d))
    for h in range(nh):
        g = h // grp
        s = Q[:, h, :] @ K[:, g, :].T / math.sqrt(d)         # [T0, T]
        s = np.where(mask, s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, h, :] = (p / p.sum(axis=1, keepdims=True)) @ V[:, g, :]
    return out


def silu(x):
    return x / (1.0 + np.exp(-x))


def swiglu(z: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray) -> np.ndarray:
    """Wd (silu(Wg z) * (Wu z)) for z of shape [..., H]."""
    return (silu(z @ Wg.T) * (z @ Wu.T)) @ Wd.T


def router_topk(logits: np.ndarray, k: int):
    """Softmax over all experts, the k most probable (ties -> lower id),
    renormalised over the selected ones.  logits: [E] -> (ids[k], weights[k], p[E])."""
    z = logits - logits.max()
    p = np.exp(z) / np.exp(z).sum()
    order = np.argsort(-p, kind="stable")
    ids = order[:k]
    w = p[ids] / p[ids].sum()
    return ids.astype(np.int64), w, p


def topk_margin(logits: np.ndarray, k: int) -> float:
    """k-th minus (k+1)-th largest logit (inf when k covers every expert)."""
    if k >= logits.shape[-1]:
        return math.inf
    s = np.sort(logits)[::-1]
    return float(s[k - 1] - s[k])


def argmax_lowest(v: np.ndarray) -> int:
    return int(np.argmax(v))          # first maximal index


def top2_margin(v: np.ndarray) -> float:
    s = np.sort(v)[::-1]
    return float(s[0] - s[1])


# ------------------------------------------------------------- KV stores

class ContiguousKV:
    """KV cache as one [T, n_kv, d] array per layer (bf16-rounded values)."""

    def __init__(self, n_layers: int, n_kv: int, d: int):
        self.k = [np.zeros((0, n_kv, d)) for _ in range(n_layers)]
        self.v = [np.zeros((0, n_kv, d)) for _ in range(n_layers)]

    def write(self, layer: int, pos: int, k: np.ndarray, v: np.ndarray):
        """Store positions pos .. pos+len(k)-1 (must extend the cache)."""
        assert pos == self.k[layer].shape[0], "positions must be appended in order"
        self.k[layer] = np.concatenate([self.k[layer], round_bf16(k)], axis=0)
        self.v[layer] = np.concatenate([self.v[layer], round_bf16(v)], axis=0)

    def read(self, layer: int, T: int):
        return self.k[layer][:T], self.v[layer][:T]

    def length(self) -> int:
        return self.k[0].shape[0]


class PagedKV:
    """KV cache in fixed-size pages of a shared pool, addressed through a
    per-sequence page table: position t lives in page table[t // P], slot t % P."""

    def __init__(self, n_layers: int, n_kv: int, d: int, n_pages: int,
                 page_tokens: int = 128, page_order=None):
        self.P = page_tokens
        self.pool_k = np.zeros((n_layers, n_pages, page_tokens, n_kv, d))
        self.pool_v = np.zeros((n_layers, n_pages, page_tokens, n_kv, d))
        self.free = list(page_order) if page_order is not None else list(range(n_pages))
        self.table: list = []
        self.T = 0

    def write(self, layer: int, pos: int, k: np.ndarray, v: np.ndarray):
        for i in range(k.shape[0]):
            t = pos + i
            while t // self.P >= len(self.table):
                self.table.append(self.free.pop(0))
            pg, sl = self.table[t // self.P], t % self.P
            self.pool_k[layer, pg, sl] = round_bf16(k[i])
            self.pool_v[layer, pg, sl] = round_bf16(v[i])
        if layer == 0:
            self.T = max(self.T, pos + k.shape[0])

    def read(self, layer: int, T: int):
        t = np.arange(T)
        pages = np.asarray(self.table, dtype=np.int64)[t // self.P]
        return self.pool_k[layer, pages, t % self.P], self.pool_v[layer, pages, t % self.P]

    def length(self) -> int:
        return self.T


# ------------------------------------------------------------- the model

class Oracle:
    """The decode step of a Flint-shaped MoE transformer.

    shape: any object with the fields of synth.ModelShape (n_layers, hidden,
    n_heads, n_kv_heads, head_dim, vocab, n_dense, dense_ffn, n_experts, top_k,
    expert_ffn, rope_theta, rms_eps).
    fetch(name, layer, expert) -> (raw, dtype): a stored tensor and its format
    ('f32', 'bf16', 'int4', 'int3').  Names: embed, final_norm, lm_head; per layer
    attn_norm, wq, wk, wv, wo, ffn_norm, and gate/up/down (dense layers) or
    router and exp_gate/exp_up/exp_down (MoE layers, per expert).
    cache_bytes: float64 weights kept after dequantisation (LRU).
    """

    def __init__(self, shape, fetch: Callable, cache_bytes: int = 4 << 30):
        self.m = shape
        self.fetch = fetch
        self.cache_bytes = cache_bytes
        self._cache: OrderedDict = OrderedDict()
        self._cached = 0

    # ---- weights
    def w(self, name: str, layer: int = -1, expert=None) -> np.ndarray:
        key = (name, layer, expert)
        if key in self._cache:
            self._cache.move_to_end(key)
            return self._cache[key]
        raw, dt = self.fetch(name, layer, expert)
        arr = to_f64(raw, dt)
        if arr.nbytes <= self.cache_bytes:
            self._cache[key] = arr
            self._cached += arr.nbytes
            while self._cached > self.cache_bytes:
                _, old = self._cache.popitem(last=False)
                self._cached -= old.nbytes
        return arr

    def embed(self, tokens) -> np.ndarray:
        E = self.w("embed")
        return E[np.asarray(tokens, dtype=np.int64)]

    def new_kv(self, paged: bool = False, n_pages: int = 0, page_order=None):
        m = self.m
        if paged:
            return PagedKV(m.n_layers, m.n_kv_heads, m.head_dim, n_pages, 128, page_order)
        return ContiguousKV(m.n_layers, m.n_kv_heads, m.head_dim)

    # ---- one layer over T0 new positions (T0 = 1 in decode)
    def _attn_block(self, l: int, x: np.ndarray, kv, start: int, incremental: bool):
        m = self.m
        T0 = x.shape[0]
        y = rmsnorm(x, self.w("attn_norm", l), m.rms_eps)
        q = (y @ self.w("wq", l).T).reshape(T0, m.n_heads, m.head_dim)
        k = (y @ self.w("wk", l).T).reshape(T0, m.n_kv_heads, m.head_dim)
        v = (y @ self.w("wv", l).T).reshape(T0, m.n_kv_heads, m.head_dim)
        pos = start + np.arange(T0)
        q = rope(q, pos[:, None], m.rope_theta)
        k = rope(k, pos[:, None], m.rope_theta)
        kv.write(l, start, k, v)
        if incremental:
            a = np.stack([attention(q[i], *kv.read(l, start + i + 1)) for i in range(T0)])
        else:
            a = causal_attention(q, *kv.read(l, start + T0), start=start)
        a = a.reshape(T0, m.q_dim)
        return x + a @ self.w("wo", l).T, a

    def _ffn_block(self, l: int, h: np.ndarray, tr: dict):
        m = self.m
        z = rmsnorm(h, self.w("ffn_norm", l), m.rms_eps)
        if l < m.n_dense:
            f = swiglu(z, self.w("gate", l), self.w("up", l), self.w("down", l))
            return h + f
        logits = z @ self.w("router", l).T                          # [T0, E]
        T0 = h.shape[0]
        ids = np.zeros((T0, m.top_k), np.int64)
        wts = np.zeros((T0, m.top_k))
        for t in range(T0):
            ids[t], wts[t], _ = router_topk(logits[t], m.top_k)
        f = np.zeros_like(h)
        for e in np.unique(ids):
            rows, slots = np.nonzero(ids == e)
            ye = swiglu(z[rows], self.w("exp_gate", l, int(e)), self.w("exp_up", l, int(e)),
                        self.w("exp_down", l, int(e)))
            f[rows] += wts[rows, slots][:, None] * ye
        tr["router_logits"].append(logits)
        tr["topk_ids"].append(ids)
        tr["topk_w"].append(wts)
        tr["topk_margin"].append(np.array([topk_margin(lg, m.top_k) for lg in logits]))
        return h + f

    def forward(self, kv, tokens, start: int, incremental: bool, all_logits: bool = False):
        """Run positions start .. start+len(tokens)-1 through the model.

        incremental=False: one batched causal pass (the full recompute);
        incremental=True: position by position against the cache (decode).
        Returns (next_token, trace) where next_token is the argmax after the
        last position and trace holds per-layer residuals and router data."""
        m = self.m
        tokens = np.asarray(tokens, dtype=np.int64)
        x = self.embed(tokens)
        tr = {"x": [], "attn": [], "router_logits": [], "topk_ids": [], "topk_w": [],
              "topk_margin": []}
        for l in range(m.n_layers):
            h, a = self._attn_block(l, x, kv, start, incremental)
            x = self._ffn_block(l, h, tr)
            tr["x"].append(x)
            tr["attn"].append(a)
        xs = x if all_logits else x[-1:]
        logits = rmsnorm(xs, self.w("final_norm"), m.rms_eps) @ self.w("lm_head").T
        tr["logits"] = logits
        tr["next_token"] = np.array([argmax_lowest(r) for r in logits])
        tr["top2_margin"] = np.array([top2_margin(r) for r in logits])
        return int(tr["next_token"][-1]), tr

    def prefill(self, kv, tokens, start: int = 0, all_logits: bool = False):
        return self.forward(kv, tokens, start, incremental=False, all_logits=all_logits)

    def decode(self, kv, token: int, pos: int):
        return self.forward(kv, [token], pos, incremental=True)
