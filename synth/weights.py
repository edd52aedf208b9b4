"""Seeded model weights in their storage formats.

Every linear weight is an i.i.d. draw from N(0, 0.02): element `i` of tensor
`t` is `TABLE[hash(key(seed, t), i) >> 16]`, where TABLE holds the 65536
quantiles 0.02 * Phi^-1((j + 0.5) / 65536) rounded to the storage dtype.  A
table lookup is exact in every backend, so NumPy and PyTorch (CPU or CUDA)
produce the same bits.  Norm weights are 1.0.

Storage formats (the logical layout handed to the library and the oracle):
  f32 / bf16   row-major [rows, K] (bf16 as raw uint16 bits in NumPy)
  int4         symmetric, groups of 64 consecutive K elements per row:
               s = bf16_rne(fp32(max|w_g|) / 7); q = clamp(rint(w / s), -8, 7),
               an all-zero group gets s = 0, q = 0; packed two's-complement
               nibbles [rows, K/2] uint8 with the even k in the low nibble,
               scales [rows, K/64] bf16.
  int3         (expert matrices of a model with expert_dtype "int3") symmetric,
               groups of 64 consecutive K elements per row:
               s = bf16_rne(fp32(max|w_g|) / 3); q = clamp(rint(w / s), -4, 3),
               an all-zero group gets s = 0, q = 0; codes [rows, 3K/8] uint8:
               every 8 consecutive k form one 24-bit little-endian word (3
               bytes) holding the 3-bit two's-complement code of k at bits
               3 (k % 8) .. 3 (k % 8) + 2; scales [rows, K/64] bf16.
The quantisers are part of defining the int4 / int3 models (their weights ARE
the codes and scales); dequantisation is left to each consumer.
"""
from __future__ import annotations

import statistics
from functools import lru_cache

import numpy as np

from .configs import ModelShape
from .hashing import hash_np, hash_torch, stream_key

# stream ids of the tensors, fixed so any tensor can be regenerated alone
_GLOBAL_IDS = {"embed": 0, "lm_head": 2}
_LAYER_SLOTS = {"wq": 1, "wk": 2, "wv": 3, "wo": 4, "router": 6,
                "gate": 7, "up": 8, "down": 9,
                "exp_gate": 7, "exp_up": 8, "exp_down": 9}
LINEAR_NAMES = ("wq", "wk", "wv", "wo", "gate", "up", "down",
                "exp_gate", "exp_up", "exp_down", "lm_head")


def tensor_id(name: str, layer: int = -1) -> int:
    if name in _GLOBAL_IDS:
        return _GLOBAL_IDS[name]
    return 16 + 16 * layer + _LAYER_SLOTS[name]


def tensor_shape(m: ModelShape, name: str) -> tuple:
    H, E = m.hidden, m.n_experts
    return {
        "embed": (m.vocab, H), "lm_head": (m.vocab, H), "final_norm": (H,),
        "attn_norm": (H,), "ffn_norm": (H,),
        "wq": (m.q_dim, H), "wk": (m.kv_dim, H), "wv": (m.kv_dim, H),
        "wo": (H, m.q_dim),
        "gate": (m.dense_ffn, H), "up": (m.dense_ffn, H), "down": (H, m.dense_ffn),
        "router": (E, H),
        "exp_gate": (E, m.expert_ffn, H), "exp_up": (E, m.expert_ffn, H),
        "exp_down": (E, H, m.expert_ffn),
    }[name]


def layer_tensor_names(m: ModelShape, layer: int) -> list:
    names = ["attn_norm", "wq", "wk", "wv", "wo", "ffn_norm"]
    if layer < m.n_dense:
        names += ["gate", "up", "down"]
    else:
        names += ["router", "exp_gate", "exp_up", "exp_down"]
    return names


EXPERT_NAMES = ("exp_gate", "exp_up", "exp_down")


def storage_dtype(m: ModelShape, name: str) -> str:
    """'f32', 'bf16', 'int4' or 'int3' for a tensor of model m."""
    if name in EXPERT_NAMES:
        return m.xdtype
    if name in LINEAR_NAMES:
        return m.wdtype
    return m.aux_dtype


# ---------------------------------------------------------------- tables

@lru_cache(maxsize=None)
def _quantiles_f64() -> np.ndarray:
    nd = statistics.NormalDist(0.0, 1.0)
    j = np.arange(65536, dtype=np.float64)
    return 0.02 * np.array([nd.inv_cdf(p) for p in (j + 0.5) / 65536.0])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest even), as uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + ((b >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@lru_cache(maxsize=None)
def normal_table(dtype: str) -> np.ndarray:
    """The 65536-entry N(0, 0.02) quantile table: float32 values or bf16 bits."""
    q32 = _quantiles_f64().astype(np.float32)
    if dtype == "f32":
        return q32
    return f32_to_bf16_bits(q32)


# ---------------------------------------------------------------- draws

def _draw_np(seed: int, tid: int, start: int, count: int, dtype: str) -> np.ndarray:
    idx = np.arange(start, start + count, dtype=np.uint64)
    h = hash_np(stream_key(seed, tid), idx) >> np.uint64(16)
    return normal_table("f32" if dtype == "f32" else "bf16")[h.astype(np.int64)]


def _elem_range(m: ModelShape, name: str, expert, rows):
    shape = tensor_shape(m, name)
    if expert is None:
        inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
        base = 0
        out_shape = shape
        if len(shape) == 3:
            raise ValueError(f"{name} needs an expert index")
    else:
        assert len(shape) == 3
        inner = shape[2]
        base = expert * shape[1] * shape[2]
        out_shape = shape[1:]
    nrows = out_shape[0]
    r0, r1 = (0, nrows) if rows is None else rows
    K = out_shape[1] if len(out_shape) > 1 else 1
    start = base + r0 * K
    count = (r1 - r0) * K
    final_shape = (r1 - r0, K) if len(out_shape) > 1 else (r1 - r0,)
    return start, count, final_shape


def raw_np(m: ModelShape, name: str, layer: int = -1, expert=None, rows=None) -> np.ndarray:
    """The unquantised seeded tensor (or one expert's matrix, or a row range):
    float32 values for the fp32 model, bf16 bits (uint16) otherwise."""
    dt = "f32" if m.aux_dtype == "f32" else "bf16"
    if name in ("attn_norm", "ffn_norm", "final_norm"):
        n = m.hidden
        ones = np.ones(n, np.float32)
        return ones if dt == "f32" else f32_to_bf16_bits(ones)
    start, count, shp = _elem_range(m, name, expert, rows)
    v = _draw_np(m.seed, tensor_id(name, layer), start, count, dt)
    return v.reshape(shp)


def quantize_int4_np(w_bits: np.ndarray):
    """bf16 bits [R, K] -> (packed uint8 [R, K/2], scale bf16 bits uint16 [R, K/64])."""
    R, K = w_bits.shape
    assert K % 64 == 0
    w = bf16_bits_to_f32(w_bits).reshape(R, K // 64, 64)
    amax = np.abs(w).max(axis=2)
    s_bits = f32_to_bf16_bits((amax / np.float32(7.0)).astype(np.float32))
    s = bf16_bits_to_f32(s_bits)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s[:, :, None] > 0, np.rint(w / s[:, :, None]), 0.0)
    q = np.clip(q, -8, 7).astype(np.int8).reshape(R, K)
    u = (q.astype(np.int16) & 0xF).astype(np.uint8)
    packed = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_bits


def _int3_codes_np(w_bits: np.ndarray):
    """bf16 bits [R, K] -> (int3 codes q int8 [R, K] in [-4, 3], scale bits [R, K/64])."""
    R, K = w_bits.shape
    assert K % 64 == 0
    w = bf16_bits_to_f32(w_bits).reshape(R, K // 64, 64)
    amax = np.abs(w).max(axis=2)
    s_bits = f32_to_bf16_bits((amax / np.float32(3.0)).astype(np.float32))
    s = bf16_bits_to_f32(s_bits)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s[:, :, None] > 0, np.rint(w / s[:, :, None]), 0.0)
    return np.clip(q, -4, 3).astype(np.int8).reshape(R, K), s_bits


def pack_int3_np(q: np.ndarray) -> np.ndarray:
    """int3 codes [R, K] (values in [-4, 3]) -> packed uint8 [R, 3K/8]: each 8
    consecutive codes as one little-endian 24-bit word, code j at bits 3j."""
    R, K = q.shape
    assert K % 8 == 0
    u = (q.astype(np.int16) & 0x7).astype(np.uint32).reshape(R, K // 8, 8)
    word = np.zeros((R, K // 8), dtype=np.uint32)
    for j in range(8):
        word |= u[:, :, j] << np.uint32(3 * j)
    out = np.empty((R, K // 8, 3), dtype=np.uint8)
    for b in range(3):
        out[:, :, b] = (word >> np.uint32(8 * b)) & np.uint32(0xFF)
    return out.reshape(R, 3 * K // 8)


def quantize_int3_np(w_bits: np.ndarray):
    """bf16 bits [R, K] -> (packed uint8 [R, 3K/8], scale bf16 bits uint16 [R, K/64])."""
    q, s_bits = _int3_codes_np(w_bits)
    return pack_int3_np(q), s_bits


def quantize_np(w_bits: np.ndarray, storage: str):
    if storage == "int4":
        return quantize_int4_np(w_bits)
    if storage == "int3":
        return quantize_int3_np(w_bits)
    return w_bits


def linear_np(m: ModelShape, name: str, layer: int = -1, expert=None, rows=None):
    """A linear weight in its storage format: an array (f32 values / bf16 bits),
    or for int4 / int3 a (packed, scale_bits) pair."""
    raw = raw_np(m, name, layer, expert, rows)
    return quantize_np(raw, storage_dtype(m, name))


# ---------------------------------------------------------------- torch

def _torch_table(dtype: str, device):
    import torch
    t = normal_table(dtype)
    if dtype == "f32":
        return torch.from_numpy(t.copy()).to(device)
    return torch.from_numpy(t.astype(np.int16)).view(torch.bfloat16).to(device)


def raw_torch(m: ModelShape, name: str, layer: int = -1, expert=None, device="cpu",
              chunk: int = 1 << 26):
    """Same values as raw_np, as a torch tensor (bfloat16 or float32) on `device`."""
    import torch
    dt = "f32" if m.aux_dtype == "f32" else "bf16"
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    if name in ("attn_norm", "ffn_norm", "final_norm"):
        return torch.ones(m.hidden, dtype=tdt, device=device)
    start, count, shp = _elem_range(m, name, expert, None)
    table = _torch_table(dt, device)
    key = stream_key(m.seed, tensor_id(name, layer))
    out = torch.empty(count, dtype=tdt, device=device)
    for c0 in range(0, count, chunk):
        c1 = min(count, c0 + chunk)
        idx = torch.arange(start + c0, start + c1, dtype=torch.int64, device=device)
        h = hash_torch(key, idx) >> 16
        out[c0:c1] = table[h]
    return out.view(shp)


def _bf16_rne_torch(x32):
    import torch
    b = x32.contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    b = (b + ((b >> 16) & 1) + 0x7FFF) >> 16
    return b.to(torch.int32).to(torch.int16).view(torch.bfloat16)


def quantize_int4_torch(w, rows_per_chunk: int = 8192):
    """torch bfloat16 [R, K] -> (packed uint8 [R, K/2], scales bfloat16 [R, K/64]);
    bit-identical to quantize_int4_np."""
    import torch
    R, K = w.shape
    packed = torch.empty(R, K // 2, dtype=torch.uint8, device=w.device)
    scales = torch.empty(R, K // 64, dtype=torch.bfloat16, device=w.device)
    for r0 in range(0, R, rows_per_chunk):
        r1 = min(R, r0 + rows_per_chunk)
        wf = w[r0:r1].float().view(r1 - r0, K // 64, 64)
        amax = wf.abs().amax(dim=2)
        sb = _bf16_rne_torch(amax / 7.0)
        s = sb.float()
        q = torch.where(s[:, :, None] > 0, torch.round(wf / s[:, :, None]),
                        torch.zeros_like(wf))
        q = q.clamp(-8, 7).to(torch.int16).view(r1 - r0, K) & 0xF
        packed[r0:r1] = (q[:, 0::2] | (q[:, 1::2] << 4)).to(torch.uint8)
        scales[r0:r1] = sb
    return packed, scales


def quantize_int3_torch(w, rows_per_chunk: int = 8192):
    """torch bfloat16 [R, K] -> (packed uint8 [R, 3K/8], scales bfloat16 [R, K/64]);
    bit-identical to quantize_int3_np."""
    import torch
    R, K = w.shape
    packed = torch.empty(R, 3 * K // 8, dtype=torch.uint8, device=w.device)
    scales = torch.empty(R, K // 64, dtype=torch.bfloat16, device=w.device)
    for r0 in range(0, R, rows_per_chunk):
        r1 = min(R, r0 + rows_per_chunk)
        wf = w[r0:r1].float().view(r1 - r0, K // 64, 64)
        amax = wf.abs().amax(dim=2)
        sb = _bf16_rne_torch(amax / 3.0)
        s = sb.float()
        q = torch.where(s[:, :, None] > 0, torch.round(wf / s[:, :, None]),
                        torch.zeros_like(wf))
        u = (q.clamp(-4, 3).to(torch.int32).view(r1 - r0, K // 8, 8) & 0x7)
        word = torch.zeros(r1 - r0, K // 8, dtype=torch.int32, device=w.device)
        for j in range(8):
            word |= u[:, :, j] << (3 * j)
        for b in range(3):
            packed[r0:r1].view(r1 - r0, K // 8, 3)[:, :, b] = ((word >> (8 * b)) & 0xFF).to(torch.uint8)
        scales[r0:r1] = sb
    return packed, scales


def quantize_torch(w, storage: str):
    if storage == "int4":
        return quantize_int4_torch(w)
    if storage == "int3":
        return quantize_int3_torch(w)
    return w


def linear_torch(m: ModelShape, name: str, layer: int = -1, device="cpu"):
    """Whole linear tensor in storage format on `device` (experts stacked)."""
    storage = storage_dtype(m, name)
    shape = tensor_shape(m, name)
    if len(shape) == 3:
        parts = [raw_torch(m, name, layer, e, device) for e in range(shape[0])]
        if storage not in ("int4", "int3"):
            return torch_stack(parts)
        qs = [quantize_torch(p, storage) for p in parts]
        return torch_stack([a for a, _ in qs]), torch_stack([b for _, b in qs])
    return quantize_torch(raw_torch(m, name, layer, None, device), storage)


def torch_stack(xs):
    import torch
    return torch.stack(xs, 0)


def model_torch(m: ModelShape, device="cuda") -> dict:
    """Every tensor of model m in storage format on `device`:
    {("embed",), ("final_norm",), ("lm_head",), (name, layer) ...} -> tensor or
    (packed, scales)."""
    out = {("embed",): raw_torch(m, "embed", -1, None, device),
           ("final_norm",): raw_torch(m, "final_norm", -1, None, device),
           ("lm_head",): linear_torch(m, "lm_head", -1, device)}
    for l in range(m.n_layers):
        for name in layer_tensor_names(m, l):
            if name in ("attn_norm", "ffn_norm", "router"):
                out[(name, l)] = raw_torch(m, name, l, None, device)
            else:
                out[(name, l)] = linear_torch(m, name, l, device)
    return out


def linear_fast(m: ModelShape, name: str, layer: int = -1, expert=None):
    """Same result as linear_np / raw_np (storage format, NumPy arrays), drawn
    with PyTorch's multithreaded CPU kernels (bit-identical, faster)."""
    import torch
    if name in ("attn_norm", "ffn_norm", "final_norm", "embed", "router"):
        t = raw_torch(m, name, layer, expert, "cpu")
        return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)
    t = raw_torch(m, name, layer, expert, "cpu")
    if storage_dtype(m, name) in ("int4", "int3"):
        p, s = quantize_torch(t, storage_dtype(m, name))
        return p.numpy(), s.view(torch.int16).numpy().view(np.uint16)
    return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)
