"""ctypes binding of libmk.so (include/mk.h): the same entry points under the
same names, argument marshalling only.  Every compute step runs in the
library's CUDA kernel; there is no fallback when the library is missing."""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmk.so")

MK_OK = 0
MK_ERR_INVALID_ARG = 1
MK_ERR_NO_PAGES = 2
MK_ERR_STATE = 3
MK_ERR_CUDA = 4
MK_ERR_UNSUPPORTED = 5
MK_ERR_BARRIER_TIMEOUT = 6
MK_ERR_DEVICE_INDEX = 7
ERR_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "NO_PAGES", 3: "STATE", 4: "CUDA",
             5: "UNSUPPORTED", 6: "BARRIER_TIMEOUT", 7: "DEVICE_INDEX"}

MK_F32, MK_BF16, MK_INT4_G64, MK_INT3_G64 = 0, 1, 2, 3
WDTYPES = {"f32": MK_F32, "bf16": MK_BF16, "int4": MK_INT4_G64, "int3": MK_INT3_G64}
MK_DBG_TRACE = 1
MK_DBG_SKIP_ARRIVAL = 2
MK_DBG_TIMING = 4
MK_DBG_SPLIT = 8


class MKError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


class mk_model_desc(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("vocab", C.c_int32),
                ("n_dense", C.c_int32), ("dense_ffn", C.c_int32), ("n_experts", C.c_int32),
                ("top_k", C.c_int32), ("expert_ffn", C.c_int32), ("rope_theta", C.c_float),
                ("rms_eps", C.c_float), ("wdtype", C.c_int32), ("page_tokens", C.c_int32),
                ("max_batch", C.c_int32), ("max_ctx", C.c_int32), ("max_seqs", C.c_int32),
                ("expert_wdtype", C.c_int32)]


class mk_linear(C.Structure):
    _fields_ = [("w", C.c_void_p), ("scales", C.c_void_p)]


class mk_layer_weights(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("wq", mk_linear), ("wk", mk_linear),
                ("wv", mk_linear), ("wo", mk_linear), ("ffn_norm", C.c_void_p),
                ("gate", mk_linear), ("up", mk_linear), ("down", mk_linear),
                ("router", C.c_void_p), ("exp_gate", mk_linear), ("exp_up", mk_linear),
                ("exp_down", mk_linear)]


class mk_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", mk_linear),
                ("layers", C.POINTER(mk_layer_weights))]


class mk_info(C.Structure):
    _fields_ = [("device", C.c_int32), ("num_sms", C.c_int32), ("grid", C.c_int32),
                ("block_threads", C.c_int32), ("smem_bytes", C.c_int32), ("n_pages", C.c_int32),
                ("free_pages", C.c_int32), ("scratch_bytes", C.c_int64), ("kv_bytes", C.c_int64),
                ("last_chunk", C.c_int32), ("last_units", C.c_int32)]


# every symbol include/mk.h declares, with its ctypes signature
SIGNATURES = {
    "mk_create": (C.c_int, [C.POINTER(mk_model_desc), C.POINTER(mk_weights), C.POINTER(C.c_void_p)]),
    "mk_kv_alloc": (C.c_int, [C.c_void_p, C.c_int32]),
    "mk_prefill_chunk": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_int32,
                                   C.c_void_p, C.c_void_p]),
    "mk_decode_step": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.c_void_p,
                                 C.POINTER(C.c_int32), C.c_int32, C.c_void_p, C.c_void_p]),
    "mk_seq_release": (C.c_int, [C.c_void_p, C.c_int32]),
    "mk_kv_write": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "mk_kv_read": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "mk_seq_fork": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p]),
    "mk_seq_length": (C.c_int32, [C.c_void_p, C.c_int32]),
    "mk_sync": (C.c_int, [C.c_void_p, C.c_void_p]),
    "mk_set_debug": (C.c_int, [C.c_void_p, C.c_uint32, C.c_uint32, C.c_void_p, C.c_size_t,
                               C.c_uint32]),
    "mk_trace_bytes": (C.c_size_t, [C.POINTER(mk_model_desc), C.c_int32]),
    "mk_get_info": (C.c_int, [C.c_void_p, C.POINTER(mk_info)]),
    "mk_attention_plan": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_int32), C.c_int32,
                                    C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    "mk_destroy": (C.c_int, [C.c_void_p]),
    "mk_last_error": (C.c_char_p, []),
    "mk_packed_bytes": (C.c_size_t, [C.POINTER(mk_model_desc)]),
    "mk_pack_weights": (C.c_int, [C.POINTER(mk_model_desc), C.POINTER(mk_weights), C.c_void_p, C.c_size_t,
                                  C.c_void_p]),
    "mk_decode_step_static": (C.c_int, [C.POINTER(mk_model_desc), C.POINTER(mk_weights), C.c_void_p,
                                        C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.POINTER(C.c_int32),
                                        C.POINTER(C.c_int32), C.POINTER(C.c_int32), C.c_int32,
                                        C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "mk_static_bytes": (C.c_int, [C.POINTER(mk_model_desc), C.c_int32, C.POINTER(C.c_int64),
                                  C.POINTER(C.c_int64)]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load libmk.so (built in-tree by __graft_entry__.build()); fails loudly."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(code: int):
    if code != MK_OK:
        raise MKError(code, (_lib.mk_last_error() or b"").decode())


def _i32(xs, n: int | None = None):
    """Host int32 array of xs; with n, xs must hold exactly n values (the
    library reads n of them)."""
    if n is not None and len(xs) != n:
        raise ValueError(f"expected {n} values, got {len(xs)}")
    arr = (C.c_int32 * len(xs))(*[int(x) for x in xs])
    return arr


# ---- thin wrappers, same names as the C ABI ----

def mk_create(desc: mk_model_desc, weights: mk_weights) -> int:
    lib = load()
    out = C.c_void_p()
    _check(lib.mk_create(C.byref(desc), C.byref(weights), C.byref(out)))
    return out.value


def mk_kv_alloc(ctx: int, n_pages: int):
    _check(load().mk_kv_alloc(ctx, n_pages))


def mk_prefill_chunk(ctx: int, seq_id: int, tokens_dev: int, n: int, start_pos: int,
                     out_token_dev: int | None, stream: int = 0):
    _check(load().mk_prefill_chunk(ctx, seq_id, tokens_dev, n, start_pos, out_token_dev, stream))


def mk_decode_step(ctx: int, seq_ids, tokens_dev: int, positions, out_tokens_dev: int,
                   stream: int = 0):
    n = len(seq_ids)
    _check(load().mk_decode_step(ctx, _i32(seq_ids), tokens_dev, _i32(positions, n), n,
                                 out_tokens_dev, stream))


def mk_seq_release(ctx: int, seq_id: int):
    _check(load().mk_seq_release(ctx, seq_id))


def mk_kv_write(ctx: int, seq_id: int, start_pos: int, n: int, src_dev: int, stream: int = 0):
    _check(load().mk_kv_write(ctx, seq_id, start_pos, n, src_dev, stream))


def mk_kv_read(ctx: int, seq_id: int, start_pos: int, n: int, dst_dev: int, stream: int = 0):
    _check(load().mk_kv_read(ctx, seq_id, start_pos, n, dst_dev, stream))


def mk_seq_fork(ctx: int, src_seq: int, dst_seq: int, n_tokens: int, stream: int = 0):
    _check(load().mk_seq_fork(ctx, src_seq, dst_seq, n_tokens, stream))


def mk_seq_length(ctx: int, seq_id: int) -> int:
    return load().mk_seq_length(ctx, seq_id)


def mk_sync(ctx: int, stream: int = 0):
    _check(load().mk_sync(ctx, stream))


def mk_set_debug(ctx: int, flags: int, arg: int = 0, trace_dev: int = 0, trace_bytes: int = 0,
                 spin_limit_us: int = 0):
    _check(load().mk_set_debug(ctx, flags, arg, trace_dev, trace_bytes, spin_limit_us))


def mk_trace_bytes(desc: mk_model_desc, rows: int) -> int:
    return load().mk_trace_bytes(C.byref(desc), rows)


def mk_attention_plan(n_kv_heads: int, grid: int, tile_tokens: int, positions) -> tuple:
    """(chunk, units) of the attention split for rows at these new positions."""
    pos = (C.c_int32 * len(positions))(*positions)
    ch, u = C.c_int32(), C.c_int32()
    _check(load().mk_attention_plan(n_kv_heads, grid, tile_tokens, pos, len(positions), C.byref(ch), C.byref(u)))
    return ch.value, u.value


def mk_get_info(ctx: int) -> dict:
    info = mk_info()
    _check(load().mk_get_info(ctx, C.byref(info)))
    return {k: getattr(info, k) for k, _ in mk_info._fields_}


def mk_destroy(ctx: int):
    _check(load().mk_destroy(ctx))


def mk_packed_bytes(desc: mk_model_desc) -> int:
    return int(load().mk_packed_bytes(C.byref(desc)))


def mk_static_bytes(desc: mk_model_desc, grid: int) -> tuple:
    """(bytes needed, bytes held) of the allocation-free entry point's array
    for this model on a device of `grid` SMs."""
    need, cap = C.c_int64(), C.c_int64()
    _check(load().mk_static_bytes(C.byref(desc), grid, C.byref(need), C.byref(cap)))
    return need.value, cap.value


def mk_pack_weights(desc: mk_model_desc, weights: mk_weights, dst_dev: int, dst_bytes: int, stream: int = 0):
    """Pack the linear weights into a caller-owned device buffer (for the
    allocation-free entry point)."""
    _check(load().mk_pack_weights(C.byref(desc), C.byref(weights), dst_dev, dst_bytes, stream))


def mk_decode_step_static(desc: mk_model_desc, weights: mk_weights, packed_dev: int, kv_dev: int, n_pages: int,
                          block_table_dev: int, max_pages_per_seq: int, slots, positions, pages,
                          tokens_dev: int, out_tokens_dev: int, status_dev: int = 0, stream: int = 0):
    """Decode step with no device allocation (scratch in the library's static
    device array); for callers that cannot call cudaMalloc."""
    n = len(slots)
    _check(load().mk_decode_step_static(C.byref(desc), C.byref(weights), packed_dev, kv_dev, n_pages,
                                        block_table_dev, max_pages_per_seq, _i32(slots),
                                        _i32(positions, n), _i32(pages, n), n, tokens_dev,
                                        out_tokens_dev, status_dev or None, stream))


def mk_last_error() -> str:
    return (load().mk_last_error() or b"").decode()
