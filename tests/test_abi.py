"""The C-ABI library: builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes as C
import os
import re

import pytest

import synth
from moe_decode_megakernel_persistent_gb300 import _build
from moe_decode_megakernel_persistent_gb300 import _lib as L
from moe_decode_megakernel_persistent_gb300.engine import make_desc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return L.load()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "mk.h")).read()
    return set(re.findall(r"MK_API\s+[\w\s\*]+?\b(mk_\w+)\s*\(", text))


def test_header_declares_the_four_boundary_calls():
    syms = header_symbols()
    assert {"mk_create", "mk_kv_alloc", "mk_decode_step", "mk_prefill_chunk"} <= syms


def test_library_exports_every_declared_symbol(lib):
    syms = header_symbols()
    for s in syms:
        assert hasattr(lib, s), s
    assert syms == set(L.SIGNATURES), "binding covers exactly the declared ABI"


def _desc(cfg=1, **kw):
    d = make_desc(synth.CONFIGS[cfg].model)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_create_rejects_bad_descriptions_without_cuda(lib):
    out = C.c_void_p()
    w = L.mk_weights()
    assert lib.mk_create(None, C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert lib.mk_create(C.byref(_desc()), C.byref(w), None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_create(C.byref(_desc(hidden=512)), C.byref(w), C.byref(out)) == L.MK_ERR_UNSUPPORTED
    assert lib.mk_create(C.byref(_desc(page_tokens=64)), C.byref(w), C.byref(out)) == L.MK_ERR_UNSUPPORTED
    assert lib.mk_create(C.byref(_desc(max_batch=17)), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert lib.mk_create(C.byref(_desc(wdtype=9)), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert lib.mk_create(C.byref(_desc(n_dense=5)), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    # host tables sized by max_ctx and max_seqs are bounded
    assert lib.mk_create(C.byref(_desc(max_ctx=(1 << 20) + 1)), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert lib.mk_create(C.byref(_desc(max_seqs=(1 << 16) + 1)), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert lib.mk_create(C.byref(_desc(max_ctx=2 ** 31 - 1)), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert lib.mk_create(C.byref(_desc()), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert "NULL" in L.mk_last_error()
    assert out.value is None


def test_create_rejects_misaligned_weights(lib):
    d = _desc()
    layers = (L.mk_layer_weights * d.n_layers)()
    w = L.mk_weights(embed=0x1000, final_norm=0x2000, lm_head=L.mk_linear(0x3008, None), layers=layers)
    out = C.c_void_p()
    assert lib.mk_create(C.byref(d), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert "lm_head" in L.mk_last_error()
    w.lm_head = L.mk_linear(0x3000, None)
    assert lib.mk_create(C.byref(d), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert "attn_norm" in L.mk_last_error()


def test_expert_format_is_validated_and_sizes_the_packed_weights(lib):
    out = C.c_void_p()
    w = L.mk_weights()
    # int3 experts only come with int4 layers
    assert lib.mk_create(C.byref(_desc(expert_wdtype=L.MK_INT3_G64)), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert "expert_wdtype" in L.mk_last_error()
    assert lib.mk_create(C.byref(_desc(expert_wdtype=L.MK_BF16)), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert "expert_wdtype" in L.mk_last_error()
    # a valid mixed description gets past the description to the weights
    d = make_desc(synth.FLINT_INT4_E3)
    assert d.expert_wdtype == L.MK_INT3_G64 and d.wdtype == L.MK_INT4_G64
    assert lib.mk_create(C.byref(d), C.byref(w), C.byref(out)) == L.MK_ERR_INVALID_ARG
    assert "NULL" in L.mk_last_error()
    # packed bytes by hand: per MoE layer the gate/up records (2 x 64 x 768 rows
    # of K = 2048) shrink from 1024 + 64 to 768 + 64 bytes, the down records
    # (64 x 2048 rows of K = 768) from 384 + 24 -> 416 to 288 + 24 -> 320 bytes
    n4 = L.mk_packed_bytes(make_desc(synth.CONFIGS[3].model))
    n3 = L.mk_packed_bytes(d)
    per_layer = 2 * 64 * 768 * (1088 - 832) + 64 * 2048 * (416 - 320)
    assert n4 - n3 == 47 * per_layer


def test_null_context_calls_fail_cleanly(lib):
    assert lib.mk_kv_alloc(None, 4) == L.MK_ERR_INVALID_ARG
    ids = (C.c_int32 * 1)(0)
    assert lib.mk_decode_step(None, ids, 16, ids, 1, 16, None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_prefill_chunk(None, 0, 16, 1, 0, None, None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_seq_release(None, 0) == L.MK_ERR_INVALID_ARG
    assert lib.mk_seq_length(None, 0) == -1
    assert lib.mk_sync(None, None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_get_info(None, None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_destroy(None) == L.MK_OK


def test_trace_bytes_layout(lib):
    m = synth.CONFIGS[3].model
    d = make_desc(m)
    per_layer = m.hidden + m.n_heads * m.head_dim + m.n_experts + 2 * m.top_k
    assert L.mk_trace_bytes(d, 3) == 4 * (m.n_layers * 3 * per_layer + 3 * m.vocab)
    assert L.mk_trace_bytes(d, 0) == 0


def test_static_array_holds_the_flint_models_on_152_sms(lib):
    """The allocation-free entry point keeps the RoPE table (8192 positions x
    head_dim / 2 cos/sin pairs of fp32), the layer table and the kernel scratch
    in one 8 MiB array: every benchmarked Flint model fits it on GB300's 152
    SMs, and a grid far above that (more blocks, more attention partials) is
    one the entry point would reject."""
    models = [c.model for c in synth.CONFIGS.values()] + [c.model for c in synth.EXTRA.values()]
    for m in models:
        d = make_desc(m)
        need, cap = L.mk_static_bytes(d, 152)
        assert cap == 8 << 20
        assert 8192 * (m.head_dim // 2) * 8 < need <= cap, (m, need)
        assert L.mk_static_bytes(d, 1)[0] <= need <= L.mk_static_bytes(d, 304)[0]
    need, cap = L.mk_static_bytes(_desc(3), 1024)
    assert need > cap
    with pytest.raises(L.MKError) as e:
        L.mk_static_bytes(_desc(3), 0)
    assert e.value.code == L.MK_ERR_INVALID_ARG
    with pytest.raises(L.MKError) as e:
        L.mk_static_bytes(_desc(3, hidden=512), 152)
    assert e.value.code == L.MK_ERR_UNSUPPORTED


def test_per_row_lists_must_match_the_row_count(lib):
    """The binding refuses lists shorter or longer than the rows it passes
    (the library reads n host values from each)."""
    with pytest.raises(ValueError):
        L.mk_decode_step(None, [0, 1], 0, [5], 0)
    with pytest.raises(ValueError):
        L.mk_decode_step_static(_desc(), L.mk_weights(), 0, 0, 1, 0, 1, [0], [3, 4], [0], 0, 0)
