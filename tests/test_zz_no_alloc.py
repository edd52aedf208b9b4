"""The allocation-free decode entry point against the context-based one.

mk_decode_step_static serves callers that cannot call cudaMalloc (code under
stream capture, hosts that hand the library a fixed memory budget, loops that
must not take an allocation's implicit synchronisation).  It runs the same
kernel with its scratch in a static device array, so on the same inputs and
the same launch shapes it must give the same tokens as mk_prefill_chunk /
mk_decode_step, bit for bit: here over a prompt that crosses a page boundary
and then two decode calls in a row.  The test allocates the caller-owned KV
pool and block table with PyTorch, as such a caller would have them.
This file sorts last so a failure here leaves every other test already run.
"""
import pytest
import torch

import synth
from synth import prompts as SP
from synth import weights as SW
from moe_decode_megakernel_persistent_gb300 import _lib as L
from moe_decode_megakernel_persistent_gb300.engine import Engine, _lin, _ptr

pytestmark = pytest.mark.gpu

PROMPT = 140          # crosses the 128-position page boundary
DECODE = 2            # two calls in a row after the prompt


def _weights_struct(m, w):
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


@pytest.mark.parametrize("wdtype", ["f32", "int4"])
def test_static_entry_matches_context_entry(gpu_lib, wdtype):
    m = synth.CONFIGS[1].model.with_(wdtype=wdtype)
    w = SW.model_torch(m, "cuda")
    prompt = torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, PROMPT)).cuda()
    max_ctx = PROMPT + DECODE + 8
    n_pages = 4

    # the existing entry points, one position per launch
    eng = Engine(m, w, n_pages=n_pages, max_ctx=max_ctx, max_seqs=4)
    ref = []
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    for p in range(PROMPT):
        L.mk_prefill_chunk(eng.ctx, 0, _ptr(prompt) + 4 * p, 1, p, _ptr(out), eng.stream)
        ref.append(int(out.item()))
    tok = out.clone()
    for i in range(DECODE):
        eng.decode_step([0], tok, [PROMPT + i], tok)
        ref.append(int(tok.item()))
    eng.sync()
    eng.close()

    # the allocation-free entry point on caller-owned packed weights, KV pool
    # and block table
    desc = eng.desc
    ws, _keep = _weights_struct(m, w)
    pbytes = L.mk_packed_bytes(desc)
    assert pbytes > 0
    packed = torch.empty(pbytes, dtype=torch.uint8, device="cuda")
    L.mk_pack_weights(desc, ws, _ptr(packed), pbytes, torch.cuda.current_stream().cuda_stream)
    page_elems = m.n_layers * 2 * m.n_kv_heads * 128 * m.head_dim
    kv = torch.zeros(n_pages * page_elems, dtype=torch.int16, device="cuda")
    maxpp = (max_ctx + 127) // 128
    table = torch.full((desc.max_seqs, maxpp), -1, dtype=torch.int32, device="cuda")
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    got = []
    for p in range(PROMPT + DECODE):
        tin = prompt[p:p + 1] if p < PROMPT else out
        L.mk_decode_step_static(desc, ws, _ptr(packed), _ptr(kv), n_pages, _ptr(table), maxpp, [0], [p],
                                [p // 128],
                                _ptr(tin), _ptr(out), _ptr(status), stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got.append(int(out.item()))
    assert got == ref
    assert table[0, :2].tolist() == [0, 1]


def test_static_entry_rejects_out_of_range_input(gpu_lib):
    m = synth.CONFIGS[1].model
    w = SW.model_torch(m, "cuda")
    from moe_decode_megakernel_persistent_gb300.engine import make_desc
    d = make_desc(m, max_ctx=16384)
    ws, _keep = _weights_struct(m, w)
    packed = torch.empty(L.mk_packed_bytes(d), dtype=torch.uint8, device="cuda")
    L.mk_pack_weights(d, ws, _ptr(packed), packed.numel(), torch.cuda.current_stream().cuda_stream)
    kv = torch.zeros(1024, dtype=torch.int16, device="cuda")
    table = torch.zeros((64, 128), dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(L.MKError) as e:      # beyond the static RoPE table
        L.mk_decode_step_static(d, ws, _ptr(packed), _ptr(kv), 1, _ptr(table), 128, [0], [8192], [0],
                                _ptr(tok), _ptr(tok))
    assert e.value.code == L.MK_ERR_INVALID_ARG and "8192" in str(e.value)
    with pytest.raises(L.MKError) as e:      # page outside the caller's pool
        L.mk_decode_step_static(d, ws, _ptr(packed), _ptr(kv), 1, _ptr(table), 128, [0], [0], [3],
                                _ptr(tok), _ptr(tok))
    assert e.value.code == L.MK_ERR_INVALID_ARG
