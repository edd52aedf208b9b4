"""The allocation-free decode entry point against the context-based one.

mk_decode_step_static is for callers that cannot call cudaMalloc: a host that
hands the library a fixed memory budget from its own allocator, or a loop
that must not take the device-wide synchronisation an allocation can bring.
It runs the same kernel with its scratch in a static device array, so on the
same inputs and the same launch shapes it must give the same tokens as
mk_prefill_chunk / mk_decode_step, bit for bit (the tolerance of the other
tests is met a fortiori): over a prompt that crosses a page boundary and then
two decode calls in a row; with two rows per launch on the Flint shape; and
with two models of different RoPE theta taking turns on the shared array.
The caller-owned KV pool and block table are allocated with PyTorch, as such
a caller would have them.  This file sorts last so a failure here leaves
every other test already run.
"""
import pytest
import torch

import synth
from synth import prompts as SP
from synth import weights as SW
from moe_decode_megakernel_persistent_gb300 import _lib as L
from moe_decode_megakernel_persistent_gb300.engine import Engine, _ptr
from tests._models import weights_struct as _weights_struct

pytestmark = pytest.mark.gpu

PROMPT = 140          # crosses the 128-position page boundary
DECODE = 2            # two calls in a row after the prompt


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


def _static_ctx(m, w, n_pages, max_ctx, max_seqs=4, max_batch=16):
    """Caller-owned buffers for the allocation-free entry point."""
    from moe_decode_megakernel_persistent_gb300.engine import make_desc
    d = make_desc(m, max_batch=max_batch, max_ctx=max_ctx, max_seqs=max_seqs)
    ws, keep = _weights_struct(m, w)
    packed = torch.empty(L.mk_packed_bytes(d), dtype=torch.uint8, device="cuda")
    L.mk_pack_weights(d, ws, _ptr(packed), packed.numel(), torch.cuda.current_stream().cuda_stream)
    page_elems = m.n_layers * 2 * m.n_kv_heads * 128 * m.head_dim
    kv = torch.zeros(n_pages * page_elems, dtype=torch.int16, device="cuda")
    maxpp = (max_ctx + 127) // 128
    table = torch.full((max_seqs, maxpp), -1, dtype=torch.int32, device="cuda")
    return dict(d=d, ws=ws, keep=keep, packed=packed, kv=kv, table=table, maxpp=maxpp, n_pages=n_pages)


def _static_step(c, slots, positions, pages, tin, tout, status):
    L.mk_decode_step_static(c["d"], c["ws"], _ptr(c["packed"]), _ptr(c["kv"]), c["n_pages"], _ptr(c["table"]),
                            c["maxpp"], slots, positions, pages, _ptr(tin), _ptr(tout), _ptr(status),
                            torch.cuda.current_stream().cuda_stream)


def test_static_entry_two_rows_flint_shape(gpu_lib):
    """Two sequences in one launch on the Flint shape (layers 0-3 of the int4
    model: two dense, two MoE), whose scratch must fit the static array: the
    prompts run one position per call, then two calls in a row decode both
    rows together; tokens equal the context entry point's."""
    m = synth.CONFIGS[3].model.with_(n_layers=4)
    w = SW.model_torch(m, "cuda")
    lens = [40, 33]
    prompts = [torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, n, seq=s)).cuda() for s, n in enumerate(lens)]
    max_ctx = 64
    eng = Engine(m, w, n_pages=4, max_ctx=max_ctx, max_seqs=4)
    out = torch.empty(2, dtype=torch.int32, device="cuda")
    for s, p in enumerate(prompts):
        for i in range(lens[s]):
            L.mk_prefill_chunk(eng.ctx, s, _ptr(p) + 4 * i, 1, i, _ptr(out[s:s + 1]), eng.stream)
    ref = [out.cpu().tolist()]
    for i in range(DECODE):
        eng.decode_step([0, 1], out, [lens[0] + i, lens[1] + i], out)
        ref.append(out.cpu().tolist())
    eng.sync()
    eng.close()

    c = _static_ctx(m, w, n_pages=4, max_ctx=max_ctx)
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got_out = torch.empty(2, dtype=torch.int32, device="cuda")
    for s, p in enumerate(prompts):         # sequence s owns page s
        for i in range(lens[s]):
            _static_step(c, [s], [i], [s], p[i:i + 1], got_out[s:s + 1], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = [got_out.cpu().tolist()]
    for i in range(DECODE):
        _static_step(c, [0, 1], [lens[0] + i, lens[1] + i], [0, 1], got_out, got_out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got.append(got_out.cpu().tolist())
    assert got == ref


def test_static_entry_models_with_different_rope_take_turns(gpu_lib):
    """Two tiny models that differ only in RoPE theta (1e4 and 10) share the static array:
    calls alternate between them (each switch rewrites the tables after the
    device is idle); each model's tokens equal its context entry point's."""
    base = synth.CONFIGS[1].model
    models = [base, base.with_(rope_theta=10.0)]
    w = SW.model_torch(base, "cuda")
    plen, steps = 20, 2
    prompt = torch.from_numpy(SP.prompt_tokens(base.seed, base.vocab, plen)).cuda()
    refs = []
    for m in models:
        eng = Engine(m, w, n_pages=2, max_ctx=64, max_seqs=2)
        out = torch.empty(1, dtype=torch.int32, device="cuda")
        toks = []
        for i in range(plen):
            L.mk_prefill_chunk(eng.ctx, 0, _ptr(prompt) + 4 * i, 1, i, _ptr(out), eng.stream)
            toks.append(int(out.item()))
        for i in range(steps):
            eng.decode_step([0], out, [plen + i], out)
            toks.append(int(out.item()))
        eng.close()
        refs.append(toks)
    assert refs[0] != refs[1]          # the theta change matters for these tokens
    cs = [_static_ctx(m, w, n_pages=2, max_ctx=64) for m in models]
    outs = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in models]
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = [[], []]
    for i in range(plen + steps):
        for k in (0, 1):               # the models take turns on every position
            tin = prompt[i:i + 1] if i < plen else outs[k]
            _static_step(cs[k], [0], [i], [0], tin, outs[k], status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            got[k].append(int(outs[k].item()))
    assert got == refs
