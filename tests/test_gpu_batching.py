"""Continuous batching, paging and error paths of the CUDA library (GPU).

A batched launch must give each sequence what it would get alone: the
kernel is the same, only the attention split (chunk size) and the expert
grouping differ, so residuals agree to rounding and tokens agree exactly
on these inputs.  The pool/page and error tests check the host-side state
machine through the C ABI on a real context.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import Oracle
from synth import prompts as SP
from synth import weights as SW
from moe_decode_megakernel_persistent_gb300 import _lib as L
from moe_decode_megakernel_persistent_gb300.engine import Batcher, Engine, Request
from tests import _parity as PR

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS[1].model


@pytest.fixture(scope="module")
def tiny_int4():
    m = TINY.with_(wdtype="int4")
    return m, SW.model_torch(m, "cuda")


def _prompt(m, n, seq):
    return torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, n, seq=seq)).cuda()


def _solo(m, w, prompt, steps, n_pages=32):
    eng = Engine(m, w, n_pages=n_pages, max_ctx=4096, max_seqs=4)
    tok = eng.prefill(0, prompt)
    toks = [int(tok.item())]
    L0 = prompt.numel()
    eng.enable_trace(1)
    xs = []
    for i in range(steps):
        eng.decode_step([0], tok, [L0 + i], tok)
        eng.sync()
        toks.append(int(tok.item()))
        xs.append(eng.split_trace(1)["x"][:, 0].clone())
    eng.close()
    return toks, xs


def test_batched_decode_matches_solo_runs(gpu_lib, tiny_int4):
    m, w = tiny_int4
    lens = [17, 130, 64]
    prompts = [_prompt(m, n, s) for s, n in enumerate(lens)]
    steps = 4
    solo = [_solo(m, w, p, steps) for p in prompts]
    eng = Engine(m, w, n_pages=32, max_ctx=4096, max_seqs=4)
    toks = torch.empty(3, dtype=torch.int32, device="cuda")
    for s, p in enumerate(prompts):
        eng.prefill(s, p, out=toks[s:s + 1])
    got = [[int(toks[s].item())] for s in range(3)]
    eng.enable_trace(3)
    for i in range(steps):
        eng.decode_step([0, 1, 2], toks, [lens[s] + i for s in range(3)], toks)
        eng.sync()
        tr = eng.split_trace(3)
        for s in range(3):
            got[s].append(int(toks[s].item()))
            xb = tr["x"][:, s].double().cpu().numpy()
            xs = solo[s][1][i].double().cpu().numpy()
            assert PR.rel_l2(xb, xs).max() < 1e-4
    for s in range(3):
        assert got[s] == solo[s][0]
    eng.close()


def test_batch_of_16_matches_the_oracle_per_sequence(gpu_lib, tiny_int4):
    m, w = tiny_int4
    lens = [1 + 23 * s for s in range(16)]
    eng = Engine(m, w, n_pages=64, max_ctx=4096, max_seqs=16)
    orc = Oracle(m, PR.host_fetch(m, w))
    toks = torch.empty(16, dtype=torch.int32, device="cuda")
    kvs, nxt = [], []
    for s in range(16):
        p = SP.prompt_tokens(m.seed, m.vocab, lens[s], seq=s)
        kv = orc.new_kv()
        t, _ = orc.prefill(kv, p)
        kvs.append(kv)
        nxt.append(t)
        eng.prefill(s, torch.from_numpy(p).cuda(), out=toks[s:s + 1])
    # teacher forcing: the GPU step gets the oracle's tokens
    toks.copy_(torch.tensor(nxt, dtype=torch.int32))
    eng.enable_trace(16)
    eng.decode_step(list(range(16)), toks, lens, toks)
    eng.sync()
    tr = eng.split_trace(16)
    rep = PR.Report()
    for s in range(16):
        _, tro = orc.decode(kvs[s], nxt[s], lens[s])
        PR.compare_trace(rep, m, tr, tro, slice(s, s + 1), slice(0, 1), PR.tol_for(m), f"seq {s}", seq=s)
        PR.check_token(rep, int(toks[s].item()), int(tro["next_token"][-1]), float(tro["top2_margin"][-1]),
                       f"seq {s}", seq=s)
    assert not rep.failures, rep
    eng.close()


def test_continuous_batching_with_staggered_arrivals(gpu_lib, tiny_int4):
    m, w = tiny_int4
    reqs_spec = [(0, 40), (2, 129), (3, 5), (7, 300), (7, 64)]   # (arrival step, prompt length)
    gen = 6
    eng = Engine(m, w, n_pages=32, max_ctx=4096, max_seqs=8, max_batch=4)
    reqs = [Request(seq_id=i, prompt=_prompt(m, n, i), max_new=gen, arrival=a)
            for i, (a, n) in enumerate(reqs_spec)]
    out = Batcher(eng).run(reqs)
    assert out["finish_step"] >= 7 + gen - 2
    for r in reqs:
        solo_toks, _ = _solo(m, w, r.prompt, gen - 1)
        assert r.generated == solo_toks, r.seq_id
    assert eng.info()["free_pages"] == 32        # every page returned
    eng.close()


def test_pages_are_reused_after_release(gpu_lib, tiny_int4):
    m, w = tiny_int4
    eng = Engine(m, w, n_pages=3, max_ctx=4096, max_seqs=2)
    a = _prompt(m, 300, 0)
    eng.prefill(0, a)
    eng.sync()
    assert eng.info()["free_pages"] == 0
    with pytest.raises(L.MKError) as e:
        eng.prefill(1, _prompt(m, 10, 1))
    assert e.value.code == L.MK_ERR_NO_PAGES
    assert eng.seq_length(1) == -1
    eng.release(0)
    assert eng.info()["free_pages"] == 3
    b = _prompt(m, 250, 1)
    tok = eng.prefill(1, b)
    eng.sync()
    ref, _ = _solo(m, w, b, 0)
    assert int(tok.item()) == ref[0]
    eng.close()


def test_state_errors_do_not_launch(gpu_lib, tiny_int4):
    m, w = tiny_int4
    eng = Engine(m, w, n_pages=8, max_ctx=256, max_seqs=2)
    tok = eng.prefill(0, _prompt(m, 20, 0))
    with pytest.raises(L.MKError) as e:             # wrong position
        eng.decode_step([0], tok, [19], tok)
    assert e.value.code == L.MK_ERR_STATE
    with pytest.raises(L.MKError) as e:             # duplicate sequence ids
        eng.decode_step([0, 0], torch.zeros(2, dtype=torch.int32, device="cuda"), [20, 20],
                        torch.zeros(2, dtype=torch.int32, device="cuda"))
    assert e.value.code == L.MK_ERR_INVALID_ARG
    with pytest.raises(L.MKError) as e:             # beyond max_ctx
        eng.prefill(1, _prompt(m, 300, 1))
    assert e.value.code == L.MK_ERR_INVALID_ARG
    assert eng.seq_length(0) == 20
    eng.decode_step([0], tok, [20], tok)
    eng.sync()
    assert eng.seq_length(0) == 21
    eng.close()


def test_out_of_range_token_is_reported_not_faulted(gpu_lib, tiny_int4):
    m, w = tiny_int4
    eng = Engine(m, w, n_pages=8, max_ctx=256, max_seqs=2)
    bad = torch.tensor([m.vocab + 5], dtype=torch.int32, device="cuda")
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    eng.decode_step([0], bad, [0], out)
    with pytest.raises(L.MKError) as e:
        eng.sync()
    assert e.value.code == L.MK_ERR_DEVICE_INDEX
    eng.sync()                                   # the error word was cleared
    eng.close()


def test_grid_barrier_timeout_is_reported_and_the_context_recovers(gpu_lib, tiny_int4):
    """Block 0 skips its arrival at the third grid barrier; the other blocks'
    bounded waits run out (limit 2 ms), the kernel returns, and mk_sync
    reports MK_ERR_BARRIER_TIMEOUT.  Nothing traps or hangs."""
    m, w = tiny_int4
    eng = Engine(m, w, n_pages=8, max_ctx=256, max_seqs=2)
    tok = eng.prefill(0, _prompt(m, 20, 0))
    eng.sync()
    L.mk_set_debug(eng.ctx, L.MK_DBG_SKIP_ARRIVAL, (3 << 16) | 0, 0, 0, 2000)
    eng.decode_step([0], tok, [20], tok)
    with pytest.raises(L.MKError) as e:
        eng.sync()
    assert e.value.code == L.MK_ERR_BARRIER_TIMEOUT
    L.mk_set_debug(eng.ctx, 0, 0, 0, 0, 0)
    eng.release(0)
    p = _prompt(m, 33, 1)
    tok = eng.prefill(1, p)
    eng.sync()
    ref, _ = _solo(m, w, p, 0)
    assert int(tok.item()) == ref[0]
    eng.close()


def test_kv_write_read_roundtrip_and_errors(gpu_lib, tiny_int4):
    m, w = tiny_int4
    eng = Engine(m, w, n_pages=4, max_ctx=1024, max_seqs=3)
    g = torch.Generator(device="cuda").manual_seed(5)
    kv = (torch.randn((m.n_layers, 300, 2, m.n_kv_heads, m.head_dim), generator=g, device="cuda")
          .to(torch.bfloat16))
    eng.kv_write(0, 0, kv)                           # opens the sequence, takes 3 pages
    assert eng.seq_length(0) == 300 and eng.info()["free_pages"] == 1
    assert torch.equal(eng.kv_read(0, 0, 300).view(torch.int16), kv.view(torch.int16))
    part = kv[:, 10:20].flip(0).contiguous()         # overwrite positions 10..19
    eng.kv_write(0, 10, part)
    got = eng.kv_read(0, 0, 300)
    assert torch.equal(got[:, 10:20].view(torch.int16), part.view(torch.int16))
    assert torch.equal(got[:, :10].view(torch.int16), kv[:, :10].view(torch.int16))
    assert torch.equal(got[:, 20:].view(torch.int16), kv[:, 20:].view(torch.int16))
    with pytest.raises(L.MKError) as e:              # a gap after the length
        eng.kv_write(0, 301, kv[:, :1].contiguous())
    assert e.value.code == L.MK_ERR_STATE
    with pytest.raises(L.MKError) as e:              # needs 2 more pages, 1 left: nothing written
        eng.kv_write(1, 0, kv[:, :200].contiguous())
    assert e.value.code == L.MK_ERR_NO_PAGES and eng.seq_length(1) == -1
    with pytest.raises(L.MKError) as e:
        eng.kv_read(0, 290, 20)                      # past the length
    assert e.value.code == L.MK_ERR_STATE
    eng.close()


def test_fork_shares_pages_and_gives_the_same_tokens(gpu_lib, tiny_int4):
    m, w = tiny_int4
    eng = Engine(m, w, n_pages=8, max_ctx=1024, max_seqs=3)
    a = _prompt(m, 300, 0)
    # the source in the same two chunks the fork replays (a chunk's GEMMs
    # are the same launches, so the results are the same bits)
    eng.prefill(0, a[:256])
    ta = eng.prefill(0, a[256:], start_pos=256).clone()
    eng.sync()
    free0 = eng.info()["free_pages"]                 # 8 - 3
    eng.fork(0, 1, 256)                              # shares 2 pages, takes none
    assert eng.info()["free_pages"] == free0 and eng.seq_length(1) == 256
    tb = eng.prefill(1, a[256:], start_pos=256)      # the same positions, same launch grouping
    eng.sync()
    assert int(tb.item()) == int(ta.item())
    assert torch.equal(eng.kv_read(1, 0, 300).view(torch.int16), eng.kv_read(0, 0, 300).view(torch.int16))
    with pytest.raises(L.MKError) as e:              # position 5 is in a shared page
        eng.kv_write(0, 5, torch.zeros((m.n_layers, 1, 2, m.n_kv_heads, m.head_dim),
                                       dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == L.MK_ERR_STATE
    with pytest.raises(L.MKError) as e:              # not whole pages
        eng.fork(0, 2, 200)
    assert e.value.code == L.MK_ERR_INVALID_ARG
    eng.release(0)                                   # the shared pages stay with sequence 1
    assert eng.info()["free_pages"] == 8 - 3
    tok = tb.clone()
    eng.decode_step([1], tok, [300], tok)
    eng.sync()
    eng.release(1)
    assert eng.info()["free_pages"] == 8
    eng.close()


def test_prefix_cache_a_a_b_a(gpu_lib, tiny_int4):
    """The prefix-cache sequence of turns A, A, B, A: the second and the last
    turn over prompt A reuse its whole pages (512 of 600 tokens); every turn's
    next token is the oracle's wherever the oracle's top-2 margin is clear."""
    from moe_decode_megakernel_persistent_gb300.engine import PrefixCache
    m, w = tiny_int4
    orc = Oracle(m, PR.host_fetch(m, w))
    ref = {}
    for name, seq in (("A", 0), ("B", 1)):
        p = SP.prompt_tokens(m.seed, m.vocab, 600, seq=seq)
        tok, tr = orc.prefill(orc.new_kv(), p)
        ref[name] = (tok, float(tr["top2_margin"][-1]))
    A, B = _prompt(m, 600, 0), _prompt(m, 600, 1)
    eng = Engine(m, w, n_pages=32, max_ctx=1024, max_seqs=8)
    pc = PrefixCache(eng, capacity=2)
    reused, rep = [], PR.Report()
    for sid, (name, p) in enumerate((("A", A), ("A", A), ("B", B), ("A", A))):
        out, n = pc.prefill(sid, p)
        eng.sync()
        reused.append(n)
        PR.check_token(rep, int(out.item()), ref[name][0], ref[name][1], f"turn {sid} ({name})", seq=sid)
        pc.keep(sid, p.cpu().tolist())
    assert reused == [0, 512, 0, 512]
    assert not rep.failures, rep
    eng.close()
