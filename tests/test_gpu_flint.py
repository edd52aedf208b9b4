"""The Flint-shaped model (hidden 2048, 16 / 4 heads of 128, 64 experts top-6,
expert FFN 768, dense FFN 6144, vocabulary 151936) against the oracle, in the
launch configuration the bench times (one block per SM).

- Full depth (49 layers): a short prompt, so that the float64 oracle finishes
  in about a minute, then teacher-forced decode over the oracle's cache.
- Reduced depth (layers 0-3 of the same model: two dense, two MoE; the
  weights of a layer do not depend on the depth) at the bench's contexts:
  a 2048-token prompt (the int4 and bf16 workloads) and an 8022-token prompt
  prefilled in 4096-token chunks (the long-context workload), and a
  continuous batch of 16 sequences joining at staggered steps (the batched
  workload, lengths and arrivals scaled down so the oracle stays within
  about a minute).
- Two runs of the same launches give the same bits.

Integer rules (top-6 ids where the oracle's margin exceeds 1e-3, tokens where
its top-2 margin exceeds 0.05) are exact; every run must pin at least 40
top-k decisions and at least one token.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import Oracle
from synth import prompts as SP
from synth import weights as SW
from moe_decode_megakernel_persistent_gb300.engine import Engine
from tests import _parity as PR

pytestmark = pytest.mark.gpu

MIN_TOPK = 40


def _check(rep):
    print(rep)
    assert not rep.failures, rep
    assert rep.topk_checked >= MIN_TOPK, rep
    assert rep.tokens_checked >= 1, rep


def _reduced(cfg, n_layers=4):
    return synth.CONFIGS[cfg].model.with_(n_layers=n_layers)


@pytest.mark.parametrize("cfg", [3, 2])
def test_flint_full_depth_matches_the_oracle(gpu_lib, cfg):
    m = synth.CONFIGS[cfg].model
    w = SW.model_torch(m, "cuda")
    rep = PR.run_single(m, prompt_len=2, n_decode=4, w=w, n_pages=8, teacher=True)
    _check(rep)
    del w
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def flint4_int4():
    m = _reduced(3)
    w = SW.model_torch(m, "cuda")
    yield m, w
    del w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", [3, 2])
def test_flint_reduced_depth_context_2048(gpu_lib, cfg):
    m = _reduced(cfg)
    w = SW.model_torch(m, "cuda")
    rep = PR.run_single(m, prompt_len=2048, n_decode=8, w=w, n_pages=24, teacher=True)
    _check(rep)


def test_flint_reduced_depth_context_8022(gpu_lib, flint4_int4):
    """8022-token prompt: the oracle's cache for the first 8006 positions, the
    GPU prefills the last 16 rows and decodes 8 steps over it."""
    m, w = flint4_int4
    rep = PR.run_single(m, prompt_len=8022, n_decode=8, w=w, n_pages=72, teacher=True)
    _check(rep)


def test_flint_chunked_prefill_writes_every_position(gpu_lib, flint4_int4):
    """The GPU's own prefill of 8022 tokens (two chunks, 4096 + 3926) over its
    own cache: layer 0's K/V depend on the embedding rows alone, so they must
    equal the oracle's at every position up to bf16 rounding flips (every
    page and slot the prefill wrote); the last launch's rows stay within the
    float tolerance."""
    m, w = flint4_int4
    n = 8022
    prompt = SP.prompt_tokens(m.seed, m.vocab, n, seq=3)
    orc = Oracle(m, PR.host_fetch(m, w), cache_bytes=8 << 30)
    kv = orc.new_kv()
    _, tr_o = orc.prefill(kv, prompt)
    eng = Engine(m, w, n_pages=72, max_ctx=n + 16, max_seqs=2)
    eng.enable_trace(16)
    eng.prefill(0, torch.from_numpy(prompt).cuda())
    eng.sync()
    assert eng.seq_length(0) == n
    rep = PR.Report()
    got = eng.kv_read(0, 0, n)[:1]
    want = PR.oracle_kv(kv, 0, n)[:1]
    PR.check_kv(rep, got, want, "layer 0", n)
    rows = n - ((n - 1) // 16) * 16
    tg = eng.split_trace(rows)
    for l in range(m.n_layers):
        e = PR.rel_l2(tg["x"][l][:rows].double().cpu().numpy(), tr_o["x"][l][n - rows:]).max()
        assert e <= PR.tol_for(m), (l, e)
    print(rep)
    assert not rep.failures, rep
    eng.close()


def test_flint_continuous_batch_of_16_staggered(gpu_lib, flint4_int4):
    """Sixteen sequences whose prompt lengths and arrival steps are those of
    the 16-client workload's schedule (seed 4) divided by 4 and by 8, joining a
    running batch as they arrive; every step is ONE decode launch over the
    active rows, teacher-forced on the oracle's tokens and cache; each row is
    compared with the oracle's decode of its own sequence."""
    m, w = flint4_int4
    sched = SP.schedule(synth.CONFIGS[5])
    lens = [max(16, L // 4) for _, L in sched]
    arr = [a // 8 for a, _ in sched]
    n_steps = max(arr) + 3
    orc = Oracle(m, PR.host_fetch(m, w), cache_bytes=8 << 30)
    eng = Engine(m, w, n_pages=sum((L + n_steps + 127) // 128 for L in lens) + 8, max_ctx=4096, max_seqs=16)
    kvs, cur, pos = {}, {}, {}
    rep = PR.Report()
    tol = PR.tol_for(m)
    for step in range(n_steps):
        for s in range(16):
            if arr[s] == step:
                p = SP.prompt_tokens(m.seed, m.vocab, lens[s], seq=200 + s)
                kv = orc.new_kv()
                cur[s], _ = orc.prefill(kv, p)
                kvs[s], pos[s] = kv, lens[s]
                eng.kv_write(s, 0, PR.oracle_kv(kv, 0, lens[s]))
        act = sorted(kvs)
        if not act:
            continue
        toks = torch.tensor([cur[s] for s in act], dtype=torch.int32, device="cuda")
        out = torch.empty_like(toks)
        eng.enable_trace(len(act))
        eng.decode_step(act, toks, [pos[s] for s in act], out)
        eng.sync()
        tg = eng.split_trace(len(act))
        outs = out.cpu().tolist()
        for r, s in enumerate(act):
            nxt, tro = orc.decode(kvs[s], cur[s], pos[s])
            key = (s, step)      # every launch starts from the oracle's cache
            PR.compare_trace(rep, m, tg, tro, slice(r, r + 1), slice(0, 1), tol, f"step {step} seq {s}", seq=key)
            PR.check_token(rep, outs[r], nxt, float(tro["top2_margin"][-1]), f"step {step} seq {s}", seq=key)
            PR.check_kv(rep, eng.kv_read(s, pos[s], 1), PR.oracle_kv(kvs[s], pos[s], 1), f"step {step} seq {s}", 1)
            eng.kv_write(s, pos[s], PR.oracle_kv(kvs[s], pos[s], 1))
            cur[s] = nxt
            pos[s] += 1
    eng.disable_trace()
    _check(rep)
    eng.close()


def test_two_identical_runs_give_identical_bits(gpu_lib, flint4_int4):
    """Router logits are summed as fixed-point integers and the tensor-core
    partials in a fixed warp order: the same launches give the same trace,
    bit for bit, so every block (and every run) takes the same experts."""
    m, w = flint4_int4
    lens = [700, 300, 129]
    prompts = [torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, n, seq=s)).cuda() for s, n in enumerate(lens)]

    def run():
        eng = Engine(m, w, n_pages=24, max_ctx=2048, max_seqs=4)
        toks = torch.empty(3, dtype=torch.int32, device="cuda")
        for s, p in enumerate(prompts):
            eng.prefill(s, p, out=toks[s:s + 1])
        traces = []
        for rows in (3, 1):
            eng.enable_trace(rows)
            for i in range(2):
                ids = [0, 1, 2][:rows]
                eng.decode_step(ids, toks[:rows], [eng.seq_length(s) for s in ids], toks[:rows])
                eng.sync()
                traces.append(eng.trace.clone())
        eng.close()
        return traces, toks.cpu()

    a, ta = run()
    b, tb = run()
    assert torch.equal(ta, tb)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_flint_int4_long_context_batched_equals_solo(gpu_lib):
    """Full depth, context 2100 and 300: a batched launch (tensor-core GEMV for
    the dense projections, another attention split) gives each sequence what a
    solo launch gives, within the parity tolerance; tokens agree where the
    top-2 margin is clear."""
    m = synth.CONFIGS[3].model
    w = SW.model_torch(m, "cuda")
    lens = [2100, 300]
    prompts = [torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, n, seq=s)).cuda()
               for s, n in enumerate(lens)]
    steps = 3
    solo = []
    for p in prompts:
        eng = Engine(m, w, n_pages=64, max_ctx=4096, max_seqs=2)
        tok = eng.prefill(0, p)
        eng.enable_trace(1)
        toks, xs, margins, tks = [int(tok.item())], [], [np.inf], []
        for i in range(steps):
            eng.decode_step([0], tok, [p.numel() + i], tok)
            eng.sync()
            tr = eng.split_trace(1)
            toks.append(int(tok.item()))
            xs.append(tr["x"][:, 0].double().cpu().numpy())
            tks.append(tr["topk"][:, 0, :m.top_k].cpu().numpy())
            lg = np.sort(tr["logits"][0].double().cpu().numpy())
            margins.append(lg[-1] - lg[-2])
        solo.append((toks, xs, margins, tks))
        eng.close()
    eng = Engine(m, w, n_pages=64, max_ctx=4096, max_seqs=2)
    toks = torch.empty(2, dtype=torch.int32, device="cuda")
    for s, p in enumerate(prompts):
        eng.prefill(s, p, out=toks[s:s + 1])
    got = [[int(toks[s].item())] for s in range(2)]
    eng.enable_trace(2)
    worst = 0.0
    for i in range(steps):
        eng.decode_step([0, 1], toks, [lens[0] + i, lens[1] + i], toks)
        eng.sync()
        tr = eng.split_trace(2)
        for s in range(2):
            got[s].append(int(toks[s].item()))
            el = PR.rel_l2(tr["x"][:, s].double().cpu().numpy(), solo[s][1][i])
            e = el.max()
            worst = max(worst, e)
            kb = tr["topk"][:, s, :m.top_k].cpu().numpy()
            other = [l for l in range(m.n_layers) if set(kb[l]) != set(solo[s][3][i][l])]
            assert e < PR.tol_for(m), (s, i, e, int(el.argmax()), "layers with other experts", other[:5])
    print(f"batched vs solo: worst per-layer residual rel L2 {worst:.2e}")
    for s in range(2):
        for k, (a, b) in enumerate(zip(got[s], solo[s][0])):
            assert a == b or solo[s][2][k] <= PR.TOKEN_MARGIN, (s, k, a, b)
    eng.close()
    del w
    torch.cuda.empty_cache()


def test_split_launches_give_the_same_bits(gpu_lib, flint4_int4):
    """MK_DBG_SPLIT runs a decode step as one launch per phase group of a
    layer (QKV | attention | o_proj | routing + gate/up + down) plus one for
    lm_head, the kernel boundary in place of the grid barrier: the same device
    code on the same inputs, so the same trace and tokens, bit for bit, at one
    row and at three."""
    from moe_decode_megakernel_persistent_gb300 import _lib as L
    m, w = flint4_int4
    lens = [300, 129, 40]
    prompts = [torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, n, seq=10 + s)).cuda() for s, n in enumerate(lens)]

    def run(split):
        eng = Engine(m, w, n_pages=16, max_ctx=1024, max_seqs=4)
        toks = torch.empty(3, dtype=torch.int32, device="cuda")
        for s, p in enumerate(prompts):
            eng.prefill(s, p, out=toks[s:s + 1])
        traces = []
        for rows in (1, 3):
            nbytes = L.mk_trace_bytes(eng.desc, rows)
            tr = torch.zeros(nbytes // 4, dtype=torch.float32, device="cuda")
            L.mk_set_debug(eng.ctx, L.MK_DBG_TRACE | (L.MK_DBG_SPLIT if split else 0), 0, tr.data_ptr(), nbytes, 0)
            ids = [0, 1, 2][:rows]
            eng.decode_step(ids, toks[:rows], [eng.seq_length(s) for s in ids], toks[:rows])
            eng.sync()
            traces.append(tr)
        eng.close()
        return traces, toks.cpu()

    a, ta = run(False)
    b, tb = run(True)
    assert torch.equal(ta, tb)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
