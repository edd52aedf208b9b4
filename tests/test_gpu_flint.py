"""The Flint-shaped model at full size (49 layers, hidden 2048, 64 experts
top-6, vocabulary 151936), in the launch configuration the bench times
(one block per SM, batch 1).

Oracle parity runs on a short prompt so that the float64 oracle finishes in
about a minute; long contexts are covered at this size by properties that
hold at any length (a sequence gives the same result batched or alone, within
the parity tolerance, since batched launches take the tensor-core GEMV), and
against the oracle on the tiny model (test_gpu_parity.py)."""
import numpy as np
import pytest
import torch

import synth
from synth import prompts as SP
from synth import weights as SW
from moe_decode_megakernel_persistent_gb300.engine import Engine
from tests import _parity as PR

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [3, 2])
def test_flint_prefill_and_decode_match_the_oracle(gpu_lib, cfg):
    m = synth.CONFIGS[cfg].model
    w = SW.model_torch(m, "cuda")
    rep = PR.run_single(m, prompt_len=2, n_decode=2, w=w, n_pages=8)
    print(rep)
    assert not rep.failures, rep
    assert rep.topk_checked > 0
    del w
    torch.cuda.empty_cache()


def test_flint_int4_long_context_batched_equals_solo(gpu_lib):
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
        toks, xs, margins = [int(tok.item())], [], [np.inf]
        for i in range(steps):
            eng.decode_step([0], tok, [p.numel() + i], tok)
            eng.sync()
            tr = eng.split_trace(1)
            toks.append(int(tok.item()))
            xs.append(tr["x"][:, 0].double().cpu().numpy())
            lg = np.sort(tr["logits"][0].double().cpu().numpy())
            margins.append(lg[-1] - lg[-2])
        solo.append((toks, xs, margins))
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
            e = PR.rel_l2(tr["x"][:, s].double().cpu().numpy(), solo[s][1][i]).max()
            worst = max(worst, e)
            assert e < PR.tol_for(m), (s, i, e)
    print(f"batched vs solo: worst per-layer residual rel L2 {worst:.2e}")
    for s in range(2):
        for k, (a, b) in enumerate(zip(got[s], solo[s][0])):
            # a batched launch takes the tensor-core GEMV for the dense
            # projections and another attention split, a solo launch the dp4a
            # GEMV: rounding differs (and drifts through bf16 K/V rounding
            # flips), so tokens must agree where the top-2 margin is clear
            assert a == b or solo[s][2][k] <= PR.TOKEN_MARGIN, (s, k, a, b)
    eng.close()
