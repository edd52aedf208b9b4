"""Writes tiny_decode.json beside this script: the float64 oracle's greedy
decode of the tiny configuration (2 layers, hidden 256, 4 q / 2 kv heads of
64, layer 0 dense, layer 1 eight experts top-2, vocabulary 1024; fp32 weights
of seed 0; 64 prompt tokens, 16 generated tokens): per generated token its id,
the top-2 logit margin and the L2 norm of the last layer's residual.

Only the oracle and the seeded input generators are called.  The file pins
the oracle against unintended change: a change of the oracle's arithmetic
regenerates it, and the commit names the passage that justifies it.

    python tests/golden/make_oracle_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import prompts as SP  # noqa: E402
from synth import weights as SW  # noqa: E402
from oracle import Oracle  # noqa: E402

PROMPT, GENERATED = 64, 16


def fetch_for(m):
    cache = {}

    def fetch(name, layer, expert):
        key = (name, layer, expert)
        if key not in cache:
            if name in ("embed", "attn_norm", "ffn_norm", "final_norm", "router"):
                cache[key] = (SW.raw_np(m, name, layer, expert), m.aux_dtype)
            else:
                cache[key] = (SW.linear_np(m, name, layer, expert), m.wdtype)
        return cache[key]
    return fetch


def tiny_decode():
    m = synth.CONFIGS[1].model
    orc = Oracle(m, fetch_for(m))
    kv = orc.new_kv()
    tok, tr = orc.prefill(kv, SP.prompt_tokens(m.seed, m.vocab, PROMPT))
    out = {"tokens": [int(tok)], "top2_margin": [float(tr["top2_margin"][-1])],
           "last_residual_norm": [float(np.linalg.norm(tr["x"][-1][-1]))]}
    for i in range(GENERATED - 1):
        tok, tr = orc.decode(kv, tok, PROMPT + i)
        out["tokens"].append(int(tok))
        out["top2_margin"].append(float(tr["top2_margin"][-1]))
        out["last_residual_norm"].append(float(np.linalg.norm(tr["x"][-1][-1])))
    return out


if __name__ == "__main__":
    res = tiny_decode()
    res["what"] = ("float64 oracle, tiny configuration (seed 0, fp32 weights), 64 prompt tokens, "
                   "16 greedy tokens: id, top-2 logit margin, last-layer residual L2 norm")
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode.json"), "w") as fh:
        json.dump(res, fh, indent=1)
    print(res["tokens"])
