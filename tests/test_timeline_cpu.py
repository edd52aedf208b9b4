"""The per-phase timeline arithmetic (host side, no GPU): `Engine.phase_times_us`
over a hand-made timing record of two blocks and two layers, the layout
include/mk.h documents for MK_DBG_TIMING ([0] block start; [1 + 16 l + 3 p + k]
with k = 0 staging done, 1 work done, 2 barrier released; [1 + 16 L] lm_head
done).  Every figure the bench's `timeline_us` reports is checked by hand."""
import types

import numpy as np

from moe_decode_megakernel_persistent_gb300.engine import Engine

US = 1000  # stamps are in ns


def _record():
    L = 2
    t = np.zeros((2, 16 * L + 2), dtype=np.int64)
    t[:, 0] = [0, 1 * US]
    clock = [0, 1 * US]
    for l in range(L):
        for p in range(5):
            base = 1 + 16 * l + 3 * p
            for b in range(2):
                stage = clock[b] + (1 + p) * US          # staging takes 1 + p us
                done = stage + (2 + b) * US              # block 1 works 1 us longer
                t[b, base], t[b, base + 1] = stage, done
            release = max(t[:, base + 1]) + 3 * US      # 3 us after the last arrival
            t[:, base + 2] = [release, release + 1 * US]  # block 1 sees it 1 us later
            clock = list(t[:, base + 2])
    t[:, 1 + 16 * L] = [clock[0] + 50 * US, clock[1] + 60 * US]
    return t, L


def test_phase_times_follow_the_documented_definitions():
    t, L = _record()
    shape = types.SimpleNamespace(n_layers=L, n_dense=0)
    fake = types.SimpleNamespace(shape=shape, timing_stamps=lambda: t, PHASES=Engine.PHASES)
    out = Engine.phase_times_us(fake)
    for p, k in enumerate(Engine.PHASES):
        ph = out[k]
        assert ph["stage"] == 1 + p                 # block 0's staging, from its own previous release
        # work, from each block's previous release: block 0 (1 + p) + 2, block 1 (1 + p) + 3
        assert ph["work_med"] == (1 + p) + 2.5
        # the last arrival, from the latest previous release
        assert ph["work_max"] == (1 + p) + 3
        assert ph["barrier"] == 3                   # last arrival to the first release
        assert ph["span"] == (1 + p) + 3 + 3 + 1    # latest previous release to the latest release
    assert out["layer_median"] == sum(out[k]["span"] for k in Engine.PHASES)
    assert out["lm_head"] == 60 + 0                 # the last lm_head stamp after the latest release
    assert out["total"] == (t[:, 1 + 16 * L].max() - t[:, 0].min()) / US
