"""The seeded input generator: determinism, backend bit-identity, formats."""
import numpy as np
import pytest
import torch

import synth
from synth import prompts as P
from synth import weights as SW
from synth.hashing import hash_int, hash_np, hash_torch, stream_key


def test_hash_backends_agree():
    key = stream_key(7, 123)
    idx = np.arange(0, 5000, 7, dtype=np.uint64)
    a = hash_np(key, idx)
    b = hash_torch(key, torch.from_numpy(idx.astype(np.int64))).numpy()
    assert np.array_equal(a.astype(np.int64), b)
    assert all(int(a[i]) == hash_int(key, int(idx[i])) for i in range(0, len(idx), 97))
    assert a.max() < 2 ** 32


def test_normal_table_is_a_symmetric_n002_quantile_table():
    t = SW.normal_table("f32")
    assert t.shape == (65536,)
    assert np.all(np.diff(t) >= 0)
    np.testing.assert_array_equal(t, -t[::-1])
    assert abs(t.std() - 0.02) < 2e-4
    tb = SW.bf16_bits_to_f32(SW.normal_table("bf16"))
    assert np.all(np.abs(tb - t) <= np.abs(t) * 2 ** -8)


@pytest.mark.parametrize("cfg", [1, 3])
def test_weights_numpy_equals_torch_and_are_deterministic(cfg):
    m = synth.CONFIGS[cfg].model
    name, kw = ("wk", {}) if cfg == 1 else ("exp_up", {"expert": 5})
    a = SW.raw_np(m, name, 1, **kw)
    b = SW.raw_np(m, name, 1, **kw)
    assert np.array_equal(a, b)
    t = SW.raw_torch(m, name, 1, kw.get("expert"))
    if m.aux_dtype == "f32":
        assert np.array_equal(a, t.numpy())
    else:
        assert np.array_equal(a.astype(np.int16), t.view(torch.int16).numpy())
        pa, sa = SW.quantize_int4_np(a)
        pt, st = SW.quantize_int4_torch(t)
        assert np.array_equal(pa, pt.numpy())
        assert np.array_equal(sa.astype(np.int16), st.view(torch.int16).numpy())
        pa, sa = SW.quantize_int3_np(a)
        pt, st = SW.quantize_int3_torch(t)
        assert np.array_equal(pa, pt.numpy())
        assert np.array_equal(sa.astype(np.int16), st.view(torch.int16).numpy())


def test_row_ranges_and_experts_are_consistent_slices():
    m = synth.CONFIGS[2].model
    full = SW.raw_np(m, "wo", 4)
    np.testing.assert_array_equal(SW.raw_np(m, "wo", 4, rows=(100, 164)), full[100:164])
    e3 = SW.raw_np(m, "exp_down", 9, expert=3, rows=(10, 12))
    assert e3.shape == (2, m.expert_ffn)
    assert not np.array_equal(SW.raw_np(m, "wo", 4), SW.raw_np(m, "wo", 5))


def test_int4_configs_share_the_bf16_source_weights():
    a = SW.raw_np(synth.CONFIGS[2].model, "wq", 0, rows=(0, 4))
    b = SW.raw_np(synth.CONFIGS[3].model, "wq", 0, rows=(0, 4))
    assert np.array_equal(a, b)
    # the int3-expert model: the same source weights, experts in int3 only
    e3 = synth.FLINT_INT4_E3
    for name, kw in (("wq", {}), ("exp_gate", {"expert": 7}), ("down", {})):
        layer = 0 if name == "down" else 4
        x = SW.raw_np(synth.CONFIGS[3].model, name, layer, rows=(0, 4), **kw)
        y = SW.raw_np(e3, name, layer, rows=(0, 4), **kw)
        assert np.array_equal(x, y)
    assert isinstance(SW.linear_np(e3, "exp_down", 4, expert=1), tuple)
    assert SW.linear_np(e3, "exp_down", 4, expert=1)[0].shape == (2048, 288)
    assert SW.linear_np(e3, "wo", 4)[0].shape == (2048, 1024)


def test_prompts_and_schedule():
    t = P.prompt_tokens(1, 151936, 4096)
    assert t.dtype == np.int32 and t.min() >= 0 and t.max() < 151936
    assert np.array_equal(t[:100], P.prompt_tokens(1, 151936, 100))
    sch = P.schedule(synth.CONFIGS[5])
    assert len(sch) == 16
    assert all(0 <= a <= 64 and 256 <= L <= 8192 for a, L in sch)
    assert P.schedule(synth.CONFIGS[3]) == [(0, 2048)]
