"""Plant plausible mistakes in the oracle (on the CPU) and check that its pins
notice: the pins must not pass for a wrong oracle."""
import numpy as np
import pytest

from oracle import model as O
from tests import test_oracle_pins as pins


def _rope_wrong_sign(x, pos, theta):
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta ** (-2.0 * i / d)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * np.cos(ang) + b * np.sin(ang), b * np.cos(ang) - a * np.sin(ang)], -1)


def _rope_interleaved(x, pos, theta):
    d = x.shape[-1]
    i = np.arange(d // 2, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta ** (-2.0 * i / d)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * np.cos(ang) - b * np.sin(ang)
    out[..., 1::2] = b * np.cos(ang) + a * np.sin(ang)
    return out


def _attention_wrong_group(q, K, V):
    nh, d = q.shape
    nkv = K.shape[1]
    out = np.empty((nh, d))
    for h in range(nh):
        g = h % nkv                                   # strided instead of contiguous
        s = K[:, g, :] @ q[h] / np.sqrt(d)
        p = np.exp(s - s.max())
        out[h] = (p / p.sum()) @ V[:, g, :]
    return out


def _attention_no_scale(q, K, V):
    nh, d = q.shape
    grp = nh // K.shape[1]
    out = np.empty((nh, d))
    for h in range(nh):
        s = K[:, h // grp, :] @ q[h]
        p = np.exp(s - s.max())
        out[h] = (p / p.sum()) @ V[:, h // grp, :]
    return out


def _rmsnorm_no_eps_mean(x, w, eps):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * w


def _topk_no_renorm(logits, k):
    z = logits - logits.max()
    p = np.exp(z) / np.exp(z).sum()
    ids = np.argsort(-p, kind="stable")[:k]
    return ids, p[ids], p


def _silu_wrong(x):
    return x / (1.0 + np.exp(x))


MUTANTS = [
    ("rope", _rope_wrong_sign),
    ("rope", _rope_interleaved),
    ("attention", _attention_wrong_group),
    ("attention", _attention_no_scale),
    ("rmsnorm", _rmsnorm_no_eps_mean),
    ("router_topk", _topk_no_renorm),
    ("silu", _silu_wrong),
]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[f"{n}:{f.__name__}" for n, f in MUTANTS])
def test_whole_step_pin_catches_mutant(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)
    with pytest.raises(AssertionError):
        pins.test_decode_step_matches_scalar_brute_force()


def test_dropped_residual_is_caught(monkeypatch):
    orig = O.Oracle._ffn_block

    def no_residual(self, l, h, tr):
        return orig(self, l, h, tr) - h
    monkeypatch.setattr(O.Oracle, "_ffn_block", no_residual)
    with pytest.raises(AssertionError):
        pins.test_decode_step_matches_scalar_brute_force()


def test_transposed_operand_is_caught(monkeypatch):
    orig = O.Oracle.w

    def transposed(self, name, layer=-1, expert=None):
        a = orig(self, name, layer, expert)
        return a.T if name in ("wo",) else a
    monkeypatch.setattr(O.Oracle, "w", transposed)
    with pytest.raises((AssertionError, ValueError)):
        pins.test_decode_step_matches_scalar_brute_force()


# ---- the int3 storage format: plausible misreadings of the packed words

def _int3_decode(packed, scale_bits, order=lambda j: j, signed=True, little=True, group=64):
    from oracle.numerics import bf16_bits_to_f64
    packed = np.asarray(packed, dtype=np.uint8)
    R, nb = packed.shape
    K = nb // 3 * 8
    b = packed.reshape(R, K // 8, 3).astype(np.int64)
    word = (b[:, :, 0] + 256 * b[:, :, 1] + 65536 * b[:, :, 2]) if little else \
           (b[:, :, 2] + 256 * b[:, :, 1] + 65536 * b[:, :, 0])
    q = np.empty((R, K // 8, 8), dtype=np.int64)
    for j in range(8):
        q[:, :, j] = (word // (8 ** order(j))) % 8
    q = q.reshape(R, K)
    if signed:
        q = np.where(q >= 4, q - 8, q)
    s = np.repeat(bf16_bits_to_f64(scale_bits), 64, axis=1)[:, :K]
    if group != 64:
        s = np.repeat(bf16_bits_to_f64(scale_bits), group, axis=1)[:, :K]
    return q.astype(np.float64) * s


INT3_MUTANTS = [
    ("reversed code order", lambda p, s: _int3_decode(p, s, order=lambda j: 7 - j)),
    ("unsigned codes", lambda p, s: _int3_decode(p, s, signed=False)),
    ("big-endian words", lambda p, s: _int3_decode(p, s, little=False)),
    ("one scale per 128 values", lambda p, s: _int3_decode(p, s, group=128)),
]


@pytest.mark.parametrize("label,fn", INT3_MUTANTS, ids=[m[0] for m in INT3_MUTANTS])
def test_int3_pins_catch_misread_words(monkeypatch, label, fn):
    # the correct decoder passes both pins ...
    pins.test_int3_dequant_of_hand_packed_words()
    pins.test_int3_quantiser_error_bound_and_exact_grid()
    # ... a misreading fails at least one
    monkeypatch.setattr(pins, "dequant_int3", fn)
    failed = 0
    for pin in (pins.test_int3_dequant_of_hand_packed_words, pins.test_int3_quantiser_error_bound_and_exact_grid):
        try:
            pin()
        except (AssertionError, ValueError):
            failed += 1
    assert failed >= 1, label
