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
