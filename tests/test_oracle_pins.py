"""Pins of the CPU oracle to facts other than itself: closed forms,
invariants, special cases and brute-force loops on tiny inputs."""
import cmath
import itertools
import math

import numpy as np
import pytest

from oracle import model as O
from oracle.numerics import dequant_int3, dequant_int4, round_bf16, bf16_bits_to_f64
from tests._models import Dims, dict_fetch, random_tensors


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    for c in (0.0, 1e-3, 1.0, -3.5, 40.0):
        x = np.full(16, c)
        w = np.linspace(0.5, 2.0, 16)
        eps = 1e-6
        y = O.rmsnorm(x, w, eps)
        np.testing.assert_allclose(y, w * c / math.sqrt(c * c + eps), rtol=1e-14, atol=0)


def test_rmsnorm_scale_invariant_and_unit_rms():
    rng = np.random.default_rng(1)
    x = rng.normal(size=33)
    w = np.ones(33)
    y = O.rmsnorm(x, w, 0.0)
    np.testing.assert_allclose(O.rmsnorm(7.25 * x, w, 0.0), y, rtol=1e-14)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    # one-hot: x = a e_0 over n elements -> y_0 = sqrt(n) sign(a)
    e = np.zeros(9)
    e[0] = -2.0
    assert abs(O.rmsnorm(e, np.ones(9), 0.0)[0] + 3.0) < 1e-14


# ------------------------------------------------------------------ RoPE

def test_rope_identity_at_position_zero():
    x = np.random.default_rng(2).normal(size=(3, 16))
    np.testing.assert_array_equal(O.rope(x, 0, 1e4), x)


def test_rope_matches_complex_rotation_of_half_pairs():
    d, theta = 8, 10000.0
    x = np.random.default_rng(3).normal(size=d)
    for pos in (1, 5, 4095):
        y = O.rope(x, pos, theta)
        for i in range(d // 2):
            ang = pos * theta ** (-(2.0 * i) / d)
            z = complex(x[i], x[i + d // 2]) * cmath.exp(1j * ang)
            assert abs(y[i] - z.real) < 1e-12 and abs(y[i + d // 2] - z.imag) < 1e-12


def test_rope_first_and_last_pair_angles():
    d, theta = 64, 1e6
    x = np.zeros(d)
    x[0] = 1.0
    x[d // 2 - 1] = 1.0
    y = O.rope(x, 3, theta)
    assert abs(y[0] - math.cos(3.0)) < 1e-14 and abs(y[d // 2] - math.sin(3.0)) < 1e-14
    a = 3 * theta ** (-(d - 2) / d)
    assert abs(y[d // 2 - 1] - math.cos(a)) < 1e-14 and abs(y[d - 1] - math.sin(a)) < 1e-14


def test_rope_keeps_pair_norms_and_is_relative():
    rng = np.random.default_rng(4)
    q, k = rng.normal(size=32), rng.normal(size=32)
    m, n = 17, 5
    rq = O.rope(q, m, 1e4)
    pn = lambda v: v[:16] ** 2 + v[16:] ** 2
    np.testing.assert_allclose(pn(rq), pn(q), rtol=1e-12)
    a = O.rope(q, m, 1e4) @ O.rope(k, n, 1e4)
    b = O.rope(q, m + 100, 1e4) @ O.rope(k, n + 100, 1e4)
    assert abs(a - b) < 1e-10


# ------------------------------------------------------------------ attention

def _attention_loops(q, K, V):
    nh, d = q.shape
    T, nkv, _ = K.shape
    grp = nh // nkv
    out = [[0.0] * d for _ in range(nh)]
    for h in range(nh):
        g = h // grp
        s = [sum(q[h][j] * K[t][g][j] for j in range(d)) / math.sqrt(d) for t in range(T)]
        mx = max(s)
        e = [math.exp(v - mx) for v in s]
        z = sum(e)
        for j in range(d):
            out[h][j] = sum(e[t] / z * V[t][g][j] for t in range(T))
    return np.array(out)


def test_attention_matches_brute_force_loops():
    rng = np.random.default_rng(5)
    q = rng.normal(size=(4, 6))
    K = rng.normal(size=(7, 2, 6))
    V = rng.normal(size=(7, 2, 6))
    np.testing.assert_allclose(O.attention(q, K, V), _attention_loops(q, K, V), rtol=1e-12, atol=1e-14)


def test_attention_single_position_returns_value_row():
    rng = np.random.default_rng(6)
    q = rng.normal(size=(4, 8))
    K = rng.normal(size=(1, 2, 8))
    V = rng.normal(size=(1, 2, 8))
    out = O.attention(q, K, V)
    for h in range(4):
        np.testing.assert_array_equal(out[h], V[0, h // 2])


def test_attention_equal_keys_give_mean_and_groups_are_contiguous():
    rng = np.random.default_rng(7)
    q = rng.normal(size=(4, 8))
    K = np.repeat(rng.normal(size=(1, 2, 8)), 5, axis=0)
    V = rng.normal(size=(5, 2, 8))
    out = O.attention(q, K, V)
    # heads 0,1 read kv head 0; heads 2,3 read kv head 1
    for h in range(4):
        np.testing.assert_allclose(out[h], V[:, h // 2].mean(axis=0), rtol=1e-12)


def test_causal_attention_equals_per_position_attention():
    rng = np.random.default_rng(8)
    Q = rng.normal(size=(5, 4, 6))
    K = rng.normal(size=(9, 2, 6))
    V = rng.normal(size=(9, 2, 6))
    start = 4
    full = O.causal_attention(Q, K, V, start)
    for i in range(5):
        T = start + i + 1
        np.testing.assert_allclose(full[i], _attention_loops(Q[i], K[:T], V[:T]), rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------------ router / MoE

def test_router_topk_matches_enumeration_with_tie_rule():
    logits = np.array([0.5, 2.0, 2.0, -1.0, 2.0, 0.7])
    ids, w, p = O.router_topk(logits, 2)
    assert list(ids) == [1, 2]                        # three-way tie -> lowest ids
    rng = np.random.default_rng(9)
    for _ in range(20):
        lg = rng.normal(size=6)
        k = 3
        best = max(itertools.combinations(range(6), k), key=lambda S: sum(lg[list(S)]))
        ids, w, p = O.router_topk(lg, k)
        assert sorted(ids) == sorted(best)
        ex = [math.exp(lg[i]) for i in ids]
        np.testing.assert_allclose(w, np.array(ex) / sum(ex), rtol=1e-12)
        assert abs(p.sum() - 1.0) < 1e-14


def _moe_dims(top_k):
    return Dims(n_layers=2, n_dense=1, top_k=top_k)


def test_moe_with_all_experts_is_the_dense_softmax_mixture():
    d = _moe_dims(top_k=5)
    t = random_tensors(d, seed=10)
    orc = O.Oracle(d, dict_fetch(t))
    rng = np.random.default_rng(11)
    h = rng.normal(size=(3, d.hidden))
    tr = {"router_logits": [], "topk_ids": [], "topk_w": [], "topk_margin": []}
    out = orc._ffn_block(1, h, tr)
    z = O.rmsnorm(h, t[("ffn_norm", 1, None)], d.rms_eps)
    lg = z @ t[("router", 1, None)].T
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ref = h.copy()
    for e in range(d.n_experts):
        ye = O.swiglu(z, t[("exp_gate", 1, e)], t[("exp_up", 1, e)], t[("exp_down", 1, e)])
        ref += p[:, e:e + 1] * ye
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_single_expert_top1_is_a_dense_swiglu():
    d = Dims(n_layers=2, n_dense=1, n_experts=1, top_k=1)
    t = random_tensors(d, seed=12)
    orc = O.Oracle(d, dict_fetch(t))
    h = np.random.default_rng(13).normal(size=(2, d.hidden))
    tr = {"router_logits": [], "topk_ids": [], "topk_w": [], "topk_margin": []}
    out = orc._ffn_block(1, h, tr)
    z = O.rmsnorm(h, t[("ffn_norm", 1, None)], d.rms_eps)
    g = z @ t[("exp_gate", 1, 0)].T
    u = z @ t[("exp_up", 1, 0)].T
    ref = h + ((g / (1 + np.exp(-g))) * u) @ t[("exp_down", 1, 0)].T
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert tr["topk_w"][0][0, 0] == 1.0


# ------------------------------------------------------------------ whole step

def _brute_step(t, d, tokens):
    """Position-by-position decode with scalar loops and lists: an independent
    restatement of the layer composition on tiny inputs."""
    H = d.hidden
    hd = d.head_dim
    cache_k = [[] for _ in range(d.n_layers)]
    cache_v = [[] for _ in range(d.n_layers)]
    res = []

    def mv(W, v):
        return [sum(W[r][c] * v[c] for c in range(len(v))) for r in range(len(W))]

    def norm(v, w):
        r = 1.0 / math.sqrt(sum(a * a for a in v) / len(v) + d.rms_eps)
        return [v[i] * r * w[i] for i in range(len(v))]

    def rot(v, pos):
        half = hd // 2
        out = list(v)
        for i in range(half):
            a = pos * d.rope_theta ** (-2.0 * i / hd)
            out[i] = v[i] * math.cos(a) - v[i + half] * math.sin(a)
            out[i + half] = v[i + half] * math.cos(a) + v[i] * math.sin(a)
        return out

    def ffn(z, g, u, dn):
        a = [(x / (1 + math.exp(-x))) * y for x, y in zip(mv(g, z), mv(u, z))]
        return mv(dn, a)

    for pos, tok in enumerate(tokens):
        x = list(t[("embed", -1, None)][tok])
        xs = []
        for l in range(d.n_layers):
            y = norm(x, t[("attn_norm", l, None)])
            q = mv(t[("wq", l, None)], y)
            k = mv(t[("wk", l, None)], y)
            v = mv(t[("wv", l, None)], y)
            qh = [rot(q[h * hd:(h + 1) * hd], pos) for h in range(d.n_heads)]
            kh = [rot(k[g * hd:(g + 1) * hd], pos) for g in range(d.n_kv_heads)]
            vh = [v[g * hd:(g + 1) * hd] for g in range(d.n_kv_heads)]
            cache_k[l].append([list(round_bf16(np.array(a))) for a in kh])
            cache_v[l].append([list(round_bf16(np.array(a))) for a in vh])
            att = []
            for h in range(d.n_heads):
                g = h * d.n_kv_heads // d.n_heads
                s = [sum(qh[h][j] * kk[g][j] for j in range(hd)) / math.sqrt(hd) for kk in cache_k[l]]
                mx = max(s)
                e = [math.exp(a - mx) for a in s]
                att += [sum(e[i] * cache_v[l][i][g][j] for i in range(len(e))) / sum(e) for j in range(hd)]
            o = mv(t[("wo", l, None)], att)
            hres = [x[i] + o[i] for i in range(H)]
            z = norm(hres, t[("ffn_norm", l, None)])
            if l < d.n_dense:
                f = ffn(z, t[("gate", l, None)], t[("up", l, None)], t[("down", l, None)])
            else:
                lg = mv(t[("router", l, None)], z)
                order = sorted(range(d.n_experts), key=lambda e: (-lg[e], e))[:d.top_k]
                ws = [math.exp(lg[e]) for e in order]
                f = [0.0] * H
                for e, wgt in zip(order, ws):
                    ye = ffn(z, t[("exp_gate", l, e)], t[("exp_up", l, e)], t[("exp_down", l, e)])
                    f = [f[i] + wgt / sum(ws) * ye[i] for i in range(H)]
            x = [hres[i] + f[i] for i in range(H)]
            xs.append(x)
        xf = norm(x, t[("final_norm", -1, None)])
        logits = mv(t[("lm_head", -1, None)], xf)
        res.append((xs, logits))
    return res


def test_decode_step_matches_scalar_brute_force():
    d = Dims()
    t = random_tensors(d, seed=14)
    orc = O.Oracle(d, dict_fetch(t))
    tokens = [3, 17, 0, 36, 9]
    brute = _brute_step(t, d, tokens)
    kv = orc.new_kv()
    for pos, tok in enumerate(tokens):
        nxt, tr = orc.decode(kv, tok, pos)
        xs, logits = brute[pos]
        for l in range(d.n_layers):
            np.testing.assert_allclose(tr["x"][l][0], xs[l], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(tr["logits"][0], logits, rtol=1e-9, atol=1e-11)
        assert nxt == int(np.argmax(logits))


def test_incremental_decode_equals_full_causal_recompute():
    d = Dims(n_layers=3, n_dense=1)
    t = random_tensors(d, seed=15)
    orc = O.Oracle(d, dict_fetch(t))
    toks = [1, 5, 9, 2, 33, 30, 7, 7, 0]
    kv_full = orc.new_kv()
    tok_full, tr_full = orc.prefill(kv_full, toks)
    kv_inc = orc.new_kv()
    orc.prefill(kv_inc, toks[:3])
    tr = None
    for i in range(3, len(toks)):
        tok_inc, tr = orc.decode(kv_inc, toks[i], i)
    for l in range(d.n_layers):
        np.testing.assert_allclose(tr["x"][l][0], tr_full["x"][l][-1], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(tr["logits"][0], tr_full["logits"][0], rtol=1e-11, atol=1e-12)
    assert tok_inc == tok_full


def test_residual_passthrough_when_blocks_are_zero():
    d = Dims()
    t = random_tensors(d, seed=16)
    for k in list(t):
        if k[0] in ("wo", "down", "exp_down"):
            t[k] = np.zeros_like(t[k])
    orc = O.Oracle(d, dict_fetch(t))
    tok, tr = orc.decode(orc.new_kv(), 11, 0)
    for l in range(d.n_layers):
        np.testing.assert_array_equal(tr["x"][l][0], t[("embed", -1, None)][11])
    ref = O.rmsnorm(t[("embed", -1, None)][11], t[("final_norm", -1, None)], d.rms_eps) @ t[("lm_head", -1, None)].T
    np.testing.assert_allclose(tr["logits"][0], ref, rtol=1e-13)


def test_paged_kv_is_bit_identical_to_contiguous_under_page_permutation():
    d = Dims(n_layers=2, n_dense=1)
    t = random_tensors(d, seed=17)
    orc = O.Oracle(d, dict_fetch(t))
    toks = list(np.random.default_rng(18).integers(0, d.vocab, 300))
    kv_c = orc.new_kv()
    order = list(np.random.default_rng(19).permutation(8))
    kv_p = orc.new_kv(paged=True, n_pages=8, page_order=order)
    _, a = orc.prefill(kv_c, toks[:260])
    _, b = orc.prefill(kv_p, toks[:260])
    assert kv_p.table[:3] == order[:3]
    for pos in range(260, 300):
        _, a = orc.decode(kv_c, toks[pos], pos)
        _, b = orc.decode(kv_p, toks[pos], pos)
        np.testing.assert_array_equal(a["x"][-1], b["x"][-1])
        np.testing.assert_array_equal(a["logits"], b["logits"])


# ------------------------------------------------------------------ formats

def test_round_bf16_ties_and_ranges():
    assert round_bf16(1.0 + 2 ** -8) == 1.0                   # tie -> even
    assert round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6      # tie -> even (up)
    assert round_bf16(1.0 + 2 ** -8 + 2 ** -30) == 1.0 + 2 ** -7
    assert round_bf16(-2.5) == -2.5
    x = np.random.default_rng(20).normal(size=1000) * 100
    r = round_bf16(x)
    assert np.all(np.abs(r - x) <= np.abs(x) * 2 ** -8)   # unit roundoff of 8 bits


def test_int4_dequant_of_hand_packed_grid_values():
    q = np.tile(np.arange(-8, 8), 8).reshape(1, 128)              # every code
    u = (q & 0xF).astype(np.uint8)
    packed = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    s_bits = np.array([[0x3F80, 0x4040]], dtype=np.uint16)        # 1.0, 3.0
    w = dequant_int4(packed, s_bits)
    np.testing.assert_array_equal(w[0, :64], q[0, :64].astype(float))
    np.testing.assert_array_equal(w[0, 64:], 3.0 * q[0, 64:])
    assert bf16_bits_to_f64(np.uint16(0xC0A0)) == -5.0


def test_int4_quantiser_error_bound_and_exact_grid():
    from synth import weights as SW
    from synth.configs import FLINT_BF16
    raw = SW.raw_np(FLINT_BF16, "wq", 3, rows=(0, 64))
    packed, s_bits = SW.quantize_int4_np(raw)
    w = bf16_bits_to_f64(raw)
    deq = dequant_int4(packed, s_bits)
    s = np.repeat(bf16_bits_to_f64(s_bits), 64, axis=1)
    assert np.all(np.abs(deq - w) <= s / 2 + 1e-12)
    # grid values with power-of-two scales are exact in bf16 and come back exactly
    rng = np.random.default_rng(21)
    q = rng.integers(-7, 8, size=(4, 128))
    q[:, 0] = 7
    q[:, 64] = -7                                    # every group reaches |q| = 7
    e = np.array([[-7, -3], [0, 2], [-12, -9], [1, -1]])
    wgrid = q * np.repeat(2.0 ** e, 64, axis=1)
    gbits = (np.asarray(wgrid, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bf16_bits_to_f64(gbits), wgrid)
    p2, s2 = SW.quantize_int4_np(gbits)
    np.testing.assert_array_equal(dequant_int4(p2, s2), wgrid)
    np.testing.assert_array_equal(bf16_bits_to_f64(s2), 2.0 ** e)


def test_int3_dequant_of_hand_packed_words():
    # 0o76543210 holds the codes 0..7 in order (code j at bits 3j): as bytes,
    # little-endian, 0x88 0xC6 0xFA; read as two's complement, 0 1 2 3 -4 -3 -2 -1.
    # 0o01234567 = 0x053977 holds them reversed; 0o77777777 is eight -1 codes.
    up = [0x88, 0xC6, 0xFA]
    down = [0x77, 0x39, 0x05]
    ones = [0xFF, 0xFF, 0xFF]
    packed = np.array([up * 4 + down * 4 + ones * 8], dtype=np.uint8)   # K = 128
    assert packed.shape == (1, 48)
    s_bits = np.array([[0x3F80, 0x4040]], dtype=np.uint16)               # 1.0, 3.0
    w = dequant_int3(packed, s_bits)
    inc = [0, 1, 2, 3, -4, -3, -2, -1]
    np.testing.assert_array_equal(w[0, :32], np.tile(inc, 4))
    np.testing.assert_array_equal(w[0, 32:64], np.tile(inc[::-1], 4))
    np.testing.assert_array_equal(w[0, 64:], np.full(64, -3.0))


def test_int3_quantiser_error_bound_and_exact_grid():
    from synth import weights as SW
    from synth.configs import FLINT_INT4_E3
    assert SW.storage_dtype(FLINT_INT4_E3, "exp_down") == "int3"
    assert SW.storage_dtype(FLINT_INT4_E3, "down") == "int4"
    raw = SW.raw_np(FLINT_INT4_E3, "exp_gate", 3, expert=5, rows=(0, 64))
    packed, s_bits = SW.quantize_int3_np(raw)
    assert packed.shape == (64, 3 * 2048 // 8) and s_bits.shape == (64, 32)
    w = bf16_bits_to_f64(raw)
    deq = dequant_int3(packed, s_bits)
    s = np.repeat(bf16_bits_to_f64(s_bits), 64, axis=1)
    assert np.all(np.abs(deq - w) <= s / 2 + 1e-12)
    # every code is within the symmetric range the quantiser produces
    assert np.all(np.abs(deq) <= 3 * s + 1e-12)
    # grid values with power-of-two scales are exact in bf16 and come back exactly
    rng = np.random.default_rng(22)
    q = rng.integers(-3, 4, size=(4, 128))
    q[:, 0] = 3
    q[:, 64] = -3                                    # every group reaches |q| = 3
    e = np.array([[-7, -3], [0, 2], [-12, -9], [1, -1]])
    wgrid = q * np.repeat(2.0 ** e, 64, axis=1)
    gbits = (np.asarray(wgrid, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    p2, s2 = SW.quantize_int3_np(gbits)
    np.testing.assert_array_equal(dequant_int3(p2, s2), wgrid)
    np.testing.assert_array_equal(bf16_bits_to_f64(s2), 2.0 ** e)


def test_argmax_ties_to_lowest_index():
    assert O.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert O.top2_margin(np.array([1.0, 3.0, 2.5])) == 0.5
    assert O.topk_margin(np.array([4.0, 1.0, 3.0, 2.0]), 2) == 1.0
    assert O.topk_margin(np.array([1.0, 2.0]), 2) == math.inf
