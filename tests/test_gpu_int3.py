"""Int3 experts (the lower-bit expert format of "rec Megakernel and Tempo9
Compared", §5 Method, where rec runs the Flint model with INT3 experts):
the expert matrices in symmetric int3 (group 64), every other linear layer
in int4, against the oracle on the same codes.

- The library's recoding of int3 rows into its bit planes, bit for bit.
- The tiny model in a 16-row launch, each row against the oracle (the expert
  GEMV with several activations per tile).
- The Flint shape, layers 0-3: a 2048-token context with teacher-forced
  decode in the launch configuration the bench times, a free-running
  64-token prompt through the chunked prefill's GEMMs (int3 widened to fp16)
  followed by decode, and four sequences in one launch.

Integer rules as everywhere: top-k ids where the oracle's margin exceeds
1e-3, tokens where its top-2 margin exceeds 0.05, exact.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import Oracle
from synth import prompts as SP
from synth import weights as SW
from moe_decode_megakernel_persistent_gb300 import _lib as L
from moe_decode_megakernel_persistent_gb300.engine import Engine, make_desc
from tests import _parity as PR
from tests._models import weights_struct

pytestmark = pytest.mark.gpu

TINY_E3 = synth.CONFIGS[1].model.with_(wdtype="int4", expert_dtype="int3")
MIN_TOPK = 40


def _check(rep, min_topk=MIN_TOPK):
    print(rep)
    assert not rep.failures, rep
    assert rep.topk_checked >= min_topk, rep
    assert rep.tokens_checked >= 1, rep


def _a256(x):
    return (x + 255) // 256 * 256


def _rec(fmt, K):
    row = {"int4": K // 2, "int3": 3 * K // 8}[fmt]
    return (row + K // 32 + 15) // 16 * 16


def _expert_sections(m):
    """Byte offsets of each layer's expert gate/up and down records in the
    packed weights, from the record rule of the packed layout (per layer the
    QKV, o_proj, gate/up and down sections, each 256-byte aligned)."""
    H, QD, KD = m.hidden, m.q_dim, m.kv_dim
    off, out = 0, {}
    for l in range(m.n_layers):
        dense = l < m.n_dense
        f = m.wdtype if dense else m.xdtype
        off = _a256(off + (QD + 2 * KD) * _rec(m.wdtype, H))
        off = _a256(off + H * _rec(m.wdtype, QD))
        gu = off
        ffn = m.dense_ffn if dense else m.n_experts * m.expert_ffn
        off = _a256(off + 2 * ffn * _rec(f, H))
        dn = off
        off = _a256(off + (H if dense else m.n_experts * H) * _rec(f, m.dense_ffn if dense else m.expert_ffn))
        out[l] = (gu, dn)
    return out, _a256(off + m.vocab * _rec(m.wdtype, H))


def _decode_planes(rec: np.ndarray, K: int):
    """The int3 codes q (in [-4, 3]) and scale bits of one packed record."""
    nch = K // 32
    lw = rec[:8 * nch].view(np.uint32).reshape(nch, 2)
    hw = rec[8 * nch:12 * nch].view(np.uint32)
    q = np.empty((nch, 32), np.int64)
    for v in range(32):
        t, i, e = v // 8, (v % 8) // 2, v % 2
        lo = (lw[:, t // 2] >> np.uint32(8 * i + 2 * (2 * (t % 2) + e))) & np.uint32(3)
        hi = (hw >> np.uint32(8 * i + 2 * t + e)) & np.uint32(1)
        q[:, v] = (lo | (hi << np.uint32(2))).astype(np.int64) - 4
    return q.reshape(K), rec[3 * K // 8:3 * K // 8 + K // 32].view(np.uint16)


def _logical_codes(packed: np.ndarray):
    """Codes of logical int3 rows [R, 3K/8] (8 per little-endian 24-bit word)."""
    R, nb = packed.shape
    b = packed.reshape(R, nb // 3, 3).astype(np.int64)
    word = b[:, :, 0] | (b[:, :, 1] << 8) | (b[:, :, 2] << 16)
    q = np.stack([(word >> (3 * j)) & 7 for j in range(8)], axis=2).reshape(R, -1)
    return np.where(q >= 4, q - 8, q)


def test_packed_int3_records_hold_the_logical_codes(gpu_lib):
    m = TINY_E3
    w = SW.model_torch(m, "cuda")
    d = make_desc(m)
    nbytes = L.mk_packed_bytes(d)
    sections, total = _expert_sections(m)
    assert nbytes == total
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ws, _keep = weights_struct(m, w)
    L.mk_pack_weights(d, ws, buf.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    H, FE = m.hidden, m.expert_ffn
    checked = 0
    for l in range(m.n_dense, m.n_layers):
        gu, dn = sections[l]
        for e in (0, m.n_experts - 1):
            for r, name in ((0, "exp_gate"), (1, "exp_up")):
                codes, scales = w[(name, l)]
                q_ref = _logical_codes(codes[e].cpu().numpy())
                s_ref = scales[e].view(torch.int16).cpu().numpy().view(np.uint16)
                for f in (0, 5, FE - 1):
                    o = gu + (2 * (e * FE + f) + r) * _rec("int3", H)
                    q, s = _decode_planes(host[o:o + _rec("int3", H)], H)
                    np.testing.assert_array_equal(q, q_ref[f])
                    np.testing.assert_array_equal(s, s_ref[f])
                    checked += 1
            codes, scales = w[("exp_down", l)]
            q_ref = _logical_codes(codes[e].cpu().numpy())
            s_ref = scales[e].view(torch.int16).cpu().numpy().view(np.uint16)
            for row in (0, 77, H - 1):
                o = dn + (e * H + row) * _rec("int3", FE)
                q, s = _decode_planes(host[o:o + _rec("int3", FE)], FE)
                np.testing.assert_array_equal(q, q_ref[row])
                np.testing.assert_array_equal(s, s_ref[row])
                checked += 1
    assert checked == 18 * (m.n_layers - m.n_dense)


def test_tiny_int3_experts_batch_of_16_matches_the_oracle(gpu_lib):
    m = TINY_E3
    w = SW.model_torch(m, "cuda")
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
    print(rep)
    assert not rep.failures, rep
    assert rep.tokens_checked >= 8, rep
    eng.close()


@pytest.fixture(scope="module")
def flint4_e3():
    m = synth.FLINT_INT4_E3.with_(n_layers=4)
    w = SW.model_torch(m, "cuda")
    yield m, w
    del w
    torch.cuda.empty_cache()


def test_flint_int3_experts_context_2048(gpu_lib, flint4_e3):
    m, w = flint4_e3
    rep = PR.run_single(m, prompt_len=2048, n_decode=8, w=w, n_pages=24, teacher=True)
    _check(rep)


def test_flint_int3_experts_chunked_prefill_then_decode(gpu_lib, flint4_e3):
    """A 64-token prompt runs through the GEMM prefill (int3 expert records
    widened to fp16); the GPU then decodes freely over its own cache."""
    m, w = flint4_e3
    rep = PR.run_single(m, prompt_len=64, n_decode=8, w=w, n_pages=8)
    _check(rep, min_topk=20)


def test_flint_int3_experts_four_rows_match_the_oracle(gpu_lib, flint4_e3):
    """Four sequences of different lengths in one launch on the Flint shape:
    the dense projections on the tensor-core path, the int3 expert rows with
    several activations per tile; every row against the oracle."""
    m, w = flint4_e3
    lens = [17, 40, 90, 130]
    eng = Engine(m, w, n_pages=16, max_ctx=256, max_seqs=4)
    orc = Oracle(m, PR.host_fetch(m, w), cache_bytes=8 << 30)
    toks = torch.empty(4, dtype=torch.int32, device="cuda")
    kvs, nxt = [], []
    for s, n in enumerate(lens):
        p = SP.prompt_tokens(m.seed, m.vocab, n, seq=40 + s)
        kv = orc.new_kv()
        t, _ = orc.prefill(kv, p)
        kvs.append(kv)
        nxt.append(t)
        eng.prefill(s, torch.from_numpy(p).cuda(), out=toks[s:s + 1])
    toks.copy_(torch.tensor(nxt, dtype=torch.int32))
    eng.enable_trace(4)
    eng.decode_step([0, 1, 2, 3], toks, lens, toks)
    eng.sync()
    tr = eng.split_trace(4)
    rep = PR.Report()
    for s in range(4):
        _, tro = orc.decode(kvs[s], nxt[s], lens[s])
        PR.compare_trace(rep, m, tr, tro, slice(s, s + 1), slice(0, 1), PR.tol_for(m), f"seq {s}", seq=s)
        PR.check_token(rep, int(toks[s].item()), int(tro["next_token"][-1]), float(tro["top2_margin"][-1]),
                       f"seq {s}", seq=s)
    print(rep)
    assert not rep.failures, rep
    assert rep.topk_checked >= 6, rep
    eng.close()
