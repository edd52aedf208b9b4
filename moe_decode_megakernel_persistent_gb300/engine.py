"""Python-side driver over the C ABI: an Engine that owns one library context
(weights borrowed from torch tensors, KV pool, trace buffer) and a Batcher
that runs continuous batching over it.  PyTorch supplies device memory and
streams only; every step of the decode path runs in the library's kernel.

Weight dict format (what `Engine` expects), torch tensors on the GPU in the
logical layouts of include/mk.h:
    ("embed",) [V, H]   ("final_norm",) [H]   ("lm_head",) W or (codes, scales)
    ("attn_norm", l) ("ffn_norm", l) [H]
    ("wq"|"wk"|"wv"|"wo", l)                   W or (codes, scales)
    dense layers: ("gate"|"up"|"down", l)      W or (codes, scales)
    MoE layers:   ("router", l) [E, H]
                  ("exp_gate"|"exp_up"|"exp_down", l)  stacked over experts (W or
                  (codes, scales) in the experts' format: int3 experts with int4
                  elsewhere, or the layers' format)
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

from . import _lib as L

MAX_PREFILL = 4096
RING_LOG = 1024      # ring items per block the timing record logs


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _i32(t, n: int, what: str):
    """The library reads n int32 values at t's address on the GPU."""
    if not (isinstance(t, torch.Tensor) and t.dtype == torch.int32 and t.is_cuda and t.is_contiguous()
            and t.numel() >= n):
        raise ValueError(f"{what} must be a contiguous int32 CUDA tensor of at least {n} elements")


def _lin(x) -> L.mk_linear:
    if isinstance(x, tuple):
        return L.mk_linear(_ptr(x[0]), _ptr(x[1]))
    return L.mk_linear(_ptr(x), None)


def make_desc(shape, max_batch: int = 16, max_ctx: int = 16384, max_seqs: int = 64) -> L.mk_model_desc:
    """mk_model_desc from an object with the model fields (n_layers, hidden, ...;
    `xdtype`, the experts' format, if it has one)."""
    xdtype = getattr(shape, "xdtype", shape.wdtype)
    return L.mk_model_desc(
        n_layers=shape.n_layers, hidden=shape.hidden, n_heads=shape.n_heads,
        n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim, vocab=shape.vocab,
        n_dense=shape.n_dense, dense_ffn=shape.dense_ffn, n_experts=shape.n_experts,
        top_k=shape.top_k, expert_ffn=shape.expert_ffn, rope_theta=shape.rope_theta,
        rms_eps=shape.rms_eps, wdtype=L.WDTYPES[shape.wdtype], page_tokens=128,
        max_batch=max_batch, max_ctx=max_ctx, max_seqs=max_seqs,
        expert_wdtype=L.WDTYPES[xdtype])


class Engine:
    """One library context: weights, KV pool, sequences."""

    def __init__(self, shape, weights: dict, n_pages: int, max_batch: int = 16,
                 max_ctx: int = 16384, max_seqs: int = 64, device: Optional[int] = None):
        L.load()
        if device is not None:
            torch.cuda.set_device(device)
        self.shape = shape
        self.desc = make_desc(shape, max_batch, max_ctx, max_seqs)
        self._weights = weights  # keep the borrowed tensors alive
        layers = (L.mk_layer_weights * shape.n_layers)()
        for l in range(shape.n_layers):
            lw = layers[l]
            lw.attn_norm = _ptr(weights[("attn_norm", l)])
            lw.ffn_norm = _ptr(weights[("ffn_norm", l)])
            for name in ("wq", "wk", "wv", "wo"):
                setattr(lw, name, _lin(weights[(name, l)]))
            if l < shape.n_dense:
                for name in ("gate", "up", "down"):
                    setattr(lw, name, _lin(weights[(name, l)]))
            else:
                lw.router = _ptr(weights[("router", l)])
                for name in ("exp_gate", "exp_up", "exp_down"):
                    setattr(lw, name, _lin(weights[(name, l)]))
        self._layers = layers
        w = L.mk_weights(embed=_ptr(weights[("embed",)]), final_norm=_ptr(weights[("final_norm",)]),
                         lm_head=_lin(weights[("lm_head",)]), layers=layers)
        self.ctx = L.mk_create(self.desc, w)
        L.mk_kv_alloc(self.ctx, n_pages)
        self.trace = None
        self.max_batch = max_batch

    @property
    def stream(self) -> int:
        return torch.cuda.current_stream().cuda_stream

    # ---- decode path
    def prefill(self, seq_id: int, tokens: torch.Tensor, start_pos: int = 0,
                out: Optional[torch.Tensor] = None) -> Optional[torch.Tensor]:
        """Run prompt tokens (int32 CUDA tensor) in chunks of at most 4096;
        returns the device int32[1] next token after the last position."""
        n = tokens.numel()
        _i32(tokens, n, "tokens")
        if out is None:
            out = torch.empty(1, dtype=torch.int32, device=tokens.device)
        _i32(out, 1, "out")
        for off in range(0, n, MAX_PREFILL):
            m = min(MAX_PREFILL, n - off)
            last = off + m == n
            L.mk_prefill_chunk(self.ctx, seq_id, _ptr(tokens) + 4 * off, m, start_pos + off,
                               _ptr(out) if last else None, self.stream)
        return out

    def decode_step(self, seq_ids, tokens: torch.Tensor, positions, out: torch.Tensor):
        n = len(seq_ids)
        _i32(tokens, n, "tokens")
        _i32(out, n, "out")
        L.mk_decode_step(self.ctx, list(seq_ids), _ptr(tokens), list(positions), _ptr(out),
                         self.stream)
        return out

    def release(self, seq_id: int):
        L.mk_seq_release(self.ctx, seq_id)

    # ---- KV transfers and page sharing
    def kv_write(self, seq_id: int, start_pos: int, kv: torch.Tensor):
        """Store K/V for positions start_pos .. start_pos+n-1: kv is a CUDA
        bfloat16 tensor [n_layers, n, 2, n_kv_heads, head_dim]."""
        assert kv.dtype == torch.bfloat16 and kv.is_cuda and kv.is_contiguous()
        L.mk_kv_write(self.ctx, seq_id, start_pos, kv.shape[1], _ptr(kv), self.stream)

    def kv_read(self, seq_id: int, start_pos: int, n: int) -> torch.Tensor:
        s = self.shape
        out = torch.empty((s.n_layers, n, 2, s.n_kv_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        L.mk_kv_read(self.ctx, seq_id, start_pos, n, _ptr(out), self.stream)
        return out

    def fork(self, src_seq: int, dst_seq: int, n_tokens: int):
        """Open dst_seq sharing the pages of src_seq's first n_tokens
        positions (a multiple of 128)."""
        L.mk_seq_fork(self.ctx, src_seq, dst_seq, n_tokens, self.stream)

    def seq_length(self, seq_id: int) -> int:
        return L.mk_seq_length(self.ctx, seq_id)

    def sync(self):
        L.mk_sync(self.ctx, self.stream)

    def info(self) -> dict:
        return L.mk_get_info(self.ctx)

    # ---- debugging
    def enable_trace(self, rows: int):
        nbytes = L.mk_trace_bytes(self.desc, rows)
        self.trace = torch.zeros(nbytes // 4, dtype=torch.float32, device="cuda")
        L.mk_set_debug(self.ctx, L.MK_DBG_TRACE, 0, _ptr(self.trace), nbytes, 0)

    def enable_timing(self):
        """Per-phase %globaltimer stamps of every block for each following launch."""
        grid = self.info()["grid"]
        R = 16 * self.shape.n_layers + 2
        self.timing = torch.zeros(grid * (R + 3 * RING_LOG), dtype=torch.int64, device="cuda")
        L.mk_set_debug(self.ctx, L.MK_DBG_TIMING, 0, _ptr(self.timing), 8 * self.timing.numel(), 0)

    PHASES = ("qkv", "attention", "oproj", "route+gateup", "down")

    def timing_stamps(self):
        """The last timed launch's stamps as float64 ns [blocks, 16 * n_layers + 2]."""
        R = 16 * self.shape.n_layers + 2
        grid = self.timing.numel() // (R + 3 * RING_LOG)
        return self.timing[:grid * R].view(grid, R).cpu().numpy().astype("float64")

    def ring_log(self):
        """The last timed launch's ring log as float64 ns [blocks, items, 3]
        (issued, landed, released by warp 0; 0 where no item)."""
        R = 16 * self.shape.n_layers + 2
        grid = self.timing.numel() // (R + 3 * RING_LOG)
        return self.timing[grid * R:].view(grid, RING_LOG, 3).cpu().numpy().astype("float64")

    def phase_times_us(self, layers=None) -> dict:
        """Per-phase times (us) of the last timed launch, medians over
        `layers` (default: the MoE layers).  For each phase, from the
        release of the previous grid barrier:
          stage      block 0's activation staging;
          work_med   the median block's time until it arrived at the barrier;
          work_max   the last block's (the critical path);
          barrier    from the last arrival to the first release;
          span       from one release to the next.
        Also lm_head (from the last release) and the launch total."""
        import numpy as np
        t = self.timing_stamps()
        Ln = self.shape.n_layers
        if layers is None:
            layers = range(self.shape.n_dense, Ln) if self.shape.n_dense < Ln else range(Ln)
        per = {k: {"stage": [], "work_med": [], "work_max": [], "barrier": [], "span": []} for k in self.PHASES}
        prev = t[:, 0]
        for l in range(Ln):
            for p, k in enumerate(self.PHASES):
                base = 1 + 16 * l + 3 * p
                st, done, rel = t[:, base], t[:, base + 1], t[:, base + 2]
                st = np.where(st == 0, prev, st)
                if l in layers:
                    start = prev.max()
                    per[k]["stage"].append((st[0] - prev[0]) / 1e3)
                    per[k]["work_med"].append(float(np.median(done - prev)) / 1e3)
                    per[k]["work_max"].append((done.max() - start) / 1e3)
                    per[k]["barrier"].append((rel.min() - done.max()) / 1e3)
                    per[k]["span"].append((rel.max() - start) / 1e3)
                prev = rel
        out = {k: {m: round(float(np.median(v)), 3) for m, v in d.items()} for k, d in per.items()}
        out["lm_head"] = round(float((t[:, 1 + 16 * Ln].max() - prev.max()) / 1e3), 3)
        out["total"] = round(float((t[:, 1 + 16 * Ln].max() - t[:, 0].min()) / 1e3), 3)
        out["layer_median"] = round(sum(out[k]["span"] for k in self.PHASES), 3)
        return out

    def disable_trace(self):
        L.mk_set_debug(self.ctx, 0, 0, 0, 0, 0)
        self.trace = None

    def split_trace(self, rows: int) -> dict:
        """Views of the trace of the last launch of `rows` rows."""
        s = self.shape
        Ln, H, QD, E, K, V = s.n_layers, s.hidden, s.n_heads * s.head_dim, s.n_experts, s.top_k, s.vocab
        t = self.trace
        o = 0
        out = {}
        for name, shp in (("x", (Ln, rows, H)), ("attn", (Ln, rows, QD)),
                          ("router_logits", (Ln, rows, E)), ("topk", (Ln, rows, 2 * K)),
                          ("logits", (rows, V))):
            sz = 1
            for d in shp:
                sz *= d
            out[name] = t[o:o + sz].view(shp)
            o += sz
        return out

    def close(self):
        if self.ctx:
            L.mk_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PrefixCache:
    """Prefix reuse on the page pool: finished sequences stay in the cache
    with their pages; a new prompt that starts with a cached sequence's
    tokens opens its sequence by sharing the longest common prefix in whole
    128-token pages (mk_seq_fork: no K/V is recomputed or copied) and
    prefills only the rest.  Entries are evicted least recently used first
    when the cache holds `capacity` sequences.  The cache owns the sequence
    ids it keeps; callers must not reuse an id the cache holds.

    The workload is the one "rec Megakernel and Tempo9 Compared", §1 (Prefix
    cache) measures: a second turn over the same 8,022-token prompt reuses
    7,936 tokens (62 pages), and returning to a prompt after another one
    reuses it again when its entry is still held."""

    def __init__(self, engine: Engine, capacity: int = 4):
        self.e = engine
        self.capacity = capacity
        self.entries: list = []      # [(seq_id, tokens as a host list)], most recent last

    def _match(self, toks: list) -> tuple:
        best, best_n = None, 0
        for sid, et in self.entries:
            n = 0
            lim = min(len(et), len(toks) - 1)   # keep >= 1 token to prefill (it yields the next token)
            while n < lim and et[n] == toks[n]:
                n += 1
            n = n // 128 * 128
            if n > best_n:
                best, best_n = sid, n
        return best, best_n

    def prefill(self, seq_id: int, tokens: torch.Tensor, out: Optional[torch.Tensor] = None):
        """Open seq_id for `tokens` (int32 CUDA); returns (next-token device
        tensor, reused token count)."""
        toks = tokens.cpu().tolist()
        src, n = self._match(toks)
        if src is not None:
            self.e.fork(src, seq_id, n)
            self.entries = [x for x in self.entries if x[0] != src] + [x for x in self.entries if x[0] == src]
        out = self.e.prefill(seq_id, tokens[n:], start_pos=n, out=out)
        return out, n

    def keep(self, seq_id: int, tokens: list):
        """Retain a finished sequence (its positions hold `tokens`) as an
        entry; evicts the least recently used entry beyond capacity."""
        self.entries.append((seq_id, list(tokens)))
        while len(self.entries) > self.capacity:
            sid, _ = self.entries.pop(0)
            self.e.release(sid)


@dataclasses.dataclass
class Request:
    seq_id: int
    prompt: torch.Tensor         # int32 CUDA tensor
    max_new: int
    arrival: int = 0             # step at which it joins
    generated: list = dataclasses.field(default_factory=list)
    finish_step: int = -1


class Batcher:
    """Continuous batching: every step, requests whose arrival step has come
    are prefilled and join; the active set (up to max_batch) runs as ONE
    decode launch; finished requests leave and release their pages.  Tokens
    stay on the device between steps (a step's inputs are the previous
    step's outputs); with read_back the host copies all generated tokens
    back in one transfer after the last step."""

    def __init__(self, engine: Engine):
        self.e = engine

    def run(self, requests: list, read_back: bool = True, timed: bool = False) -> dict:
        """timed: CUDA events around every decode launch; the result then has
        "decode_ms" (sum over launches) and "steps_ms" [(active rows, ms)]."""
        e = self.e
        dev = getattr(e, "out_device", None) or torch.device("cuda")  # where the step's tokens live
        events = []
        pending = sorted(requests, key=lambda r: (r.arrival, r.seq_id))
        active: list = []
        tok_dev = {}           # seq_id -> device int32[1] with its next input token
        step = 0
        steps_run = 0
        while pending or active:
            while pending and pending[0].arrival <= step and len(active) < e.max_batch:
                r = pending.pop(0)
                out = e.prefill(r.seq_id, r.prompt)
                tok_dev[r.seq_id] = out
                r.generated.append(out)  # first generated token (device)
                if len(r.generated) >= r.max_new:  # the prefill's token was all it asked for
                    r.finish_step = step
                    e.release(r.seq_id)
                else:
                    active.append(r)
            if active:
                ids = [r.seq_id for r in active]
                pos = [e.seq_length(i) for i in ids]
                toks = torch.cat([tok_dev[i] for i in ids])
                outs = torch.empty(len(ids), dtype=torch.int32, device=dev)
                if timed:
                    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    ev[0].record(torch.cuda.current_stream())
                e.decode_step(ids, toks, pos, outs)
                if timed:
                    ev[1].record(torch.cuda.current_stream())
                    events.append((len(ids), ev))
                steps_run += 1
                still = []
                for k, r in enumerate(active):
                    o = outs[k:k + 1]
                    tok_dev[r.seq_id] = o
                    r.generated.append(o)
                    if len(r.generated) >= r.max_new:
                        r.finish_step = step
                        e.release(r.seq_id)
                    else:
                        still.append(r)
                active = still
            step += 1
        if read_back:
            flat = [t for r in requests for t in r.generated]
            host = torch.cat(flat).cpu().tolist() if flat else []
            k = 0
            for r in requests:
                n = len(r.generated)
                r.generated, k = host[k:k + n], k + n
        out = {"steps": step, "launches": steps_run, "finish_step": max(r.finish_step for r in requests)}
        if timed:
            torch.cuda.synchronize()
            out["steps_ms"] = [(n, a.elapsed_time(b)) for n, (a, b) in events]
            out["decode_ms"] = sum(t for _, t in out["steps_ms"])
        return out
