"""Decode benchmark of the persistent MoE megakernel.

Default workload: the Flint-shaped int4 model (49 layers, hidden 2048, 64
experts top-6, layers 0-1 dense; symmetric int4 group-64 weights from seeded
bf16 N(0, 0.02)), a 2048-token seeded prompt prefilled, then greedy decode
at batch 1.  A step = one decode launch (the whole model, one token).
Timed: exactly --steps steps after --warmup untimed ones (on another
sequence), CUDA events on the launching stream, barrier + synchronize on
both sides.  The step streams ~1.2 GB of weights, far more than L2 (129 MB),
so no L2 flush is needed between steps.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the baseline arm).  Multi-GPU: independent replicas, one process
per GPU (no collective on the data path), `value` = tokens of all ranks /
max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
METRIC = "decode tok/s at batch 1 and 16; achieved HBM GB/s vs GB300 peak"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ------------------------------------------------------------------ bytes model

def step_bytes(m, ctxs, distinct_experts_per_layer) -> int:
    """Algorithmic HBM bytes of one decode step: every weight byte the step
    needs once (norms, attention, router, the distinct selected experts,
    dense MLPs, lm_head, the embedding rows) + the KV cache read (all cached
    positions incl. the new one) + the KV written."""
    H, E = m.hidden, m.n_experts

    def lin(rows, K, fmt=m.wdtype):
        if fmt == "int4":
            return rows * K // 2 + rows * (K // 64) * 2
        if fmt == "int3":
            return rows * 3 * K // 8 + rows * (K // 64) * 2
        return rows * K * (2 if fmt == "bf16" else 4)
    aux = 2 if m.aux_dtype == "bf16" else 4
    attn = lin(m.q_dim, H) + 2 * lin(m.kv_dim, H) + lin(H, m.q_dim) + 2 * H * aux
    xd = getattr(m, "xdtype", m.wdtype)
    expert = 2 * lin(m.expert_ffn, H, xd) + lin(H, m.expert_ffn, xd)
    dense = 2 * lin(m.dense_ffn, H) + lin(H, m.dense_ffn)
    total = 0
    for l in range(m.n_layers):
        total += attn
        if l < m.n_dense:
            total += dense
        else:
            total += E * H * aux + distinct_experts_per_layer * expert
    total += lin(m.vocab, H) + H * aux + len(ctxs) * H * aux
    kv_tok = m.n_layers * 2 * m.kv_dim * 2
    total += sum(ctxs) * kv_tok                 # read (includes the new position)
    total += len(ctxs) * kv_tok                 # write
    return int(total)


# the decode kernel's own sources: its translation unit and the library headers
# that hold its code and data structures (host-only code, the prefill and the
# packer do not change the kernel the DRAM traffic figure was measured on)
KERNEL_SOURCES = ("csrc/mk_kernel.cu", "csrc/mk_device.cuh", "csrc/mk_internal.h")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "moe_decode_megakernel_persistent_gb300")
    for f in KERNEL_SOURCES:
        with open(os.path.normpath(os.path.join(pkg, f)), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"step_kernel_{workload}.md")
    if not os.path.exists(p):
        return None
    src = None
    traffic = None
    for line in open(p):
        if line.startswith("kernel_source_hash:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    if src != kernel_source_hash():
        return None
    return traffic


# ------------------------------------------------------------------ replicas

def aggregate_over_ranks(ms: float, tokens: int, device):
    """Replicas only: every rank decodes its own sequences, no data-path
    collective.  The step time is the slowest rank's, the throughput all
    ranks' tokens over it."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return ms, tokens
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    k = torch.tensor([tokens], dtype=torch.int64, device=device)
    dist.all_reduce(k, op=dist.ReduceOp.SUM)
    return float(t.item()), int(k.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU baseline

def cpu_baseline(m, weights, n_steps: int = 2, prompt_len: int = 4):
    """The oracle as it stands, on this host's cores: a bounded sample of the
    workload (batch-1 decode steps at a short context; weight dequantisation
    included; copying the generator's weights to the host excluded)."""
    from oracle import Oracle
    from synth import prompts as SP
    from tests._parity import host_fetch
    base = host_fetch(m, weights)
    spent = [0.0]

    def fetch(*k):
        t0 = time.perf_counter()
        r = base(*k)
        spent[0] += time.perf_counter() - t0
        return r
    prompt = SP.prompt_tokens(m.seed, m.vocab, prompt_len)
    orc = Oracle(m, fetch, cache_bytes=1 << 30)
    kv = orc.new_kv()
    tok, _ = orc.prefill(kv, prompt)
    s0 = spent[0]
    t0 = time.perf_counter()
    for i in range(n_steps):
        tok, _ = orc.decode(kv, tok, prompt_len + i)
    dt = time.perf_counter() - t0 - (spent[0] - s0)
    return {"value": round(n_steps / dt, 5), "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_steps} float64 oracle decode steps of the same model at batch 1, context "
                      f"{prompt_len + 1}..{prompt_len + n_steps} (the workload's is 2048+), "
                      f"dequantisation included, BLAS single-threaded"}


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, world):
    import torch
    import synth
    from synth import prompts as SP
    from synth import weights as SW
    from moe_decode_megakernel_persistent_gb300 import _build
    from moe_decode_megakernel_persistent_gb300.engine import Engine

    _build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = synth.CONFIGS[args.config]
    m = w.model
    K, W = args.steps, args.warmup
    t0 = time.time()
    weights = SW.model_torch(m, dev)
    torch.cuda.synchronize()
    gen_s = time.time() - t0
    prompt_len = w.prompt_len
    max_ctx = prompt_len + K + 2 * args.e2e_steps + W + 64 + args.split_steps + 2
    pages = 3 * ((max_ctx + 127) // 128) + 8
    eng = Engine(m, weights, n_pages=pages, max_ctx=max_ctx, max_seqs=4)

    def eng_factory(n_pages, max_ctx16, max_seqs):
        return Engine(m, weights, n_pages=n_pages, max_ctx=max_ctx16, max_seqs=max_seqs)
    stream = torch.cuda.current_stream()

    # warm-up sequence: a short prompt and W decode steps
    wtok = torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, 64, seq=1)).to(dev)
    tok1 = eng.prefill(1, wtok)
    for i in range(W):
        eng.decode_step([1], tok1, [64 + i], tok1)
    eng.sync()
    eng.release(1)

    # the measured sequence: prefill the prompt, then K timed decode steps
    prompt = torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, prompt_len)).to(dev)
    t0 = time.time()
    tok = eng.prefill(0, prompt)
    eng.sync()
    prefill_s = time.time() - t0
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        eng.decode_step([0], tok, [prompt_len + i], tok)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    eng.sync()
    ms, total_tokens = aggregate_over_ranks(e0.elapsed_time(e1), K, dev)
    ms_per_step = ms / K

    # the same decode step run as one launch per phase group of a layer and
    # one for lm_head (MK_DBG_SPLIT): kernel boundaries in place of the grid
    # barriers between groups, on the same device code
    split = None
    if args.split_steps > 0:
        from moe_decode_megakernel_persistent_gb300 import _lib as Lb
        Ks = args.split_steps
        pos_s = prompt_len + K
        Lb.mk_set_debug(eng.ctx, Lb.MK_DBG_SPLIT, 0, 0, 0, 0)
        for i in range(2):
            eng.decode_step([0], tok, [pos_s], tok)
            pos_s += 1
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(Ks):
            eng.decode_step([0], tok, [pos_s + i], tok)
        e1.record(stream)
        torch.cuda.synchronize()
        Lb.mk_set_debug(eng.ctx, 0, 0, 0, 0, 0)
        eng.sync()
        split_ms = e0.elapsed_time(e1) / Ks
        groups = 4 * m.n_layers
        split = {"ms_per_step": round(split_ms, 4), "persistent_ms_per_step": round(ms_per_step, 4),
                 "launches_per_step": groups + 1,
                 # one-row persistent step: four grid barriers per layer, the residual
                 # passed to the next layer by flagged words, one barrier before lm_head
                 "grid_barriers_per_step_persistent": 4 * m.n_layers + 1,
                 "boundaries_replacing_barriers": groups,
                 "us_per_boundary_minus_barrier": round((split_ms - ms_per_step) * 1e3 / groups, 3),
                 "note": "context grows by 2 + K steps before the split run; a boundary replaces a "
                         "grid barrier or, after a layer's down phase, the flagged-word exchange"}
        K_extra = Ks + 2
    else:
        K_extra = 0

    # end to end through the public API with host buffers: each step copies
    # its input token from pinned host memory, runs, reads the result back
    E = args.e2e_steps
    h_in = torch.empty(1, dtype=torch.int32, pin_memory=True)
    h_out = torch.empty(1, dtype=torch.int32, pin_memory=True)
    d_in = torch.empty(1, dtype=torch.int32, device=dev)
    d_out = torch.empty(1, dtype=torch.int32, device=dev)
    tok2 = eng.prefill(2, prompt)
    h_in.copy_(tok2.cpu())
    eng.sync()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(E):
        d_in.copy_(h_in, non_blocking=True)
        eng.decode_step([2], d_in, [prompt_len + i], d_out)
        h_out.copy_(d_out, non_blocking=True)
        stream.synchronize()
        h_in[0] = h_out[0]
    e2e_s = time.perf_counter() - t0
    eng.sync()

    # the 16-client workload: 16 sequences, prompt lengths U[256, 8192] and
    # arrival steps U[0, 64] from the schedule (seed 4), 256 generated tokens
    # each, continuously batched (one decode launch per step for the active
    # sequences; arrivals prefilled when they join)
    b16 = None
    if args.batch16_steps > 0 and args.config in (3, 5):
        b16 = run_batch16(eng_factory, m, dev, world, args)

    # per-phase timeline of one more decode launch (MK_DBG_TIMING), outside
    # the timed region: medians over the MoE layers
    timeline = None
    if not args.no_timeline:
        eng.enable_timing()
        pos_t = prompt_len + K + K_extra
        for _ in range(2):          # the second launch is the one kept
            eng.decode_step([0], tok, [pos_t], tok)
            pos_t += 1
        eng.sync()
        timeline = eng.phase_times_us()
        if args.timeline_out:
            np.savez(args.timeline_out, stamps=eng.timing_stamps(), ring=eng.ring_log(),
                     n_layers=m.n_layers, n_dense=m.n_dense)
        eng.disable_trace()

    ctxs = [prompt_len + i + 1 for i in range(K)]
    bytes_avg = sum(step_bytes(m, [c], m.top_k) for c in ctxs) / K
    peaks, peak_kind = load_peaks()
    achieved = bytes_avg / (ms_per_step * 1e-3) / 1e9
    traffic = measured_traffic(w.name)
    out = {
        "metric": METRIC,
        "value": round(total_tokens / (ms / 1e3), 2),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4 weights x 24-bit fixed-point activations (dp4a), fp32 accumulate" if m.wdtype == "int4"
                 else f"{m.wdtype} weights, fp32 activations and accumulate",
        "data": "synthetic: seeded N(0,0.02) weights, seeded uniform prompt tokens",
        "config": {"workload": f"{w.name}: Flint-shaped MoE (49 layers, hidden 2048, 64 experts top-6, "
                               f"dense layers 0-1), {m.wdtype} linear layers, {prompt_len}-token prompt, "
                               f"greedy decode batch 1",
                   "batch": 1, "context": [prompt_len + 1, prompt_len + K],
                   "l2": "inputs larger than L2 (~1.2 GB of weights streamed per step); no flush",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(world * E / e2e_s, 2), "unit": "tok/s",
                "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 4},
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "peak_kind": peak_kind,
                     "bytes_per_step": int(bytes_avg)},
        "clocks": clk,
        "setup_s": {"weights": round(gen_s, 1), "prefill": round(prefill_s, 3)},
    }
    if timeline is not None:
        out["timeline_us"] = timeline
    if split is not None:
        out["dispatch_vs_barrier"] = split
    if b16 is not None:
        out["batch16"] = b16
        if "full_batch" in b16:
            fb = b16["full_batch"]
            # bytes of one full-batch step: 16 rows at the workload's mean
            # context, the distinct experts of 16 uniformly routed rows
            sched = __import__("synth").prompts.schedule(__import__("synth").CONFIGS[5])
            mean_ctx = statistics.mean(L for _, L in sched) + 128
            distinct = 64 * (1 - (1 - 6 / 64) ** 16)
            bps = step_bytes(m, [int(mean_ctx)] * 16, distinct)
            ach = bps / (fb["ms_per_step"] * 1e-3) / 1e9
            fb["roofline"] = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": round(ach / peaks["hbm_gbs"], 4), "bytes_per_step": int(bps),
                              "bytes_model": "16 rows at the mean context of the workload + 128, distinct experts "
                                             "64 (1 - (1 - 6/64)^16) per MoE layer"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(m, weights)
    eng.close()
    if args.int3_steps > 0 and args.config == 3:
        del weights
        torch.cuda.empty_cache()
        out["int3_experts"] = run_int3(args, dev)
    return out


def run_int3(args, dev):
    """The lower-bit expert variant: the same Flint model and workload as the
    batch-1 line (2048-token prompt, greedy decode), the expert matrices in
    int3 and every other linear layer in int4."""
    import torch
    import synth
    from synth import prompts as SP
    from synth import weights as SW
    from moe_decode_megakernel_persistent_gb300.engine import Engine
    wl = synth.EXTRA["flint-int4e3-ctx2048"]
    m, K, W = wl.model, args.int3_steps, max(args.warmup, 3)
    weights = SW.model_torch(m, dev)
    prompt_len = wl.prompt_len
    max_ctx = prompt_len + K + W + 72
    eng = Engine(m, weights, n_pages=2 * ((max_ctx + 127) // 128) + 8, max_ctx=max_ctx, max_seqs=4)
    stream = torch.cuda.current_stream()
    wtok = torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, 64, seq=1)).to(dev)
    tok1 = eng.prefill(1, wtok)
    for i in range(W):
        eng.decode_step([1], tok1, [64 + i], tok1)
    eng.sync()
    eng.release(1)
    prompt = torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, prompt_len)).to(dev)
    t0 = time.time()
    tok = eng.prefill(0, prompt)
    eng.sync()
    prefill_s = time.time() - t0
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        eng.decode_step([0], tok, [prompt_len + i], tok)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    eng.sync()
    eng.close()
    ms = e0.elapsed_time(e1) / K
    ctxs = [prompt_len + i + 1 for i in range(K)]
    bytes_avg = sum(step_bytes(m, [c], m.top_k) for c in ctxs) / K
    peaks, peak_kind = load_peaks()
    achieved = bytes_avg / (ms * 1e-3) / 1e9
    return {"workload": f"{wl.name}: the batch-1 workload with int3 experts (group 64), int4 elsewhere",
            "value": round(1e3 / ms, 2), "unit": "tok/s", "steps": K, "ms_per_step": round(ms, 4),
            "gpu_launches": K, "setup_s": {"prefill": round(prefill_s, 3)},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_kind": peak_kind,
                         "bytes_per_step": int(bytes_avg)},
            "clocks": clk}


def run_batch16(eng_factory, m, dev, world, args):
    """The 16-client workload through the continuous batcher.  Reported:
    aggregate decode tok/s (generated tokens / summed decode-launch device
    time), end-to-end tok/s (generated tokens / wall time including every
    prefill), the finish step, and for the steps with all 16 sequences active
    their mean time and roofline."""
    import torch
    import synth
    from synth import prompts as SP
    from moe_decode_megakernel_persistent_gb300.engine import Batcher, Request
    w5 = synth.CONFIGS[5]
    sched = SP.schedule(w5)
    gen = w5.decode_tokens
    pages = sum((L + gen + 127) // 128 for _, L in sched) + 16
    eng = eng_factory(pages, max(L for _, L in sched) + gen + 8, 16)
    reqs = [Request(seq_id=i, prompt=torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, L, seq=300 + i)).to(dev),
                    max_new=gen, arrival=a) for i, (a, L) in enumerate(sched)]
    # warm-up: a short request through the same engine
    Batcher(eng).run([Request(seq_id=0, prompt=reqs[0].prompt[:64], max_new=4, arrival=0)])
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    out = Batcher(eng).run(reqs, read_back=False, timed=True)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    eng.sync()
    tokens = sum(r.max_new for r in reqs)
    full = [t for n, t in out["steps_ms"] if n == 16]
    # distinct experts per MoE layer of a 16-row launch, from one traced step
    # over 16 fresh sequences at the workload's mean prompt length
    eng.close()
    res = {"workload": f"{w5.name}: 16 sequences, prompt lengths U[256, 8192] and arrival steps U[0, 64] "
                       f"(seed 4), {gen} greedy tokens each, continuous batching",
           "value": round(world * tokens / (out["decode_ms"] / 1e3), 2), "unit": "tok/s",
           "decode_ms_total": round(out["decode_ms"], 1), "launches": out["launches"],
           "e2e": {"value": round(world * tokens / wall, 2), "unit": "tok/s",
                   "wall_s": round(wall, 2), "includes": "every prefill and decode launch"},
           "finish_step": out["finish_step"], "prompt_tokens": sum(L for _, L in sched),
           "clocks": clocks}
    if full:
        ms16 = statistics.median(full)
        res["full_batch"] = {"steps": len(full), "ms_per_step": round(ms16, 3),
                             "value": round(world * 16 / (ms16 / 1e3), 2), "unit": "tok/s"}
    return res


class TimedFetch:
    """Oracle weight source over the seeded generator that keeps what it
    produced and the time spent producing it (excluded from oracle timings).
    The experts of a layer are drawn together in a thread pool."""

    def __init__(self, m, threads: int):
        from concurrent.futures import ThreadPoolExecutor
        from synth import weights as SW
        self.m, self.SW = m, SW
        self.pool = ThreadPoolExecutor(threads)
        self.cache = {}
        self.seconds = 0.0

    def __call__(self, name, layer, expert):
        key = (name, layer, expert)
        if key not in self.cache:
            t0 = time.perf_counter()
            m, SW = self.m, self.SW
            if expert is not None:
                futs = {e: self.pool.submit(SW.linear_np, m, name, layer, e) for e in range(m.n_experts)}
                for e, f in futs.items():
                    self.cache[(name, layer, e)] = (f.result(), m.wdtype)
            elif name in ("embed", "attn_norm", "ffn_norm", "final_norm", "router"):
                self.cache[key] = (SW.raw_np(m, name, layer), m.aux_dtype)
            else:
                shp = SW.tensor_shape(m, name)
                step = max(1, shp[0] // 16)
                parts = [self.pool.submit(SW.linear_np, m, name, layer, None, (r, min(shp[0], r + step)))
                         for r in range(0, shp[0], step)]
                res = [f.result() for f in parts]
                if m.wdtype == "int4":
                    val = (np.concatenate([a for a, _ in res]), np.concatenate([b for _, b in res]))
                else:
                    val = np.concatenate(res)
                self.cache[key] = (val, m.wdtype)
            self.seconds += time.perf_counter() - t0
        return self.cache[key]


def run_reference(args, rank, world):
    """The CPU oracle on a bounded sample of the same workload.  A step is one
    MoE decoder layer of a batch-1 decode token (attention block and FFN
    block, weight dequantisation included), cycling over a few consecutive
    MoE layers; tok/s counts a step as 1 / (layers of the model) tokens.  The
    oracle's weight cache is off: in a full-model run every layer's weights
    are evicted before their next use, so each use pays the dequantisation;
    a cached sample of a few layers would hide it.  Left out of the per-token
    estimate: the embedding row and the lm_head (once per token), and the
    two dense layers' extra width (within 1 % of the token)."""
    if rank != 0:
        return None
    import synth
    from oracle import Oracle
    w = synth.CONFIGS[args.config]
    m = w.model
    threads = os.cpu_count() or 1
    fetch = TimedFetch(m, threads)
    orc = Oracle(m, fetch, cache_bytes=0)
    L = m.n_layers
    sample = list(range(m.n_dense, min(L, m.n_dense + 4)))
    prompt_len = 2
    rng = np.random.default_rng(m.seed + 7)
    kv = orc.new_kv()
    # the sampled layers' cache for a short prompt (a seeded residual stands
    # in for the embedding rows: the cost does not depend on the values;
    # layers outside the sample are never read)
    x = 0.02 * rng.standard_normal((prompt_len, m.hidden))
    for l in sample:
        h, _ = orc._attn_block(l, x, kv, 0, False)
        x = orc._ffn_block(l, h, {"router_logits": [], "topk_ids": [], "topk_w": [], "topk_margin": []})
    state = {"i": 0, "pos": prompt_len, "x": 0.02 * rng.standard_normal((1, m.hidden))}

    def step():
        l = sample[state["i"]]
        tr = {"router_logits": [], "topk_ids": [], "topk_w": [], "topk_margin": []}
        h, _ = orc._attn_block(l, state["x"], kv, state["pos"], True)
        state["x"] = orc._ffn_block(l, h, tr)
        state["i"] += 1
        if state["i"] == len(sample):  # next token
            state["i"] = 0
            state["pos"] += 1
            state["x"] = 0.02 * rng.standard_normal((1, m.hidden))

    for _ in range(args.warmup):
        step()
    g0 = fetch.seconds
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0 - (fetch.seconds - g0)
    toks = args.steps / L
    v = toks / dt
    sample = (f"{args.steps} steps of one MoE decoder layer each (layers {sample[0]}..{sample[-1]} in turn) = "
              f"{toks:.2f} batch-1 decode tokens of the {w.name} model in float64 at context "
              f"{prompt_len + 1}+ (the workload's context is {w.prompt_len}+); weight dequantisation included "
              f"(no weight cache), weight generation excluded, embedding row and lm_head left out; "
              f"BLAS single-threaded")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded N(0,0.02) weights; seeded N(0,0.02) residual vectors in place of embedding rows",
            "config": {"workload": w.name, "batch": 1},
            "cpu_baseline": {"value": round(v, 5), "unit": "tok/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 5), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """A short run for ncu captures of the decode launch: --rows sequences
    with the workload's prompt (rows > 1: the first 2048 tokens of it)
    prefilled, then --steps decode launches of all rows; nothing else (no
    CPU baseline, no e2e).  --layers keeps the first layers of the model (the
    same layer weights; a reduced-depth case for captures that must stay
    small)."""
    import torch
    import synth
    from synth import prompts as SP
    from synth import weights as SW
    from moe_decode_megakernel_persistent_gb300 import _build
    from moe_decode_megakernel_persistent_gb300.engine import Engine

    _build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = synth.CONFIGS[args.config]
    m = w.model if not args.layers else w.model.with_(n_layers=args.layers)
    weights = SW.model_torch(m, dev)
    rows = args.rows
    prompt_len = w.prompt_len if rows == 1 else min(2048, w.prompt_len or 2048)
    max_ctx = prompt_len + args.steps + 16
    eng = Engine(m, weights, n_pages=rows * ((max_ctx + 127) // 128 + 1), max_ctx=max_ctx, max_seqs=rows)
    toks = torch.empty(rows, dtype=torch.int32, device=dev)
    for r in range(rows):
        prompt = torch.from_numpy(SP.prompt_tokens(m.seed, m.vocab, prompt_len, seq=r)).to(dev)
        eng.prefill(r, prompt, out=toks[r:r + 1])
    ids = list(range(rows))
    for i in range(args.steps):
        eng.decode_step(ids, toks, [prompt_len + i] * rows, toks)
    eng.sync()
    print(json.dumps({"profile_case": w.name, "layers": m.n_layers, "rows": rows, "prompt": prompt_len,
                      "decode_launches": args.steps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch16-steps", type=int, default=1,
                    help="run the 16-client continuous-batching workload (0 = skip)")
    ap.add_argument("--no-timeline", action="store_true", help="skip the per-phase timeline launch")
    ap.add_argument("--int3-steps", type=int, default=64,
                    help="decode steps timed on the int3-expert model (0 = skip)")
    ap.add_argument("--split-steps", type=int, default=16,
                    help="decode steps timed as one launch per phase group (0 = skip)")
    ap.add_argument("--timeline-out", default="", help="save the timeline launch's raw stamps (.npz)")
    ap.add_argument("--profile-case", action="store_true",
                    help="prefill + --steps decode launches only (for an ncu capture)")
    ap.add_argument("--layers", type=int, default=0, help="profile case: keep the first N layers")
    ap.add_argument("--rows", type=int, default=1, help="profile case: rows per decode launch")
    args = ap.parse_args()
    if args.profile_case:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        run_profile_case(args)
        return
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out))
        return
    import torch
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    out = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
