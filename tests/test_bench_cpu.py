"""Host-side pieces of bench.py that need no GPU: the algorithmic bytes the
roofline divides by, the rule that ties the reported DRAM traffic to the
kernel source it was measured on, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_step_bytes_of_the_flint_int4_step_by_hand():
    # Flint int4, batch 1, six distinct experts.  An int4 row of K values is
    # K/2 bytes of codes + K/64 bf16 scales = K * 17/32 bytes.
    m = synth.CONFIGS[3].model
    row = lambda rows, K: rows * K * 17 // 32  # noqa: E731
    attn = row(2048 + 2 * 512, 2048) + row(2048, 2048) + 2 * 2048 * 2  # q, k, v; o; two bf16 norms
    moe = 64 * 2048 * 2 + 6 * 3 * row(768, 2048)                          # bf16 router + 6 experts
    dense = 3 * row(6144, 2048)
    head = row(151936, 2048) + 2048 * 2 + 2048 * 2                        # lm_head, final norm, embed row
    kv_pos = 49 * 2 * 512 * 2                                             # K and V of one position, bf16
    for ctx in (1, 2049, 8023):
        want = 49 * attn + 2 * dense + 47 * moe + head + ctx * kv_pos + kv_pos
        assert bench.step_bytes(m, [ctx], 6) == want
    assert kv_pos == 100352


def test_step_bytes_of_the_int3_expert_step_by_hand():
    # int3 experts: a row of K values is 3K/8 bytes of codes + K/64 bf16
    # scales = K * 13/32 bytes; every other linear layer as in the int4 model
    m4, m3 = synth.CONFIGS[3].model, synth.FLINT_INT4_E3
    row4 = lambda rows, K: rows * K * 17 // 32  # noqa: E731
    row3 = lambda rows, K: rows * K * 13 // 32  # noqa: E731
    per_layer = 6 * 3 * (row4(768, 2048) - row3(768, 2048))
    for ctx in (1, 2049):
        assert bench.step_bytes(m4, [ctx], 6) - bench.step_bytes(m3, [ctx], 6) == 47 * per_layer


def test_reported_traffic_follows_the_kernel_source(monkeypatch):
    wl = "flint-int4-ctx2048"
    with open(os.path.join(ROOT, "profiles", f"step_kernel_{wl}.md")) as fh:
        text = fh.read()
    src = [ln.split(":", 1)[1].strip() for ln in text.splitlines() if ln.startswith("kernel_source_hash:")][0]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: src)
    v = bench.measured_traffic(wl)
    assert v is not None and v > 1e9
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.measured_traffic(wl) is None


def test_reference_arm_prints_its_json_line_on_the_host():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "1", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 1
    assert line["higher_is_better"] is True and line["unit"] == "tok/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
