"""Host-side pieces of bench.py that the GPU runs rely on: the committed ncu traffic
records, the backward prologue's byte count, and the reference arm's JSON line
(the fp64 oracle timed on the host, which needs no GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mqa_attention_gb300.workloads import by_name  # noqa: E402


def test_traffic_records_match_their_sources():
    """Each record in profiles/traffic.json is read back while its kernel sources are
    unchanged, and only for the workload it was captured on."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for kernel, recs in rec.items():
        if kernel.startswith("_"):
            continue
        for r in recs if isinstance(recs, list) else [recs]:
            got = bench.ncu_traffic(kernel, r["workload"])
            assert got == float(r["bytes"]), (kernel, r["workload"],
                                              "source hash no longer matches the record")
        assert bench.ncu_traffic(kernel, "tiny_mqa_fwd") is None


def test_backward_prologue_bytes_llama3_8b():
    # q, dO, out: 33,554,432 B each (bf16 [1,32,4096,128]); k, v: 8,388,608 B each;
    # lse, delta, lse*log2e: 524,288 B each; dQ accumulator: 67,108,864 B.
    q, kv, row, acc = 33554432, 8388608, 524288, 67108864
    absmax = 2 * q + 2 * kv
    rows = (3 * q + 2 * kv + row) + (2 * q + 2 * kv + acc + 2 * row)
    assert bench.bwd_prologue_bytes(by_name("llama3_8b_gqa_s4096")) == absmax + rows == 353894400


def test_reference_arm_prints_one_json_line():
    res = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
         "--warmup", "3", "--workload", "palm_mqa_s2048"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["config"]["workload"] == "palm_mqa_s2048"


def test_launch_accounting():
    """gpu_launches counts the library's kernels per step: RoPE pre-pass + forward, then
    zeroing of the abs-max words, abs-max, row pass, main kernel and dq finalisation; the
    exact delta pass by default above 8 query heads per K/V head; two dk / dv passes for
    bf16 gradients or padded rows; the forward-only workload two."""
    llama = by_name("llama3_8b_gqa_s4096")
    assert bench.launches_per_step(llama) == 7
    assert bench.launches_per_step(llama, "exact") == 8
    assert bench.launches_per_step(llama, "auto", "bf16") == 9
    assert bench.launches_per_step(by_name("tiny_mqa_fwd")) == 2
    assert bench.bwd_launches(4096) == 5
    assert bench.bwd_launches(1000) == 7
    assert bench.bwd_launches(4096, "bf16", True) == 8
