"""Throughput benchmark: causal RoPE GQA attention forward + backward on GB300.

One step = attn_fwd + attn_bwd (every kernel of the hot path) over one batch
of seeded synthetic bf16 inputs of the chosen workload (default: the
Llama-3-8B attention layer, B=1, Hq=32, Hkv=8, S=4096, D=128). Prints one
JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

value: causal-pair FLOPs (fwd 4*D, bwd 10*D per unmasked (query, key) pair)
of all ranks / device time of K steps (CUDA events on the launching stream,
L2 flushed between steps, inputs resident in HBM). e2e: the same metric with
host buffers: each step copies the inputs from pinned host memory, runs the
C-ABI calls and copies every output back; the copies of neighbouring steps run
on two copy streams while a step computes (two device buffer sets). roofline: the dominant kernel's
achieved TFLOP/s from library-recorded CUDA events over the timed region,
against the measured dense bf16 peak. cpu_baseline: the fp64 oracle on a
bounded sample, on this host's cores. --impl reference times that oracle as
the reference arm.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mqa_attention_gb300 import inputs as I  # noqa: E402
from mqa_attention_gb300.workloads import WORKLOADS, by_name  # noqa: E402

DEFAULT_WORKLOAD = "llama3_8b_gqa_s4096"
METRIC = ("causal GQA attn fwd+bwd TFLOP/s (Llama-3-8B S=4096 shape), % of GB300 bf16 peak in "
          "roofline")
L2_FLUSH_BYTES = 256 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=[w.name for w in WORKLOADS])
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rope", choices=["half", "interleaved"], default="half",
                    help="RoPE pair layout (interleaved runs attn_fwd_ex / attn_bwd_ex)")
    ap.add_argument("--grads", choices=["fp32", "bf16"], default="fp32",
                    help="gradient dtype (bf16 runs attn_bwd_bf16)")
    ap.add_argument("--delta", choices=["auto", "exact", "from_out"], default="auto",
                    help="delta of the backward: attn_bwd's choice, the exact pass over the "
                         "scores (ATTN_DELTA_EXACT) or dout . out (ATTN_DELTA_FROM_OUT)")
    ap.add_argument("--exact-rope", action="store_true",
                    help="rotated q, k rounded as the exact rotation rounds (ATTN_ROPE_EXACT)")
    ap.add_argument("--decode", type=int, default=0, metavar="SQ",
                    help="SQ > 0: time attn_decode, SQ new tokens per sequence against a "
                         "cache of the workload's S keys (HBM-bound: reported in GB/s)")
    ap.add_argument("--single", action="store_true",
                    help="time only --workload (by default the other workloads follow the "
                         "headline under other_workloads)")
    ap.add_argument("--blocks", type=int, default=1,
                    help="N > 1: run the step as N x N query / key-value blocks through "
                         "attn_fwd_partial, attn_merge and attn_bwd_partial")
    a = ap.parse_args()
    a.warmup = max(3, a.warmup)
    return a


def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu records
    (one record, or a list of them, per kernel), or None when there is no record for
    that workload or the kernel source changed since it was taken."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            recs = json.load(f)[kernel]
        for rec in recs if isinstance(recs, list) else [recs]:
            if rec["workload"] != workload:
                continue
            h = hashlib.sha256()
            for src in rec["sources"]:
                with open(os.path.join(ROOT, src), "rb") as f:
                    h.update(f.read())
            return float(rec["bytes"]) if h.hexdigest()[:16] == rec["source_sha256_16"] else None
        return None
    except Exception:
        return None


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ inputs
def host_inputs(wl, rank):
    """Seeded bf16 bit patterns (uint16) per tensor; ranks draw distinct streams."""
    return {n: I.normal_bf16_bits(I.seed_for(wl.index, n) + 100 * rank, s)
            for n, s in wl.shapes().items()}


def to_bf16_tensor(bits, device=None, pin=False):
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    if pin:
        return t.pin_memory()
    return t.to(device) if device is not None else t


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons (200 ms period)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [r for t, r in self.rows if t0 <= t <= t1 + 0.2]
        used = inside if inside else [r for _, r in self.rows]
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in used:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ oracle timing
def oracle_sample_heads(wl, host, budget_s=10.0):
    """fp64 oracle forward + backward of whole query heads (each with its KV
    head) until `budget_s` of CPU time is spent. Returns (TFLOP/s, heads, s)."""
    import oracle as O

    f = {n: torch.from_numpy(I.bf16_bits_to_f64(host[n])) for n in host}
    G = wl.Hq // wl.Hkv
    per_head = (4 + (10 if wl.backward else 0)) * wl.D * (wl.S * (wl.S + 1) // 2)
    t0 = time.perf_counter()
    done = 0
    for b in range(wl.B):
        for h in range(wl.Hq):
            g = h // G
            q = f["q"][b:b + 1, h:h + 1]
            k, v = f["k"][b:b + 1, g:g + 1], f["v"][b:b + 1, g:g + 1]
            O.attention_forward(q, k, v, wl.scale, wl.theta, wl.causal)
            if wl.backward:
                O.attention_backward(q, k, v, f["dout"][b:b + 1, h:h + 1], wl.scale, wl.theta,
                                     wl.causal)
            done += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return done * per_head / dt / 1e12, done, dt


def oracle_sample_rows(wl, host, rows_per_head=64, budget_s=5.0):
    """fp64 oracle out, lse and dq of `rows_per_head` seeded query rows of successive
    heads (for sequences too long for whole heads), until `budget_s` is spent.
    Credited 10*D FLOPs per causal pair of those rows (the reference arm's unit).
    Returns (TFLOP/s, heads, s)."""
    import oracle as O

    f = {n: torch.from_numpy(I.bf16_bits_to_f64(host[n])) for n in host}
    G = wl.Hq // wl.Hkv
    rng = np.random.default_rng(4321)
    t0 = time.perf_counter()
    flops, done = 0, 0
    while time.perf_counter() - t0 < budget_s and done < wl.B * wl.Hq:
        b, h = divmod(done, wl.Hq)
        rows = torch.from_numpy(np.sort(rng.choice(wl.S, size=rows_per_head, replace=False)))
        q = f["q"][b:b + 1, h:h + 1]
        k, v = f["k"][b:b + 1, h // G:h // G + 1], f["v"][b:b + 1, h // G:h // G + 1]
        O.forward_rows(q, k, v, rows, wl.scale, wl.theta, wl.causal)
        O.backward_dq_rows(q, k, v, f["dout"][b:b + 1, h:h + 1], rows, wl.scale, wl.theta,
                           wl.causal)
        flops += 10 * wl.D * (int((rows + 1).sum()) if wl.causal else rows_per_head * wl.S)
        done += 1
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, done, dt


def cpu_baseline_of(wl, host, budget_s):
    """The oracle on this host: whole heads (fwd(+bwd)) where a head takes at most a few
    seconds, sampled rows otherwise."""
    threads = torch.get_num_threads()
    if wl.S <= 8192:
        tf, heads, secs = oracle_sample_heads(wl, host, budget_s)
        sample = (f"{heads} of {wl.B * wl.Hq} query heads, full S={wl.S}, "
                  f"fwd{'+bwd' if wl.backward else ''} in fp64 ({secs:.1f} s)")
    else:
        tf, heads, secs = oracle_sample_rows(wl, host, budget_s=budget_s)
        sample = (f"64 seeded query rows of each of {heads} heads (out, lse, dq in fp64), "
                  f"{secs:.1f} s")
    return {"value": tf, "unit": "TFLOP/s", "cores": threads, "host_cores": os.cpu_count(),
            "kind": "oracle", "sample": sample}


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    """The fp64 oracle timed as the reference arm (rank 0 only). Each step: the
    out, lse and dq rows of 64 query rows of one head (rows spread over the
    sequence), credited 10*D FLOPs per causal pair of those rows (Q.Kᵀ, P.V,
    recomputed Q.Kᵀ, dO.Vᵀ, dS.K)."""
    if rank != 0:
        return
    import oracle as O

    wl = by_name(args.workload)
    host = host_inputs(wl, 0)
    f = {n: torch.from_numpy(I.bf16_bits_to_f64(host[n])) for n in host}
    G = wl.Hq // wl.Hkv
    R = 64
    rng = np.random.default_rng(12345)
    times, flops = [], []
    for step in range(args.warmup + args.steps):
        h = step % wl.Hq
        b = (step // wl.Hq) % wl.B
        rows = torch.from_numpy(np.sort(rng.choice(wl.S, size=R, replace=False)))
        q = f["q"][b:b + 1, h:h + 1]
        k, v = f["k"][b:b + 1, h // G:h // G + 1], f["v"][b:b + 1, h // G:h // G + 1]
        t0 = time.perf_counter()
        O.forward_rows(q, k, v, rows, wl.scale, wl.theta, wl.causal)
        O.backward_dq_rows(q, k, v, f["dout"][b:b + 1, h:h + 1], rows, wl.scale, wl.theta,
                           wl.causal)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            pairs = int((rows + 1).sum()) if wl.causal else R * wl.S
            flops.append(10 * wl.D * pairs)
    total = sum(times)
    value = sum(flops) / total / 1e12
    unit = "TFLOP/s"
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value, "unit": unit, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic N(0,1) bf16 inputs, seeded",
        "config": config_of(wl, args.gpus),
        "cpu_baseline": {"value": value, "unit": unit, "cores": torch.get_num_threads(),
                         "host_cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"per step {R} query rows of one head (out, lse, dq)"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bwd_prologue_bytes(wl):
    """Algorithmic HBM bytes of the backward prologue (abs-max pass + row pass) for an
    unpadded self-attention shape: the abs-max pass reads q, k, v, dO; the row pass
    reads q, dO, out, k, v, lse and writes fp16 q~, dO, k~, v, the zeroed fp32 dQ
    accumulator (twice a bf16 tensor), delta and lse * log2 e."""
    qb = wl.B * wl.Hq * wl.S * wl.D * 2       # one bf16 / fp16 [B,Hq,S,D] tensor
    kb = wl.B * wl.Hkv * wl.S * wl.D * 2      # one bf16 / fp16 [B,Hkv,S,D] tensor
    rb = wl.B * wl.Hq * wl.S * 4              # one fp32 [B,Hq,S] row vector
    absmax = 2 * qb + 2 * kb
    reads = 3 * qb + 2 * kb + rb
    writes = 2 * qb + 2 * kb + 2 * qb + 2 * rb
    return absmax + reads + writes


L2_NOTE = ("GPU arm: L2 flushed between steps (256 MiB write); the host oracle arm has no "
           "device cache")


def config_of(wl, n, rope="half", grads="fp32", l2=L2_NOTE, delta="auto", exact_rope=False):
    c = {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "S": wl.S, "D": wl.D,
         "rope_theta": wl.theta, "rope": rope, "grads": grads, "causal": wl.causal,
         "passes": "fwd+bwd" if wl.backward else "fwd", "parallelism": f"replicas x{n}",
         "l2": l2}
    if delta != "auto":
        c["delta"] = delta
    if exact_rope:
        c["rope_rounding"] = "exact"
    return c


# ------------------------------------------------------------------ our arm
def kernel_names(M):
    return ((M.KERNEL_ROPE, "rope"), (M.KERNEL_FWD, "attn_fwd"), (M.KERNEL_BWD_PREP, "bwd_prep"),
            (M.KERNEL_DELTA, "delta"), (M.KERNEL_BWD_MAIN, "attn_bwd_main"),
            (M.KERNEL_DQ_FINAL, "dq_finalize"))


def bwd_launches(rows, grads="fp32", exact_delta=False):
    """Our kernels in one backward call over `rows` query and key rows per head: zeroing
    of the abs-max words + abs-max + pre-pass (+ the exact delta pass) + main + dq
    finalisation, and two dk / dv passes for bf16 gradients or padded rows."""
    padded = rows % 128 != 0
    return 5 + (1 if exact_delta else 0) + (2 if padded or grads == "bf16" else 0)


def launches_per_step(wl, delta="auto", grads="fp32"):
    """Our kernels in one step: RoPE pre-pass + forward, then the backward call's
    (bwd_launches; the exact delta pass by default for groups above 8)."""
    if not wl.backward:
        return 2
    exact = delta == "exact" or (delta == "auto" and wl.Hq // wl.Hkv > 8)
    return 2 + bwd_launches(wl.S, grads, exact)


def roofline_of(wl, kern, peak_tf, peak_src, value):
    dom = max(kern.items(), key=lambda kv: kv[1]["avg_ms"])
    algo_flops = {"attn_fwd": wl.fwd_flops, "attn_bwd_main": wl.bwd_flops}
    if dom[0] not in algo_flops:
        return None
    achieved = algo_flops[dom[0]] / (dom[1]["avg_ms"] * 1e-3) / 1e12
    return {"bound": "tensor", "kernel": dom[0], "achieved": achieved, "peak": peak_tf,
            "unit": "TFLOP/s", "frac": achieved / peak_tf,
            "traffic": ncu_traffic(dom[0], wl.name),
            "peak_source": f"{peak_src} bf16 dense (burst)",
            "step_frac_of_peak": value / peak_tf}


def time_workload(M, wl, steps, warmup, flush, stream):
    """Device time of `steps` fwd(+bwd) steps of `wl` (inputs resident, L2 flushed between
    steps, CUDA events on the launching stream) and the per-kernel times of a second run
    of the same steps. Returns (ms per step, {kernel: {launches, avg_ms}})."""
    host = host_inputs(wl, 0)
    dev = {n: to_bf16_tensor(h, "cuda") for n, h in host.items()}
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["dout"]
    out = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.Hq, wl.S), dtype=torch.float32, device="cuda")
    dq = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(k.shape, dtype=torch.float32, device="cuda")
    dv = torch.empty(v.shape, dtype=torch.float32, device="cuda")
    dims = (wl.B, wl.Hq, wl.Hkv, wl.S, wl.D, wl.theta, wl.scale, wl.causal)

    def step():
        M.attn_fwd(q, k, v, out, lse, *dims, stream=stream)
        if wl.backward:
            M.attn_bwd(q, k, v, out, lse, do, dq, dk, dv, *dims, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if M.sync_status() != 0:
        raise SystemExit(f"device status error during warm-up ({wl.name})")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
    M.profile_begin(max(4096, 2 * steps))
    for i in range(steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    M.profile_end()
    kern = {}
    for kind, name in kernel_names(M):
        n, tot = M.profile_query(kind)
        if n:
            kern[name] = {"launches": n, "avg_ms": tot / n}
    if M.sync_status() != 0:
        raise SystemExit(f"device status error ({wl.name})")
    return ms, kern


def other_workload_lines(args, M, flush, stream, peak_tf, peak_src):
    """The other benchmark workloads (their shapes are in the workloads module), each
    with its own step time, per-kernel times, roofline fraction and oracle baseline."""
    lines = []
    for wl in WORKLOADS:
        if wl.name == args.workload:
            continue
        steps = max(3, min(args.steps, 10 if wl.S > 8192 else 20))
        ms, kern = time_workload(M, wl, steps, max(3, args.warmup), flush, stream)
        value = wl.flops / (ms * 1e-3) / 1e12
        entry = {"workload": wl.name, "config": config_of(wl, 1), "value": value,
                 "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
                 "kernels_ms": {n: round(d["avg_ms"], 5) for n, d in kern.items()},
                 "gpu_launches": launches_per_step(wl) * steps,
                 "roofline": roofline_of(wl, kern, peak_tf, peak_src, value),
                 "cpu_baseline": None}
        if not args.no_cpu_baseline:
            entry["cpu_baseline"] = cpu_baseline_of(wl, host_inputs(wl, 0), 4.0)
        lines.append(entry)
    return lines


def run_ours(args, rank, world, local):
    import mqa_attention_gb300 as M
    from mqa_attention_gb300 import build as B

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (GB300)")
    torch.cuda.set_device(local)
    if rank == 0 or not os.path.exists(B.LIB_PATH):
        B.build()
    barrier(world)
    M.lib()
    wl = by_name(args.workload)
    host = host_inputs(wl, rank)
    dev = {n: to_bf16_tensor(h, "cuda") for n, h in host.items()}
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["dout"]
    out = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.Hq, wl.S), dtype=torch.float32, device="cuda")
    gdt = torch.bfloat16 if args.grads == "bf16" else torch.float32
    dq = torch.empty(q.shape, dtype=gdt, device="cuda")
    dk = torch.empty(k.shape, dtype=gdt, device="cuda")
    dv = torch.empty(v.shape, dtype=gdt, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    dims = (wl.B, wl.Hq, wl.Hkv, wl.S, wl.D, wl.theta, wl.scale, wl.causal)
    mode = M.ROPE_MODES[args.rope] | (M.ROPE_EXACT if args.exact_rope else 0)
    bmode = mode | M.DELTA_MODES[args.delta]
    dims_ex = (wl.B, wl.Hq, wl.Hkv, wl.S, wl.D, wl.theta, mode, wl.scale, wl.causal)
    bdims_ex = (wl.B, wl.Hq, wl.Hkv, wl.S, wl.D, wl.theta, bmode, wl.scale, wl.causal)

    def fwd(q_, k_, v_, out_, lse_, st):
        if mode == 0:
            M.attn_fwd(q_, k_, v_, out_, lse_, *dims, stream=st)
        else:
            M.attn_fwd_ex(q_, k_, v_, out_, lse_, *dims_ex, stream=st)

    def bwd(q_, k_, v_, out_, lse_, do_, dq_, dk_, dv_, st):
        if args.grads == "bf16":
            M.attn_bwd_bf16(q_, k_, v_, out_, lse_, do_, dq_, dk_, dv_, *bdims_ex, stream=st)
        elif bmode == 0:
            M.attn_bwd(q_, k_, v_, out_, lse_, do_, dq_, dk_, dv_, *dims, stream=st)
        else:
            M.attn_bwd_ex(q_, k_, v_, out_, lse_, do_, dq_, dk_, dv_, *bdims_ex, stream=st)

    def step():
        fwd(q, k, v, out, lse, stream)
        if wl.backward:
            bwd(q, k, v, out, lse, do, dq, dk, dv, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if M.sync_status() != 0:
        raise SystemExit("device status error during warm-up")

    sampler = ClockSampler(local)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()  # L2 flush between steps (outside the events)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms_local, world)
    # Per-kernel durations: the library's events around each launch, over a second
    # run of the same steps (an event between two launches would hold back the
    # programmatic early start of the second, so the timed run above records none).
    M.profile_begin(max(4096, 2 * args.steps))
    for i in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    M.profile_end()
    status = M.sync_status()
    kern = {}
    for kind, name in kernel_names(M):
        n, tot = M.profile_query(kind)
        if n:
            kern[name] = {"launches": n, "avg_ms": tot / n}

    # ---- end to end through host buffers
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 50))
    hp = {n: to_bf16_tensor(h, pin=True) for n, h in host.items()}
    ho = {"out": torch.empty(out.shape, dtype=torch.bfloat16).pin_memory(),
          "lse": torch.empty(lse.shape, dtype=torch.float32).pin_memory()}
    if wl.backward:
        for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            ho[n] = torch.empty(t.shape, dtype=gdt).pin_memory()
    h2d = sum(t.numel() * t.element_size() for n, t in hp.items()
              if wl.backward or n != "dout")
    d2h = sum(t.numel() * t.element_size() for t in ho.values())

    # Steps stream through three device buffer sets: while step i computes, the
    # inputs of step i+1 go host -> device on one copy stream and the results of
    # earlier steps device -> host on another (the device -> host copies, larger than
    # one step's compute, get two steps of slack). Every step's copies lie inside the
    # timed region; events order the reuse of each buffer set.
    NB = 3
    names_in = [n for n in ("q", "k", "v", "dout") if wl.backward or n != "dout"]
    bufs = [dict(q=q, k=k, v=v, dout=do, out=out, lse=lse, dq=dq, dk=dk, dv=dv)]
    for _ in range(NB - 1):
        bufs.append({n: torch.empty_like(t) for n, t in bufs[0].items()})
    s_in = torch.cuda.Stream()
    s_out = torch.cuda.Stream()
    ev = {key: [torch.cuda.Event() for _ in range(NB)] for key in ("in", "comp", "out")}
    used = [False] * NB

    def e2e_step(i):
        b = i % NB
        d = bufs[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev["comp"][b])  # step i-NB has read these inputs
            for n in names_in:
                d[n].copy_(hp[n], non_blocking=True)
            ev["in"][b].record(s_in)
        stream.wait_event(ev["in"][b])
        if used[b]:
            stream.wait_event(ev["out"][b])  # step i-NB's results have left the device
        fwd(d["q"], d["k"], d["v"], d["out"], d["lse"], stream)
        if wl.backward:
            bwd(d["q"], d["k"], d["v"], d["out"], d["lse"], d["dout"], d["dq"], d["dk"], d["dv"],
                stream)
        ev["comp"][b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            for n in ho:
                ho[n].copy_(d[n], non_blocking=True)
            ev["out"][b].record(s_out)
        used[b] = True

    for i in range(NB):
        e2e_step(i)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    if rank != 0:
        return
    peak_tf, peak_hbm, peak_src = peaks()
    total_flops = wl.flops * world
    value = total_flops / (ms * 1e-3) / 1e12
    # dominant kernel: the one with the largest share of the step
    roof = roofline_of(wl, kern, peak_tf, peak_src, value / world)
    # the backward prologue (abs-max pass + row pass) is HBM-bound: its algorithmic bytes
    # against the measured copy bandwidth
    prologue = None
    if "bwd_prep" in kern:
        nbytes = bwd_prologue_bytes(wl)
        gbs = nbytes / (kern["bwd_prep"]["avg_ms"] * 1e-3) / 1e9
        prologue = {"kernel": "bwd_prep (abs-max pass + row pass)", "bound": "hbm",
                    "bytes": nbytes, "achieved": gbs, "peak": peak_hbm, "unit": "GB/s",
                    "frac": gbs / peak_hbm,
                    "reads": "abs-max: q, k, v, dO; row pass: q, k, v, dO, out, lse",
                    "writes": "fp16 q~, k~, v, dO; zeroed fp32 dQ accumulator; delta; lse*log2e"}
    passes = {}
    if "attn_fwd" in kern:
        passes["fwd"] = kern["attn_fwd"]["avg_ms"] + kern.get("rope", {"avg_ms": 0.0})["avg_ms"]
    if "attn_bwd_main" in kern:
        passes["bwd"] = sum(kern[k]["avg_ms"] for k in ("bwd_prep", "delta", "attn_bwd_main",
                                                        "dq_finalize") if k in kern)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline_of(wl, host, 10.0)
    others = None
    if (world == 1 and args.rope == "half" and args.grads == "fp32" and args.delta == "auto"
            and not args.exact_rope and not args.single):
        others = other_workload_lines(args, M, flush, stream, peak_tf, peak_src)
    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic N(0,1) bf16 q/k/v/dO, seeded (splitmix64 + Box-Muller)",
        "config": config_of(wl, world, rope=args.rope, grads=args.grads, delta=args.delta,
                            exact_rope=args.exact_rope),
        "e2e": {"value": total_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "pinned host buffers; each step's inputs in and results out on two "
                          "copy streams over three device buffer sets, overlapped with "
                          "the neighbouring steps' compute"},
        "gpu_launches": launches_per_step(wl, args.delta, args.grads) * args.steps,
        "roofline": roof,
        "prologue_roofline": prologue,
        "passes_ms": {k: round(v, 5) for k, v in passes.items()},
        "kernels_ms": {n: round(d["avg_ms"], 5) for n, d in kern.items()},
        "cpu_baseline": cpu,
        "clocks": clocks,
        "device_status": status,
        "other_workloads": others,
    }
    print(json.dumps(line), flush=True)


def run_blocks(args, rank, world, local):
    """The step as a context-parallel block schedule on one GPU: the sequence is cut
    into N query and N key/value blocks; each query block's partial forwards over
    the key blocks it can see are merged in place, then every such block pair runs
    its partial backward. Credited the same causal-pair FLOPs as the full step;
    device time only (each block's outputs stay on the device)."""
    import mqa_attention_gb300 as M
    from mqa_attention_gb300 import build as B

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (GB300)")
    torch.cuda.set_device(local)
    if rank == 0 or not os.path.exists(B.LIB_PATH):
        B.build()
    barrier(world)
    M.lib()
    wl = by_name(args.workload)
    nb = args.blocks
    if wl.S % (nb * 128) or not wl.backward:
        raise SystemExit("--blocks needs a fwd+bwd workload whose S is a multiple of 128 * N")
    blk = wl.S // nb
    host = host_inputs(wl, rank)
    dev = {n: to_bf16_tensor(h, "cuda") for n, h in host.items()}
    cut = lambda t, i: t[:, :, i * blk:(i + 1) * blk].contiguous()
    qb = [cut(dev["q"], i) for i in range(nb)]
    kb = [cut(dev["k"], i) for i in range(nb)]
    vb = [cut(dev["v"], i) for i in range(nb)]
    dob = [cut(dev["dout"], i) for i in range(nb)]
    pairs = [(i, j) for i in range(nb) for j in range(nb) if not wl.causal or j <= i]
    outs = [torch.empty_like(qb[i]) for i in range(nb)]
    lses = [torch.empty((wl.B, wl.Hq, blk), dtype=torch.float32, device="cuda") for _ in range(nb)]
    po, pl = torch.empty_like(qb[0]), torch.empty_like(lses[0])
    grads = {p: (torch.empty(qb[0].shape, dtype=torch.float32, device="cuda"),
                 torch.empty(kb[0].shape, dtype=torch.float32, device="cuda"),
                 torch.empty(kb[0].shape, dtype=torch.float32, device="cuda")) for p in pairs}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    mode = M.ROPE_MODES[args.rope]
    D = wl.D

    def step():
        for i in range(nb):
            first = True
            for (a, j) in pairs:
                if a != i:
                    continue
                o, l = (outs[i], lses[i]) if first else (po, pl)
                M.attn_fwd_partial(qb[i], kb[j], vb[j], o, l, wl.B, wl.Hq, wl.Hkv, blk, blk, D,
                                   i * blk, j * blk, wl.theta, mode, wl.scale, wl.causal, stream)
                if not first:
                    M.attn_merge(outs[i], lses[i], po, pl, outs[i], lses[i], lses[i].numel(), D,
                                 stream)
                first = False
        for (i, j) in pairs:
            g = grads[(i, j)]
            M.attn_bwd_partial(qb[i], kb[j], vb[j], outs[i], lses[i], dob[i], g[0], g[1], g[2],
                               wl.B, wl.Hq, wl.Hkv, blk, blk, D, i * blk, j * blk, wl.theta,
                               mode, wl.scale, wl.causal, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if M.sync_status() != 0:
        raise SystemExit("device status error during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps, world)
    M.profile_begin(max(4096, 16 * len(pairs) * args.steps))  # per-kernel times: a second run
    for i in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    M.profile_end()
    status = M.sync_status()
    kern = {}
    for kind, name in kernel_names(M):
        n, tot = M.profile_query(kind)
        if n:
            kern[name] = tot / args.steps  # ms per step over all blocks
    sampler.stop()
    if rank != 0:
        return
    peak_tf, _, peak_src = peaks()
    value = wl.flops * world / (ms * 1e-3) / 1e12
    achieved = wl.bwd_flops / (kern["attn_bwd_main"] * 1e-3) / 1e12
    nfwd = sum(1 for _ in pairs)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic N(0,1) bf16 q/k/v/dO, seeded (splitmix64 + Box-Muller)",
        "config": dict(config_of(wl, world, rope=args.rope), blocks=f"{nb} x {nb}", block_rows=blk,
                       block_pairs=len(pairs)),
        "e2e": None,
        "note": "block schedule through the partial entry points; device time only",
        # per pair: RoPE pre-pass + forward (+ merge), and a backward call
        "gpu_launches": (2 * nfwd + (nfwd - nb) + bwd_launches(blk) * nfwd) * args.steps,
        "roofline": {"bound": "tensor", "kernel": "attn_bwd_main", "achieved": achieved,
                     "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved / peak_tf,
                     "traffic": None, "peak_source": f"{peak_src} bf16 dense (burst)"},
        "kernels_ms": {n: round(v, 5) for n, v in kern.items()},
        "cpu_baseline": None,
        "clocks": sampler.summary(t0, t1),
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def run_decode(args, rank, world, local):
    """Decode shape: SQ new query rows per head (at the cache's last SQ positions)
    against a rotated key / value cache of the workload's S rows. The work is one
    read of the cache, so the metric is bytes moved (caches, q, out, lse) per second
    against the measured HBM copy bandwidth. Device time only."""
    import mqa_attention_gb300 as M
    from mqa_attention_gb300 import build as B

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (GB300)")
    torch.cuda.set_device(local)
    if rank == 0 or not os.path.exists(B.LIB_PATH):
        B.build()
    barrier(world)
    M.lib()
    wl = by_name(args.workload)
    sq = args.decode
    host = host_inputs(wl, rank)
    dev = {n: to_bf16_tensor(h, "cuda") for n, h in host.items()}
    q = dev["q"][:, :, :sq].contiguous()
    mode = M.ROPE_MODES[args.rope]
    cache = 2 * wl.B * wl.Hkv * wl.S * wl.D * 2
    # Enough copies of the cache (>= 256 MiB in all) that each call reads its own
    # copy cold from HBM; one graph launches one call per copy.
    ncopy = max(1, -(-L2_FLUSH_BYTES // cache))
    k_rot = M.rope(dev["k"], wl.theta, rope=args.rope)
    caches = [(k_rot, dev["v"])] + [(k_rot.clone(), dev["v"].clone()) for _ in range(ncopy - 1)]
    out = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.Hq, sq), dtype=torch.float32, device="cuda")
    qpos = wl.S - sq

    def calls(st):
        for kc, vc in caches:
            M.attn_decode(q, kc, vc, out, lse, wl.B, wl.Hq, wl.Hkv, sq, wl.S, wl.D, qpos,
                          wl.theta, mode, wl.scale, st)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(max(3, args.warmup)):
            calls(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    if M.sync_status() != 0:
        raise SystemExit("device status error during warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls(torch.cuda.current_stream())
    stream = torch.cuda.current_stream()
    graph.replay()
    torch.cuda.synchronize()
    # A replay lasts microseconds: replay enough (>= 0.5 s) that the clock sampler
    # sees the timed region.
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(10):
        graph.replay()
    p1.record(stream)
    torch.cuda.synchronize()
    per_replay_s = p0.elapsed_time(p1) / 10 * 1e-3
    reps = max(1, args.steps // ncopy, int(0.5 / max(per_replay_s, 1e-9)) + 1)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    status = M.sync_status()
    ms = max_over_ranks(e0.elapsed_time(e1) / (reps * ncopy), world)
    sampler.stop()
    # End to end: each call takes its new query rows from pinned host memory and
    # returns out and lse to it (the cache stays resident, as in serving).
    hq = q.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    n_e2e = 200
    for i in range(n_e2e + 10):
        if i == 10:
            torch.cuda.synchronize()
            e0.record(stream)
        kc, vc = caches[i % ncopy]
        q.copy_(hq, non_blocking=True)
        M.attn_decode(q, kc, vc, out, lse, wl.B, wl.Hq, wl.Hkv, sq, wl.S, wl.D, qpos, wl.theta,
                      mode, wl.scale, stream)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world)
    if rank != 0:
        return
    _, peak_hbm, peak_src = peaks()
    moved = cache + 2 * q.numel() * 2 + lse.numel() * 4
    gbs = moved * world / (ms * 1e-3) / 1e9
    line = {
        "metric": f"decode attention GB/s ({sq} new tokens per sequence, cache S={wl.S})",
        "value": gbs, "unit": "GB/s", "n_gpus": world,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic N(0,1) bf16 q/k/v, seeded (splitmix64 + Box-Muller)",
        "config": dict(config_of(wl, world, rope=args.rope,
                                 l2=f"each call reads its own cache copy ({ncopy} copies, "
                                    ">= 256 MiB)"),
                       passes="decode fwd", new_tokens=sq, bytes_per_step=moved),
        "e2e": {"value": moved * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": out.numel() * 2 + lse.numel() * 4,
                "copies": "pinned host q in, out and lse out, every call; calls issued "
                          "one after another on the stream (no graph)"},
        "note": "value: decode entry point replayed from a CUDA graph, device time",
        "steps": reps * ncopy,
        "gpu_launches": 2 * reps * ncopy,  # chunk kernel and merge per call
        "roofline": {"bound": "hbm", "kernel": "attn_decode", "achieved": gbs / world,
                     "peak": peak_hbm, "unit": "GB/s", "frac": gbs / world / peak_hbm,
                     # the committed ncu record is for one new token per sequence
                     "traffic": ncu_traffic("attn_decode", wl.name) if sq == 1 else None,
                     "peak_source": f"{peak_src} HBM copy"},
        "cpu_baseline": None,
        "clocks": sampler.summary(t0, t1),
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.decode > 0:
        run_decode(args, rank, world, local)
    elif args.blocks > 1:
        run_blocks(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
