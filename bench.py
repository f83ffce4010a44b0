#!/usr/bin/env python3
"""Benchmark: causal RoPE attention forward on GB300 through libattnfuse.

Default: the Llama-3-8B attention shape (B=1, Hq=32, Hkv=8, N=4096, d=128, bf16, rope base 5e5),
fused mode, one step = one attnfuse_rope_causal_fwd call.  Prints ONE JSON line (rank 0):
value = causal TFLOP/s (2*B*Hq*N^2*d per step) over all ranks, plus roofline, e2e (host buffers,
copies inside the timed region), the pre-rotate path (RoPE pass GB/s and pipeline TFLOP/s), clocks
sampled during the timed region and the CPU oracle's throughput on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
  python bench.py --sweep      # crossover sweep: fused vs pre-rotate at every N, then N* per family

Timing: inputs resident in HBM; W untimed warm-up steps; K timed steps, each bracketed by CUDA
events on the launching stream; a 512 MiB write flushes L2 (129 MB) before every step, outside the
events; barrier + synchronize on both sides; max over ranks.  Multi-GPU runs are replicas (the
forward pass needs no collective): every rank runs the full workload on its own GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RoPE+causal attn fwd TFLOP/s and % of GB300 bf16 peak; fused vs pre-rotate N*"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 512 * 1024 * 1024
_CSRC = "attention_rope_causal_gb300/csrc/"
# The sources each profiled kernel is compiled from (the kernel code; not the host-side launch code).
KERNEL_SOURCES = {
    "attn_fwd": tuple(_CSRC + f for f in ("attn_fwd.cu", "ptx.cuh", "rope.cuh")),
    "rope_apply": tuple(_CSRC + f for f in ("rope_apply.cu", "rope.cuh")),
    "attn_bwd": tuple(_CSRC + f for f in ("attn_bwd.cu", "ptx.cuh", "rope.cuh")),
}
TRAFFIC_KINDS = {"attn_fwd_fused": "attn_fwd", "attn_fwd_plain": "attn_fwd", "attn_fwd_split": "attn_fwd",
                 "rope_apply_qk": "rope_apply", "bwd_dkdv": "attn_bwd", "bwd_dq": "attn_bwd"}


# ----------------------------------------------------------------------------------------------
# host-side helpers (no GPU needed; unit-tested on CPU)


def load_peaks(path=None):
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def kernel_source_hash(group: str = "attn_fwd") -> str:
    """Hash of the sources one kernel group is compiled from (`KERNEL_SOURCES`)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[group]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kind: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None if absent or taken on other code."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kind][workload]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_hash") != kernel_source_hash(TRAFFIC_KINDS.get(kind, "attn_fwd")):
        return None
    return float(rec["dram_bytes_per_launch"])


def aggregate(units_per_rank_step: float, steps: int, n_ranks: int, max_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed, over the slowest rank's time."""
    return units_per_rank_step * steps * n_ranks / max_seconds


def crossover(ns, t_fused, t_pre):
    """N* where fused and pre-rotate times cross: linear interpolation in N of log(t_fused/t_pre)
    between the two bracketing sweep points.  Returns (n_star or None, description)."""
    import math
    r = [math.log(a / b) for a, b in zip(t_fused, t_pre)]
    for i in range(len(ns) - 1):
        if r[i] == 0.0:
            return float(ns[i]), "equal at a sweep point"
        if (r[i] < 0) != (r[i + 1] < 0):
            n = ns[i] + (ns[i + 1] - ns[i]) * (0.0 - r[i]) / (r[i + 1] - r[i])
            who = "fused faster below N*" if r[i] < 0 else "pre-rotate faster below N*"
            return n, who
    if all(x < 0 for x in r):
        return None, f"fused faster at every N in [{ns[0]}, {ns[-1]}]"
    return None, f"pre-rotate faster at every N in [{ns[0]}, {ns[-1]}]"


def parse_clocks(csv_text: str, t0: float, t1: float):
    """Median SM clock and throttle reasons from nvidia-smi CSV samples taken in [t0, t1] (epoch s)."""
    import datetime
    mhz, maxmhz, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in csv_text.strip().splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10 or parts[0].startswith("timestamp"):
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            continue
        if not (t0 - 0.25 <= ts <= t1 + 0.25):
            continue
        try:
            mhz.append(float(parts[2].split()[0]))
            maxmhz = float(parts[3].split()[0])
        except (ValueError, IndexError):
            continue
        for name, val in zip(names, parts[6:10]):
            if val.lower() == "active":
                reasons.add(name)
    if not mhz:
        return None
    return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": maxmhz, "samples": len(mhz), "reasons": sorted(reasons)}


class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader", "-lms", "100"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as f:
            text = f.read()
        os.unlink(self.file.name)
        return parse_clocks(text, t0, t1)


# ----------------------------------------------------------------------------------------------
# distributed plumbing (replicas; the only collectives are the timing barrier and max)


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------------------
# the CPU oracle as a baseline (bounded row samples of the same workload)


def oracle_rows_flops(w, rows):
    return float(sum(4 * w.d * (int(i) + 1) for i in rows)) * w.Hq * w.B


def oracle_sample_rows(w, target_s: float, q, k, v):
    """Pick an evenly strided row sample whose oracle run takes about target_s on this host."""
    import numpy as np
    import oracle
    probe = np.arange(0, w.N, max(1, w.N // 32))
    t = time.perf_counter()
    oracle.rope_causal(q, k, v, w.rope_base, rows=probe)
    dt = max(time.perf_counter() - t, 1e-3)
    rate = oracle_rows_flops(w, probe) / dt
    want = target_s * rate
    stride = max(1, int(round(oracle_rows_flops(w, np.arange(w.N)) / max(want, 1.0))))
    return stride


def rows_phrase(stride: int) -> str:
    """'every query row' or 'one query row in <stride>'."""
    return "every query row" if stride == 1 else f"one query row in {stride}"


def run_cpu_baseline(w, target_s=12.0):
    import numpy as np
    import oracle
    from attention_rope_causal_gb300 import inputs
    q, k, v = inputs.make_inputs(w)
    stride = oracle_sample_rows(w, target_s, q, k, v)
    rows = np.arange(0, w.N, stride)
    t = time.perf_counter()
    oracle.rope_causal(q, k, v, w.rope_base, rows=rows)
    dt = time.perf_counter() - t
    fl = oracle_rows_flops(w, rows)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.default_threads(), "kind": "oracle",
            "sample": f"{w.name}: {rows_phrase(stride)} ({len(rows)} rows x {w.Hq} heads), fp64 C oracle, "
                      f"{dt:.1f} s, {fl / 1e9:.1f} GFLOP causal-equivalent"}


def run_reference_arm(args):
    """The reference arm of this benchmark is the CPU oracle, timed as it stands on this host."""
    import numpy as np
    import oracle
    from attention_rope_causal_gb300 import inputs
    rank, world, _ = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0
    if rank != 0:
        return 0
    w = inputs.NAMED[args.workload]
    q, k, v = inputs.make_inputs(w)
    budget = 150.0 / max(1, args.steps + args.warmup)  # seconds per step: the whole run in a few minutes
    stride = oracle_sample_rows(w, budget, q, k, v)
    fl_total, t_total = 0.0, 0.0
    for s in range(args.warmup + args.steps):
        rows = np.arange(s % stride, w.N, stride)
        t = time.perf_counter()
        oracle.rope_causal(q, k, v, w.rope_base, rows=rows)
        dt = time.perf_counter() - t
        if s >= args.warmup:
            fl_total += oracle_rows_flops(w, rows)
            t_total += dt
    value = fl_total / t_total / 1e12
    sample = (f"{w.name}: each step {rows_phrase(stride)} (offset rotating) x {w.Hq} heads, fp64 C oracle "
              f"on {oracle.default_threads()} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_total / max(1, args.steps) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                       "rope_base": w.rope_base},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.default_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------------------
# GPU timing


WARMUP_MIN_S = 0.05   # warm-up runs at least this long, whatever --warmup says
SLEEP_HZ = 2.07e9     # SM cycles per second at the maximum clock (a slower clock only lengthens a sleep)
CHUNK = 64            # steps enqueued behind one sleep


def time_steps(fn, steps, flush, stream, clean_l2=False):
    """Per-step CUDA-event times (ms) of fn() with an L2 flush before each step, outside the events.

    The flush writes a 512 MiB buffer (L2 then holds dirty lines of it); with clean_l2 it is read
    back as well (clean lines).  The GPU is kept behind the host: each chunk of steps is enqueued
    behind a spin (torch.cuda._sleep) longer than the host takes to enqueue the chunk, so no step
    ever waits for the host and host-side overhead cannot enter the measured times."""
    import torch
    times = []
    host_per_step = 3e-4  # s; measured on every chunk afterwards
    scratch = torch.empty(1, dtype=torch.float32, device=flush.device) if clean_l2 else None
    with torch.cuda.stream(stream):
        done = 0
        while done < steps:
            n = min(CHUNK, steps - done)
            torch.cuda._sleep(int((1.5 * host_per_step * n + 2e-4) * SLEEP_HZ))
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            t = time.perf_counter()
            for a, b in evs:
                flush.zero_()
                if clean_l2:
                    torch.sum(flush, dim=0, out=scratch.view(()))
                a.record(stream)
                fn()
                b.record(stream)
            host_per_step = max(host_per_step, (time.perf_counter() - t) / n)
            stream.synchronize()
            times += [a.elapsed_time(b) for a, b in evs]
            done += n
    return times


def run_warmup(run_batch, steps, min_s=WARMUP_MIN_S, clock=time.perf_counter):
    """Calls run_batch(n) until at least `steps` steps have run and at least min_s seconds have
    passed (the page-4 protocol's >= 50 ms warm-up, whatever the step count says); returns
    (steps run, seconds)."""
    t0 = clock()
    n = 0
    while n < steps or clock() - t0 < min_s:
        batch = max(1, steps - n) if n < steps else 8
        run_batch(batch)
        n += batch
    return n, clock() - t0


def warm_up(fn, steps, flush, stream):
    """Untimed steps of fn (with the flush, as timed) under run_warmup's rule."""
    import torch
    torch.cuda.synchronize()
    return run_warmup(lambda n: time_steps(fn, n, flush, stream), steps)


def e2e_pipelined(w, q0, k0, v0, steps, warmup, nb=2):
    """End to end through the C ABI with host inputs and outputs: every step copies its q, k, v from
    pinned host memory to the device, runs the fused forward, and copies out and lse back to pinned
    host memory.  Steps are pipelined over two device buffer sets on three streams (H2D, compute,
    D2H), so one step's copies overlap its neighbours' compute; the time is that of the whole
    sequence (first H2D to last D2H).  Returns (ms per step, h2d bytes, d2h bytes)."""
    import torch
    from attention_rope_causal_gb300 import binding
    qh, kh, vh = (t.cpu().pin_memory() for t in (q0, k0, v0))
    lse_shape = (w.B, w.Hq, w.N)
    dev = [dict(q=torch.empty_like(q0), k=torch.empty_like(k0), v=torch.empty_like(v0), out=torch.empty_like(q0),
                lse=torch.empty(lse_shape, dtype=torch.float32, device="cuda")) for _ in range(nb)]
    host = [(torch.empty(q0.shape, dtype=q0.dtype, pin_memory=True),
             torch.empty(lse_shape, dtype=torch.float32, pin_memory=True)) for _ in range(nb)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(nb)]
    cmp_done = [torch.cuda.Event() for _ in range(nb)]
    out_done = [torch.cuda.Event() for _ in range(nb)]

    def run(n):
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        for i in range(n):
            b, d = i % nb, dev[i % nb]
            if i >= nb:
                s_in.wait_event(cmp_done[b])  # the compute of step i - nb has read this buffer set
            with torch.cuda.stream(s_in):
                d["q"].copy_(qh, non_blocking=True)
                d["k"].copy_(kh, non_blocking=True)
                d["v"].copy_(vh, non_blocking=True)
            in_done[b].record(s_in)
            s_cmp.wait_event(in_done[b])
            if i >= nb:
                s_cmp.wait_event(out_done[b])  # the D2H of step i - nb has read out / lse
            binding.rope_causal_fwd(d["q"], d["k"], d["v"], w.rope_base, mode="fused", out=d["out"], lse=d["lse"],
                                    stream=s_cmp)
            cmp_done[b].record(s_cmp)
            s_out.wait_event(cmp_done[b])
            with torch.cuda.stream(s_out):
                host[b][0].copy_(d["out"], non_blocking=True)
                host[b][1].copy_(d["lse"], non_blocking=True)
            out_done[b].record(s_out)
        end.record(s_out)  # after the last D2H, which follows every earlier operation
        end.synchronize()
        return start.elapsed_time(end)

    run(warmup)
    ms = run(steps) / steps
    h2d = sum(t.numel() * t.element_size() for t in (q0, k0, v0))
    d2h = q0.numel() * q0.element_size() + w.B * w.Hq * w.N * 4
    return ms, h2d, d2h


def gpu_setup(w, modes):
    import torch
    from attention_rope_causal_gb300 import binding, inputs
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")
    ws = {m: torch.empty(max(256, binding.workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d, m, q.dtype)),
                         dtype=torch.uint8, device="cuda") for m in modes}
    return q, k, v, out, lse, ws


def fwd_fn(w, q, k, v, out, lse, ws, mode, stream):
    from attention_rope_causal_gb300 import binding
    return lambda: binding.rope_causal_fwd(q, k, v, w.rope_base, mode=mode, out=out, lse=lse, workspace=ws,
                                           stream=stream)


def rope_pass_fn(w, stream):
    """The RoPE pass of the pre-rotate path as one launch over Q and K: attnfuse_rope_apply on a
    [B, N, Hq + Hkv, d] tensor moves the same bytes as the pipeline's combined Q/K launch."""
    import torch
    from attention_rope_causal_gb300 import binding
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    x = torch.randn((w.B, w.N, w.Hq + w.Hkv, w.d), generator=g).to(w.torch_dtype).cuda()
    y = torch.empty_like(x)
    return lambda: binding.rope_apply(x, w.rope_base, out=y, stream=stream)


def plain_fn(w, q, k, v, out, lse, stream):
    """The plain attention kernel alone (mode "none") on Q and K rotated once beforehand: the second
    stage of the pre-rotate pipeline, timed without the RoPE pass."""
    from attention_rope_causal_gb300 import binding
    qr, kr = binding.rope_apply(q, w.rope_base), binding.rope_apply(k, w.rope_base)
    return lambda: binding.rope_causal_fwd(qr, kr, v, w.rope_base, mode="none", out=out, lse=lse, stream=stream)


def measure_point(w, steps, warmup):
    """Median-of-steps times (ms) for fused, the pre-rotate and split pipelines, the plain attention
    kernel alone (mode none) and the RoPE pass alone."""
    import torch
    from attention_rope_causal_gb300 import binding
    stream = torch.cuda.current_stream()
    q, k, v, out, lse, ws = gpu_setup(w, ("fused", "prerotate", "split"))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    fns = {mode: fwd_fn(w, q, k, v, out, lse, ws[mode], mode, stream) for mode in ("fused", "prerotate", "split")}
    fns["plain"] = plain_fn(w, q, k, v, out, lse, stream)
    fns["rope"] = rope_pass_fn(w, stream)
    res = {}
    for name, f in fns.items():
        warm_up(f, warmup, flush, stream)
        res[name] = statistics.median(time_steps(f, steps, flush, stream))
    if binding.device_status() != 0:
        raise RuntimeError(f"device status: {binding.last_error()}")
    return res


def rope_bytes(w) -> float:
    """Algorithmic bytes of the pre-rotation pass: Q and K read and written once (16-bit elements)."""
    return 2.0 * w.B * w.N * (w.Hq + w.Hkv) * w.d * 2


def rotation_calculus(points, peak_tflops, hbm_gbs):
    """The crossover model of the AttnFuse report (paragraph 3: pre-rotation costs memory bandwidth,
    in-kernel rotation costs compute) set beside the measured crossover, for one family and dtype.

    points: dicts with N, B, Hq, Hkv, d and the measured ms of fused, prerotate, plain and rope.
    Per point: alpha = T_fused / T_plain - 1 (in-kernel rotation as a fraction of attention time),
    rho = (T_prerotate - T_plain) / T_plain (what the pass adds to the pipeline, relative) and
    rope_frac = T_rope / T_plain (the pass timed alone).
    Model: T_fused = (1 + a) T_attn(N) and T_pre = T_attn(N) + bytes(N) / BW, with T_attn(N) =
    flops(N) / (eta P), a = median alpha and eta = median plain-kernel efficiency over the points.
    At fixed tokens B N (the sweep's 16384) flops grow as N and bytes do not, so the two meet at
        N* = 2 (Hq + Hkv) eta P / (a Hq BW)
    -- with BW the measured HBM copy bandwidth ("peak" model) and with the RoPE pass's own measured
    GB/s ("calibrated" model).  The measured N* interpolates log(T_fused / T_pre) between points."""
    pts = sorted(points, key=lambda r: r["N"])
    rows = []
    for r in pts:
        flops = 2.0 * r["B"] * r["Hq"] * r["N"] ** 2 * r["d"]
        rows.append(dict(N=r["N"], alpha=r["fused_ms"] / r["plain_ms"] - 1.0,
                         rho=(r["prerotate_ms"] - r["plain_ms"]) / r["plain_ms"],
                         rope_frac=r["rope_ms"] / r["plain_ms"],
                         eta=flops / (r["plain_ms"] * 1e-3) / (peak_tflops * 1e12),
                         rope_gbs=2.0 * r["B"] * r["N"] * (r["Hq"] + r["Hkv"]) * r["d"] * 2 / (r["rope_ms"] * 1e-3) / 1e9))
    a = statistics.median(x["alpha"] for x in rows)
    eta = statistics.median(x["eta"] for x in rows)
    bw_rope = statistics.median(x["rope_gbs"] for x in rows)
    Hq, Hkv = pts[0]["Hq"], pts[0]["Hkv"]
    P = peak_tflops * 1e12

    def n_star(bw_gbs):
        return 2.0 * (Hq + Hkv) * eta * P / (a * Hq * bw_gbs * 1e9) if a > 0 else None

    measured, how = crossover([r["N"] for r in pts], [r["fused_ms"] for r in pts], [r["prerotate_ms"] for r in pts])
    return {"points": rows, "alpha_median": a, "eta_plain_median": eta, "rope_gbs_median": bw_rope,
            "model_n_star_peak_bw": n_star(hbm_gbs), "model_n_star_measured_rope_bw": n_star(bw_rope),
            "measured_n_star": measured, "measured_note": how}


def run_sweep(args):
    from attention_rope_causal_gb300 import inputs
    peaks = load_peaks()
    rows = []
    for w in inputs.sweep_workloads(extra=True):
        t = measure_point(w, args.steps, args.warmup)
        fl = w.causal_flops
        rec = {"workload": w.name, "N": w.N, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "dtype": w.dtype,
               "fused_ms": t["fused"], "prerotate_ms": t["prerotate"], "split_ms": t["split"],
               "plain_ms": t["plain"], "rope_ms": t["rope"],
               "fused_tflops": fl / t["fused"] / 1e9, "prerotate_tflops": fl / t["prerotate"] / 1e9,
               "split_tflops": fl / t["split"] / 1e9, "plain_tflops": fl / t["plain"] / 1e9,
               "rope_gbs": rope_bytes(w) / t["rope"] / 1e6,
               "alpha": t["fused"] / t["plain"] - 1.0, "rope_over_plain": t["rope"] / t["plain"],
               "fused_over_prerotate": t["fused"] / t["prerotate"],
               "fastest": min(("fused", "prerotate", "split"), key=lambda m: t[m])}
        rows.append(rec)
        print(json.dumps(rec), flush=True)
    summary = {}
    for fam in ("gqa", "mha"):
        for dt in ("bf16", "fp16"):
            pts = [r for r in rows if r["workload"].startswith(f"sweep_{fam}_") and r["dtype"] == dt]
            summary[f"{fam}_{dt}"] = rotation_calculus(pts, peaks["bf16_tflops"], peaks["hbm_gbs"])
    print(json.dumps({"sweep_summary": summary, "peaks": peaks}), flush=True)
    return 0


def bwd_fn(w, q, k, v, out, lse, stream):
    """One backward step (attnfuse_rope_causal_bwd) on the forward's out / lse with a fixed dout and
    preallocated gradients and workspace."""
    import torch
    from attention_rope_causal_gb300 import binding
    g = torch.Generator(device="cpu").manual_seed(w.seed + 1000)
    dout = torch.randn(q.shape, generator=g).to(q.dtype).cuda()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d, q.dtype), dtype=torch.uint8,
                     device="cuda")
    return lambda: binding.rope_causal_bwd(q, k, v, out, lse, dout, w.rope_base, dq=dq, dk=dk, dv=dv, workspace=ws,
                                           stream=stream)


def decode_fn(w, mode, stream):
    """One decode step of the workload's heads: B queries (N = 1), each against w.N cached keys,
    through attnfuse_rope_causal_fwd_ex in `mode` ("fused" runs the split-KV decode kernels)."""
    import torch
    from attention_rope_causal_gb300 import binding, inputs
    q, k, v = (t.cuda() for t in inputs.make_kv_inputs(w.B, 1, w.N, w.Hq, w.Hkv, w.d, w.dtype, seed=w.seed + 7))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(256, binding.workspace_bytes(w.B, w.Hq, w.Hkv, 1, w.d, mode, q.dtype, kv_len=w.N)),
                     dtype=torch.uint8, device="cuda")
    return lambda: binding.rope_causal_fwd(q, k, v, w.rope_base, mode=mode, out=out, lse=lse, workspace=ws,
                                           stream=stream)


def run_only(args):
    """Run one path alone (for profilers): W + K steps of `fused`, `prerotate` or `rope` with L2 flushes."""
    import torch
    from attention_rope_causal_gb300 import binding, build, inputs
    build.build()
    binding.load()
    torch.cuda.set_device(0)
    w = inputs.NAMED[args.workload]
    stream = torch.cuda.current_stream()
    q, k, v, out, lse, ws = gpu_setup(w, ("fused", "prerotate", "split"))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    if args.only == "rope":
        f = rope_pass_fn(w, stream)
    elif args.only == "backward":
        fwd_fn(w, q, k, v, out, lse, ws["fused"], "fused", stream)()
        f = bwd_fn(w, q, k, v, out, lse, stream)
    elif args.only == "decode":
        f = decode_fn(w, "fused", stream)
    elif args.only != "plain":
        f = fwd_fn(w, q, k, v, out, lse, ws[args.only], args.only, stream)
    if args.only == "plain":
        f = plain_fn(w, q, k, v, out, lse, stream)
    warm_up(f, args.warmup, flush, stream)
    ms = time_steps(f, args.steps, flush, stream)
    st = binding.device_status()
    print(json.dumps({"only": args.only, "workload": w.name, "median_ms": statistics.median(ms), "status": st}))
    return 0 if st == 0 else 1


def run_ours(args):
    import torch
    from attention_rope_causal_gb300 import binding, build, inputs
    rank, world, local = dist_setup(args)
    build.build()
    binding.load()
    w = inputs.NAMED[args.workload]
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    q, k, v, out, lse, ws = gpu_setup(w, ("fused", "prerotate", "split"))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    step = fwd_fn(w, q, k, v, out, lse, ws["fused"], "fused", stream)

    warm_steps, warm_s = warm_up(step, args.warmup, flush, stream)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    ms = time_steps(step, args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    st = binding.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}: {binding.last_error()}")
    total_s = max_over_ranks(sum(ms) / 1e3, world)
    value = aggregate(w.causal_flops / 1e12, args.steps, world, total_s)
    per_launch_ms = statistics.mean(ms)

    # end to end through the C ABI with host buffers (pinned H2D of q, k, v, the call, D2H of out and
    # lse every step), pipelined over two buffer sets
    barrier(world)
    e2e_step_ms, h2d, d2h = e2e_pipelined(w, q, k, v, args.steps, max(args.warmup, 3))
    barrier(world)
    e2e_s = max_over_ranks(e2e_step_ms * args.steps / 1e3, world)

    # the competing pre-rotation path, and the RoPE pass alone (HBM-bound)
    side_steps = max(20, args.steps // 10)

    def median_ms(f, clean_l2=False):
        warm_up(f, args.warmup, flush, stream)
        return statistics.median(time_steps(f, side_steps, flush, stream, clean_l2=clean_l2))

    pre_ms = median_ms(fwd_fn(w, q, k, v, out, lse, ws["prerotate"], "prerotate", stream))
    split_ms = median_ms(fwd_fn(w, q, k, v, out, lse, ws["split"], "split", stream))
    plain_ms = median_ms(plain_fn(w, q, k, v, out, lse, stream))
    rope_pass = rope_pass_fn(w, stream)
    rope_ms = median_ms(rope_pass)
    rope_ms_clean = median_ms(rope_pass, clean_l2=True)
    rope_b = 2 * (q.numel() + k.numel()) * q.element_size()
    # the backward pass on the forward's out / lse (a training step's second half)
    fwd_fn(w, q, k, v, out, lse, ws["fused"], "fused", stream)()
    bwd_ms = median_ms(bwd_fn(w, q, k, v, out, lse, stream))
    # one decode step against w.N cached keys: the decode kernels (fused mode) and the tile kernels
    dec_ms = {mode: median_ms(decode_fn(w, mode, stream)) for mode in ("fused", "split")}
    kv_bytes = 2 * k.numel() * k.element_size()
    if binding.device_status() != 0:
        raise RuntimeError(f"device status: {binding.last_error()}")

    if rank != 0:
        return 0
    achieved = w.causal_flops / (per_launch_ms / 1e3) / 1e12
    traffic = load_traffic("attn_fwd_fused", w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                   "rope_base": w.rope_base, "mode": "fused", "parallelism": f"replicas x{world}",
                   "l2": "flushed before every step (512 MiB write, outside the timed events)",
                   "queue": "steps enqueued behind a GPU spin, so the host never gates a step"},
        "pct_of_bf16_peak": 100.0 * achieved / peaks["bf16_tflops"],
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                     "kernel": "attn_fwd_kernel<d=128, fused RoPE, bf16>",
                     "peak_source": f"{peaks['source']} (dense bf16 burst)"},
        "e2e": {"value": aggregate(w.causal_flops / 1e12, args.steps, world, e2e_s), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "schedule": "H2D, compute and D2H on three streams over two buffer sets; time from the first "
                            "H2D to the last D2H"},
        "gpu_launches": args.steps,
        "warmup_run": {"steps": warm_steps, "seconds": warm_s, "rule": f">= {args.warmup} steps and >= "
                                                                           f"{WARMUP_MIN_S * 1e3:.0f} ms"},
        "prerotate": {"ms": pre_ms, "tflops": w.causal_flops / (pre_ms / 1e3) / 1e12,
                      "fused_over_prerotate": per_launch_ms / pre_ms,
                      "rope_pass": {"bytes": rope_b,
                                    "ms_after_write_flush": rope_ms,
                                    "gbs_after_write_flush": rope_b / (rope_ms / 1e3) / 1e9,
                                    "ms_after_clean_flush": rope_ms_clean,
                                    "gbs_after_clean_flush": rope_b / (rope_ms_clean / 1e3) / 1e9,
                                    "frac_of_hbm_after_clean_flush": rope_b / (rope_ms_clean / 1e3) / 1e9 / peaks["hbm_gbs"],
                                    "note": "CUDA events; the write flush leaves L2 full of dirty lines that drain "
                                            "during the pass, the clean flush reads its buffer back first; ncu's "
                                            "figure for the same launch (cold, serialised) is in profiles/"}},
        "plain_attention": {"ms": plain_ms, "tflops": w.causal_flops / (plain_ms / 1e3) / 1e12,
                            "alpha_fused": per_launch_ms / plain_ms - 1.0,
                            "note": "mode none: the pre-rotate path's attention kernel alone on rotated Q, K"},
        "split": {"ms": split_ms, "tflops": w.causal_flops / (split_ms / 1e3) / 1e12,
                  "note": "K rotated by the pre-rotation pass, query tiles rotated on chip"},
        "backward": {"ms": bwd_ms, "tflops": 2.5 * w.causal_flops / (bwd_ms / 1e3) / 1e12,
                     "flops_note": "2.5 x the causal forward FLOPs (dS^T Q, dS K, P^T dO, dO V^T and the "
                                   "recomputed Q K^T); the kernels compute Q K^T and dO V^T twice",
                     "kernels": "rope_apply (q', k') + bwd_prep (D) + bwd_dkdv + bwd_dq"},
        "decode": {"workload": f"{w.B} x 1 query per head against {w.N} cached keys, Hq/Hkv = {w.Hq}/{w.Hkv}, d = {w.d}",
                   "ms": dec_ms["fused"], "tile_kernels_ms": dec_ms["split"],
                   "kv_gbs": kv_bytes / (dec_ms["fused"] / 1e3) / 1e9,
                   "kv_frac_of_hbm": kv_bytes / (dec_ms["fused"] / 1e3) / 1e9 / peaks["hbm_gbs"],
                   "kernels": "attn_decode_kernel + attn_decode_combine_kernel (split-KV, 16-row MMA tiles)"},
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = run_cpu_baseline(w)
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    from attention_rope_causal_gb300 import inputs
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=inputs.LLAMA.name, choices=sorted(inputs.NAMED))
    ap.add_argument("--sweep", action="store_true", help="run the crossover sweep instead")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=("fused", "prerotate", "split", "plain", "rope", "backward", "decode"),
                    help="time one path alone (for profilers)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference_arm(args)
    if args.only:
        return run_only(args)
    if args.sweep:
        from attention_rope_causal_gb300 import binding, build
        import torch
        build.build()
        binding.load()
        torch.cuda.set_device(0)
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
