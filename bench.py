#!/usr/bin/env python3
"""Throughput of the projected-feature attention forward on GB300.

One pass = the whole forward (projection of Q and K, scores, online softmax,
value product) over one batch of a workload, inputs resident in HBM.  The
default workload is
    C4: B=1, H=32, N=32768, d=128, m=32, d_v=128, bf16, non-causal,
        Q, K, V iid N(0, 1), P iid N(0, 1/m) per head;
--config picks any of the method's workloads (C1 fp32 N=256; C2 N=2048;
C3 N=8192 causal; C4 N=32768 with --m 16|32|64; C5 N=131072 causal; C5ctl,
the exact-attention control m=d=128, P=I), and --sweep measures all of them
(the metric is quoted against N and m), one JSON line each, optionally
appended to a --results file that a rerun resumes from.  The metric is
TFLOP/s with
    FLOPs = 4 B H N d m + 2 B H N^2 (m + d_v)     (N^2 term halved if causal)
and its fraction of the measured bf16 tensor-core peak.  A timed step holds
enough passes (repeats_per_step) that the timed region lasts at least
--min-seconds; workloads whose inputs fit in L2 get an L2 flush between
passes, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config C1|C2|C3|C4|C5|C5ctl] [--m 16|32|64] [--sweep]
    python bench.py --decode     (the decode row: projected key cache, workload D1)
    python bench.py --backward   (the backward row, workload C3)
    python bench.py --sfa        (the Sparse Feature Attention row, C4 shape)

Under torchrun (N > 1) the ranks split the B*H independent (batch, head)
pairs of one problem (shard.shard_pairs; no data-path collective, strong
scaling); rank 0 prints one JSON line.  --impl reference times the fp64 CPU
oracle on a bounded sample of the same workload on the host cores (rank 0
only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "projected-attention fwd TFLOP/s and % of GB300 bf16 tensor peak vs N, m"
UNIT = "TFLOP/s"
FALLBACK_PEAK_TFLOPS = 1900.0


# ------------------------------------------------------------------ FLOP model
def proj_flops(B, H, N, d, m) -> float:
    """Projection of Q and K: 2 GEMMs of (B H N) x d x m."""
    return 4.0 * B * H * N * d * m


def attn_flops(B, H, N, m, dv, causal) -> float:
    """Scores (2 N^2 m) and value product (2 N^2 d_v) per head, halved when causal."""
    f = 2.0 * B * H * float(N) * N * (m + dv)
    return f / 2 if causal else f


def flops(B, H, N, d, m, dv, causal) -> float:
    return proj_flops(B, H, N, d, m) + attn_flops(B, H, N, m, dv, causal)


def speedup_vs_standard(d, m, dv, N=None) -> float:
    """Cost ratio standard / projected attention at the same N (N -> inf if None)."""
    if N is None:
        return (d + dv) / (m + dv)
    std = 2.0 * N * N * (d + dv)
    return std / (proj_flops(1, 1, N, d, m) + attn_flops(1, 1, N, m, dv, False))


# ------------------------------------------------------------------ multi-GPU host logic
def shard_range(total: int, world: int, rank: int):
    """Contiguous share [lo, hi) of `total` independent units owned by `rank`."""
    from projected_feature_efficient_gb300.shard import shard_range as _sr
    return _sr(total, world, rank)


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest of every rank's value (identity on one process)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ peaks / counters
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), \
            "measured"
    except Exception:
        return FALLBACK_PEAK_TFLOPS, 1700.0, "fallback"


ATTN_SOURCES = ("projected_feature_efficient_gb300/csrc/attn_ws.cu",
                "projected_feature_efficient_gb300/csrc/ptx.cuh",
                "projected_feature_efficient_gb300/csrc/waits.cuh")
TOPK_SOURCES = ("projected_feature_efficient_gb300/csrc/topk.cu",)


def kernel_source_hash(sources=ATTN_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str = None, profile: str = None, sources=ATTN_SOURCES):
    """DRAM bytes per launch from a committed ncu summary (the attention
    kernel's for `workload` by default), if it was taken on the current kernel
    source; else None."""
    name = profile or f"attn_ws_{workload}_dram.md"
    path = os.path.join(ROOT, "profiles", name)
    try:
        vals = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.startswith("- "):
                    k, v = line[2:].split(":", 1)
                    vals[k.strip()] = v.strip().strip("`")
        if vals.get("kernel_source_sha256_16") != kernel_source_hash(sources):
            return None
        return float(vals["dram_bytes_per_full_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: str):
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", device_index],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line.strip()))

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return None
        rows = [s for t, s in self.samples if self.t0 is not None and self.t0 <= t <= self.t1]
        if not rows:  # the timed region was shorter than one sampling period
            rows = [s for _, s in self.samples[-3:]]
        sm, mx, reasons = [], [], set()
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def physical_device(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ------------------------------------------------------------------ oracle (CPU)
def oracle_sample(w, q, k, v, P, target_s: float):
    """Time the fp64 oracle on a bounded sample of the workload: query rows of
    head 0 (evenly spaced) and, when every row of one head fits in the time,
    whole heads.  Returns (flops, seconds, description, threads)."""
    import numpy as np

    import oracle

    def run(heads, rows):
        idx = np.linspace(0, w.N - 1, rows).round().astype(np.int64)
        qs, ks, vs = (t[:1, :heads].contiguous() for t in (q, k, v))
        t0 = time.perf_counter()
        oracle.attention(qs, ks, vs, P[:heads].contiguous(), causal=w.causal, rows=idx)
        dt = time.perf_counter() - t0
        keys = float((idx + 1).sum()) if w.causal else float(rows) * w.N
        fl = heads * (2.0 * w.N * w.d * w.m + 2.0 * rows * w.d * w.m + 2.0 * keys * (w.m + w.dv))
        return fl, dt

    _, t1 = run(1, 1)
    _, t64 = run(1, 64)
    per_row = max((t64 - t1) / 63.0, 1e-6)
    rows = int(max(1, min(w.N, (target_s - t1) / per_row)))
    heads = 1
    if rows == w.N:
        per_head = t1 + w.N * per_row
        heads = int(max(1, min(w.H, target_s / per_head)))
    fl, dt = run(heads, rows)
    desc = (f"{heads} of {w.H} heads, {rows} of {w.N} query rows each (evenly spaced), full key "
            f"range, projection of all keys of those heads; {dt:.1f} s")
    return fl, dt, desc, oracle.num_threads()


# ------------------------------------------------------------------ arms
FWD_CONFIGS = ("C1", "C2", "C3", "C4", "C5", "C5ctl")
# every point of the metric's sweep over N and m: (workload, m)
SWEEP = (("C1", None), ("C2", None), ("C3", None), ("C4", 16), ("C4", 32), ("C4", 64),
         ("C5", None), ("C5ctl", None))


def workload(name="C4", heads=None, m=None):
    """A forward workload by name, optionally with fewer heads (smaller case
    for profiler captures); m picks a point of C4's projection-width sweep."""
    import spa_inputs as si
    w = si.WORKLOADS[name]
    if m is not None and m != w.m:
        if name != "C4":
            raise SystemExit("--m applies to C4 only (its sweep is m in 16, 32, 64)")
        w = w.with_m(m)
    return w.scaled(H=heads) if heads else w


def input_bytes(w) -> int:
    es = 4 if w.dtype == "f32" else 2
    return w.B * w.H * w.N * (2 * w.d + w.dv) * es


def describe(w) -> str:
    import spa_inputs as si
    full = si.WORKLOADS[w.name]
    qk = "rows rescaled to L2 norm sqrt(d)" if w.qk == "norm" else "iid N(0,1)"
    proj = "P = I (exact-attention control)" if w.identity_P else "P iid N(0,1/m) per head"
    return (f"{w.name}{'' if w.H == full.H else '-subset'}: B={w.B} H={w.H} N={w.N} d={w.d} "
            f"m={w.m} d_v={w.dv} {w.dtype} {'causal' if w.causal else 'non-causal'}; "
            f"Q,K {qk}; V iid N(0,1); {proj}")


def config_of(w, world, flush=False, repeats=1, l2=None):
    l2_mb = (l2 or 0) / 1e6
    return {
        "workload": describe(w),
        "B": w.B, "H": w.H, "N": w.N, "d": w.d, "m": w.m, "d_v": w.dv, "causal": w.causal,
        "l2": (f"inputs ({input_bytes(w) / 1e6:.0f} MB) smaller than L2 ({l2_mb:.0f} MB): a "
               f"buffer of twice L2 is written between forwards, outside the timed events"
               if flush else
               f"inputs ({input_bytes(w) / 1e6:.0f} MB) larger than L2 ({l2_mb:.0f} MB); "
               f"no flush between forwards"),
        "repeats_per_step": repeats,
        "api": "spa_attention_prepare + spa_attention_apply on a preallocated workspace",
        "parallelism": (f"dp{world}: the B*H (batch, head) pairs of one problem split across "
                        f"ranks, no data-path collective") if world > 1 else "dp1",
    }


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import spa_inputs as si
    name = args.config or "C4"
    w = workload(name, args.heads, args.m if name == "C4" else None)
    q, k, v = si.make_qkv(w)
    P = si.make_P(w)
    per_step = max(0.5, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    # each step is one bounded sample of about per_step seconds
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, P, per_step)
    fl_tot = dt = 0.0
    for _ in range(args.steps):
        fl, t1, sample, threads = oracle_sample(w, q, k, v, P, per_step)
        fl_tot += fl
        dt += t1
    value = fl_tot / dt / 1e12
    sample = "per step: " + sample
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def fp32_fma_peak(sms: int) -> float:
    """fp32 FMA roofline in TFLOP/s: 128 FMA lanes per SM per clock, 2 FLOPs
    each, at the maximum SM clock."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", 2070.0))
    except (OSError, ValueError):
        mhz = 2070.0
    return 2.0 * 128 * sms * mhz * 1e6 / 1e12


def measure_forward(args, w, rank, world, dev, dist):
    """One JSON line (rank 0) for the forward on workload w."""
    import torch

    import projected_feature_efficient_gb300 as spa
    import spa_inputs as si

    q_h, k_h, v_h = si.make_qkv(w)
    P_h = si.make_P(w)
    # rank r computes its own contiguous share of the problem's (batch, head)
    # pairs (the heads are independent); the shares of all ranks make up the
    # whole problem, so the throughput is that of the whole job
    if world > 1:
        from projected_feature_efficient_gb300.shard import shard_pairs
        _, _, q_h, k_h, v_h, P_h = shard_pairs(q_h, k_h, v_h, P_h, world, rank)
    Bl, Hl = q_h.shape[0], q_h.shape[1]
    q, k, v, P = (t.to(dev) for t in (q_h, k_h, v_h, P_h))
    N, d, m, dv = w.N, w.d, w.m, w.dv
    dcode = spa.SPA_F32 if w.dtype == "f32" else spa.SPA_BF16
    nbytes = spa.spa_attention_workspace_size(Bl, Hl, N, d, m, dv, dcode)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((Bl, Hl, N, dv), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 1024 * 1024)
    flush = input_bytes(w) < l2
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev) if flush else None

    def prepare():
        spa.spa_attention_prepare(q, k, P, dv, ws)

    def apply():
        spa.spa_attention_apply(v, ws, Bl, Hl, N, d, m, causal=w.causal, out=out)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    W = max(3, args.warmup)
    for i in range(W):
        prepare()
        apply()
        if flush:
            flush_buf.fill_(i & 255)
    torch.cuda.synchronize(dev)
    if spa.device_error() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait during warm-up")
    # repeats per step, so that the timed region lasts at least --min-seconds
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(3):
        prepare()
        apply()
        if flush:
            flush_buf.fill_(i & 255)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_iter = max(e0.elapsed_time(e1) / 3 * 1e-3, 1e-6)
    K = args.steps
    R = max(1, math.ceil(args.min_seconds / (K * t_iter)))
    R = min(R, max(1, 20000 // K))
    n = K * R

    def timed_region(sampler):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * n)]
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        sampler.mark_start()
        r0.record(stream)
        for i in range(n):
            ev[3 * i].record(stream)
            prepare()
            ev[3 * i + 1].record(stream)
            apply()
            ev[3 * i + 2].record(stream)
            if flush:
                flush_buf.fill_(i & 255)
        r1.record(stream)
        barrier()
        sampler.mark_end()
        fwd = sum(ev[3 * i].elapsed_time(ev[3 * i + 2]) for i in range(n))
        attn = sum(ev[3 * i + 1].elapsed_time(ev[3 * i + 2]) for i in range(n))
        return fwd, attn, fwd - attn, r0.elapsed_time(r1)

    sampler = ClockSampler(physical_device(dev.index))
    time.sleep(0.3)
    fwd, attn, proj, region = timed_region(sampler)
    clocks = sampler.summary()
    remeasured = False
    if clocks and BAD_REASONS & set(clocks["reasons"]):
        sampler.stop()
        sampler = ClockSampler(physical_device(dev.index))
        time.sleep(0.3)
        fwd, attn, proj, region = timed_region(sampler)
        clocks = sampler.summary()
        remeasured = True
    sampler.stop()
    if spa.device_error() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait")

    fwd_max_ms = max_over_ranks(fwd, dist, dev)
    f_all = flops(w.B, w.H, N, d, m, dv, w.causal)  # the whole problem, all ranks
    value = f_all * n / (fwd_max_ms * 1e-3) / 1e12

    # ---- end to end through the public host-buffer entry point (this rank's share)
    qp, kp, vp, Pp = (x.pin_memory() for x in (q_h, k_h, v_h, P_h))
    out_h = torch.empty((Bl, Hl, N, dv), dtype=torch.float32).pin_memory()
    t0 = time.perf_counter()
    spa.spa_attention_fwd_host(qp, kp, vp, Pp, causal=w.causal, out=out_h)
    t_one = max(time.perf_counter() - t0, 1e-6)
    Ke = int(max(3, min(2000, math.ceil(0.5 / t_one))))
    barrier()
    t0 = time.perf_counter()
    for _ in range(Ke):
        spa.spa_attention_fwd_host(qp, kp, vp, Pp, causal=w.causal, out=out_h)
    te = max_over_ranks(time.perf_counter() - t0, dist, dev)
    e2e_value = f_all * Ke / te / 1e12
    h2d = sum(x.numel() * x.element_size() for x in (qp, kp, vp, Pp))
    d2h = out_h.numel() * out_h.element_size()
    if spa.device_error() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait")

    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        fl, dt, desc, threads = oracle_sample(w, q_h, k_h, v_h, P_h, args.cpu_seconds)
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": desc}
    if rank != 0:
        return None
    peak, peak_sus, peak_src = load_peaks()
    attn_ms = attn / n
    a_fl = attn_flops(Bl, Hl, N, m, dv, w.causal)
    achieved = a_fl / (attn_ms * 1e-3) / 1e12
    if w.dtype == "f32":
        fpk = fp32_fma_peak(props.multi_processor_count)
        roof = {"bound": "alu", "achieved": achieved, "peak": fpk, "unit": "TFLOP/s",
                "frac": achieved / fpk, "traffic": None,
                "kernel": "attn_f32_kernel (scores + softmax + PV in fp32 FMA)",
                "peak_source": "fp32 FMA: 128 lanes/SM/clock x 2 FLOPs x SMs x max SM clock"}
        pct = None
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": (recorded_traffic(f"{w.name}_m{m}") if world == 1 and
                            Hl == workload(w.name, m=w.m).H else None),
                "kernel": "attn_ws_kernel (scores + softmax + PV)",
                "peak_source": f"{peak_src} bf16 burst",
                "frac_of_sustained": achieved / peak_sus}
        pct = 100.0 * value / world / peak
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": fwd_max_ms / K,
        "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "f32" if w.dtype == "f32" else "bf16",
        "data": "synthetic",
        "config": config_of(w, world, flush, R, l2),
        "pct_of_peak": pct,
        "roofline": roof,
        "kernels_ms_per_forward": {"projection": proj / n, "attention": attn_ms},
        "timed_region_ms": region,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "api": "spa_attention_fwd_host", "steps": Ke},
        "gpu_launches": 2 * n,
        "clocks": clocks,
    }
    if remeasured:
        line["remeasured_after_throttle"] = True
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def repeats_for(fn, steps, min_seconds, stream, cap=100000):
    """Repeats per step so that `steps` steps of `fn` last at least min_seconds
    (one pass of fn timed with CUDA events after the warm-up)."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fn()
    e1.record(stream)
    torch.cuda.synchronize()
    t = max(e0.elapsed_time(e1) * 1e-3, 1e-7)
    return int(max(1, min(cap, math.ceil(min_seconds / (steps * t)))))


def results_done(path, key, src_hash):
    """True if the results file already holds the line of `key` measured on the
    current kernel source (a sweep resumes where it stopped)."""
    try:
        with open(path) as f:
            for raw in f:
                try:
                    rec = json.loads(raw)
                except ValueError:
                    continue
                if rec.get("sweep_key") == key and rec.get("kernel_source") == src_hash:
                    return True
    except OSError:
        pass
    return False


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if args.sweep:
        points = [(c, m) for c, m in SWEEP]
    else:
        name = args.config or "C4"
        points = [(name, args.m if name == "C4" else None)]
    src_hash = kernel_source_hash()
    for name, m in points:
        w = workload(name, args.heads, m)
        key = f"{w.name}_m{w.m}"
        if args.results and results_done(args.results, key, src_hash):
            continue
        line = measure_forward(args, w, rank, world, dev, dist)
        if line is not None:
            if args.sweep or args.results:
                line["sweep_key"] = key
                line["kernel_source"] = src_hash
            print(json.dumps(line), flush=True)
            if args.results:
                with open(args.results, "a") as f:
                    f.write(json.dumps(line) + "\n")
        torch.cuda.empty_cache()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


DECODE_METRIC = "projected-key-cache decode GB/s and % of measured GB300 HBM bandwidth"


def decode_bytes(B, H, L, m, dv) -> int:
    """Bytes a decode step must read: per key 2m (fp16 K~) + 4 (row multiplier)
    + 2 d_v (bf16 V); the query and output rows are negligible."""
    return B * H * L * (2 * m + 4 + 2 * dv)


def run_decode(args, rank, world, local_rank):
    """The decode row: one query per (batch, head) against the projected key
    cache of workload D1 (cache filled once, outside the timed region)."""
    import torch
    import torch.distributed as dist

    import projected_feature_efficient_gb300 as spa
    import spa_inputs as si

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = si.WORKLOADS["D1"]
    if args.decode_batch:
        w = w.scaled(B=args.decode_batch)
    B, H, L, d, m, dv = w.B, w.H, w.N, w.d, w.m, w.dv
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + w.number + 7919 * rank)
    k = torch.randn((B, H, L, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((B, H, L, dv), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((B, H, d), generator=g, device=dev).to(torch.bfloat16)
    P = (torch.randn((H, d, m), generator=g, device=dev) / math.sqrt(m)).to(torch.bfloat16)
    kc, kmul = spa.kcache_new(B, H, L, m, device=dev)
    stream = torch.cuda.current_stream(dev)
    # prefill: project every key into the cache (timed separately, after a warm-up call)
    spa.spa_kcache_append(k, P, kc, kmul, 0)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    spa.spa_kcache_append(k, P, kc, kmul, 0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    append_ms = e0.elapsed_time(e1)
    # CPU oracle baseline on heads of batch entry 0 (rank 0, one GPU only)
    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        k0, v0, q0, P0 = k[0:1].cpu(), v[0:1].cpu(), q[0:1].cpu(), P.cpu()
        done, t_used = 0, 0.0
        while done < H and t_used < args.cpu_seconds / 2:
            h = done
            qf = torch.zeros((1, 1, L, d), dtype=torch.bfloat16)
            qf[0, 0, L - 1] = q0[0, h]
            t0 = time.perf_counter()
            oracle.attention(qf, k0[:, h:h + 1], v0[:, h:h + 1], P0[h:h + 1], causal=True,
                             rows=[L - 1])
            t_used += time.perf_counter() - t0
            done += 1
        cpu = {"value": done * L * (2 * m + 4 + 2 * dv) / t_used / 1e9, "unit": "GB/s",
               "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{done} of {B * H} (batch, head) decode rows, all {L} keys each, "
                         f"including the fp64 projection of those keys; {t_used:.1f} s"}
    del k
    out = torch.empty((B, H, dv), dtype=torch.float32, device=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        spa.spa_attention_decode(q, P, kc, kmul, v, L, out=out)
    barrier()
    K = args.steps
    R = repeats_for(lambda: spa.spa_attention_decode(q, P, kc, kmul, v, L, out=out), K,
                    args.min_seconds, stream)
    sampler = ClockSampler(physical_device(local_rank))
    time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    barrier()
    sampler.mark_start()
    ev[0].record(stream)
    for _ in range(K * R):
        spa.spa_attention_decode(q, P, kc, kmul, v, L, out=out)
    ev[1].record(stream)
    barrier()
    sampler.mark_end()
    clocks = sampler.summary()
    sampler.stop()
    t_ms = max_over_ranks(ev[0].elapsed_time(ev[1]), dist, dev) / R  # per K decode steps
    nbytes = decode_bytes(B, H, L, m, dv)
    value = world * nbytes * K / (t_ms * 1e-3) / 1e9

    # end to end: the query from pinned host memory in, the output row out
    q_h = q.cpu().pin_memory()
    out_h = torch.empty((B, H, dv), dtype=torch.float32).pin_memory()
    q_d = torch.empty_like(q)
    Ke = max(1, min(K, 20))
    barrier()
    t0 = time.perf_counter()
    for _ in range(Ke):
        q_d.copy_(q_h, non_blocking=True)
        spa.spa_attention_decode(q_d, P, kc, kmul, v, L, out=out)
        out_h.copy_(out, non_blocking=True)
        torch.cuda.synchronize(dev)
    te = max_over_ranks(time.perf_counter() - t0, dist, dev)
    if spa.device_error() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait")

    if rank == 0:
        hbm = load_hbm_peak()
        achieved = nbytes / (t_ms / K * 1e-3) / 1e9
        line = {
            "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": max(3, args.warmup), "ms_per_step": t_ms * R / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"D1{'' if B == 8 else '-subset'}: decode, B={B} H={H} cached keys L={L} d={d} m={m} "
                                   f"d_v={dv} bf16; K,V,q iid N(0,1); P iid N(0,1/m)",
                       "B": B, "H": H, "L": L, "d": d, "m": m, "d_v": dv,
                       "bytes_per_key": 2 * m + 4 + 2 * dv,
                       "bytes_per_key_k_v_cache": 2 * d + 2 * dv,
                       "l2": f"cache and values ({nbytes / 1e9:.2f} GB) larger than L2; no flush",
                       "repeats_per_step": R,
                       "api": "spa_attention_decode on a resident cache",
                       "parallelism": f"dp{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm[0], "unit": "GB/s",
                         "frac": achieved / hbm[0], "traffic": None,
                         "kernel": "decode_kernel + decode_combine_kernel (one step)",
                         "peak_source": hbm[1]},
            "e2e": {"value": world * nbytes * Ke / te / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": q_h.numel() * q_h.element_size(),
                    "d2h_bytes_per_step": out_h.numel() * out_h.element_size(),
                    "api": "query copy in + spa_attention_decode + output copy out, synchronised",
                    "steps": Ke},
            "cache_append": {"ms": append_ms, "GB/s": B * H * L * (2 * d + 2 * m + 4) / append_ms / 1e6,
                             "api": "spa_kcache_append of all L keys (prefill)"},
            "gpu_launches": 2 * K * R,
            "clocks": clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


BWD_METRIC = "projected-attention backward TFLOP/s (products of dq, dk, dv, dP)"


def bwd_flops(B, H, N, d, m, dv, causal) -> float:
    """FLOPs of the backward's products: the score recompute S, dA = dO V^T,
    dQp, dKp and dV (N^2 terms halved if causal), plus the projections Qp, Kp,
    dq, dk and the two halves of dP (2 N d m each)."""
    n2 = 2.0 * B * H * N * N * (3 * m + 2 * dv) * (0.5 if causal else 1.0)
    return n2 + 6 * 2.0 * B * H * N * d * m


def bwd_kernel_flops(B, H, N, m, dv, causal) -> float:
    """Algorithmic FLOPs of one fused backward kernel launch: the score
    recompute S, dA = dO V^T, dV, dQp and dKp (N^2 terms, halved if causal)."""
    return 2.0 * B * H * N * N * (3 * m + 2 * dv) * (0.5 if causal else 1.0)


def run_backward(args, rank, world, local_rank):
    """The backward row on workload C3 (B=2 H=16 N=8192 d=128 m=32 d_v=128,
    causal); inputs resident; the forward's output and row log-sum-exp are
    computed once beforehand (spa_attention_fwd_lse).  A step is the fused
    backward in its three stages (prepare, the tensor-core kernel, finish);
    the kernel is also timed alone for the roofline."""
    import torch
    import torch.distributed as dist

    import projected_feature_efficient_gb300 as spa
    import spa_inputs as si

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    name = args.config if args.config in ("C3", "C4") else "C3"
    w = workload(name, args.heads, args.m if name == "C4" else None)
    B, H, N, d, m, dv = w.B, w.H, w.N, w.d, w.m, w.dv
    q_h, k_h, v_h = si.make_qkv(w, seed=None if rank == 0 else 1000 + w.number + 7919 * rank)
    P_h = si.make_P(w)
    g = torch.Generator().manual_seed(3000 + rank)
    dO_h = torch.randn((B, H, N, dv), generator=g, dtype=torch.float64).to(torch.bfloat16)
    q, k, v, P, dO = (t.to(dev) for t in (q_h, k_h, v_h, P_h, dO_h))
    out, lse = spa.spa_attention_fwd_lse(q, k, v, P, causal=w.causal)
    ws = torch.empty(spa.spa_attention_bwd_workspace_size(B, H, N, d, m, dv, spa.SPA_BF16),
                     dtype=torch.uint8, device=dev)
    dq = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    dk = torch.empty_like(dq)
    dvo = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    dP = torch.empty((H, d, m), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        spa.spa_attention_bwd_prepare(q, k, P, out, lse, dO, ws)
        spa.spa_attention_bwd_apply(v, dO, dvo, ws, B, H, N, d, m, causal=w.causal)
        spa.spa_attention_bwd_finish(q, k, P, dq, dk, dP, dv, ws)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    W = max(3, args.warmup)
    for _ in range(W):
        step()
    barrier()
    K = args.steps
    R = repeats_for(step, K, args.min_seconds, stream)
    sampler = ClockSampler(physical_device(local_rank))
    time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    barrier()
    sampler.mark_start()
    ev[0].record(stream)
    for _ in range(K * R):
        step()
    ev[1].record(stream)
    barrier()
    # the tensor-core kernel alone (same inputs; the dQp accumulator keeps adding)
    ev[2].record(stream)
    for _ in range(K):
        spa.spa_attention_bwd_apply(v, dO, dvo, ws, B, H, N, d, m, causal=w.causal)
    ev[3].record(stream)
    barrier()
    sampler.mark_end()
    clocks = sampler.summary()
    sampler.stop()
    t_ms = max_over_ranks(ev[0].elapsed_time(ev[1]), dist, dev)
    k_ms = ev[2].elapsed_time(ev[3]) / K
    fl = bwd_flops(B, H, N, d, m, dv, w.causal)
    value = world * fl * K * R / (t_ms * 1e-3) / 1e12
    if spa.device_error() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait")
    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        # whole heads of batch entry 0 at the full N, as many as fit the budget
        done, dt = 0, 0.0
        while done < H and (done == 0 or dt * (done + 1) / done <= args.cpu_seconds):
            h = done
            t0 = time.perf_counter()
            oracle.attention_bwd(q_h[:1, h:h + 1], k_h[:1, h:h + 1], v_h[:1, h:h + 1],
                                 P_h[h:h + 1], dO_h[:1, h:h + 1], causal=w.causal)
            dt += time.perf_counter() - t0
            done += 1
        cpu = {"value": bwd_flops(1, done, N, d, m, dv, w.causal) / dt / 1e12, "unit": UNIT,
               "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{done} of {B * H} (batch, head) pairs at the full N={N} (causal), all "
                         f"gradients; {dt:.1f} s"}
    if rank == 0:
        peak, peak_sus, peak_src = load_peaks()
        achieved = bwd_kernel_flops(B, H, N, m, dv, w.causal) / (k_ms * 1e-3) / 1e12
        line = {
            "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": t_ms / K, "ms_per_backward": t_ms / (K * R),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{w.name} backward: B={B} H={H} N={N} d={d} m={m} d_v={dv} "
                                   f"bf16 {'causal' if w.causal else 'non-causal'}; upstream "
                                   f"gradient iid N(0,1)",
                       "B": B, "H": H, "N": N, "d": d, "m": m, "d_v": dv, "causal": w.causal,
                       "api": "spa_attention_bwd_prepare / _apply / _finish (forward output "
                              "and lse computed once, outside)",
                       "l2": "inputs and workspace (q, k, v, dO and the workspace) exceed L2",
                       "repeats_per_step": R,
                       "parallelism": f"dp{world}"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                         "kernel": "bwd_ws_kernel (S, dP, dV, dKp, dQp on tcgen05)",
                         "peak_source": f"{peak_src} bf16 burst",
                         "frac_of_sustained": achieved / peak_sus},
            "kernels_ms_per_backward": {"bwd_ws_kernel": k_ms, "rest": t_ms / (K * R) - k_ms},
            # ours per backward: projection, statistics, the kernel, the finish
            # (plus two memsets)
            "gpu_launches": 4 * K * R,
            "clocks": clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


SFA_METRIC = "sparse-feature attention fwd TFLOP/s, dense-equivalent (2 B H N^2 (d + d_v))"


def sfa_flops(B, H, N, d, dv, causal) -> float:
    """The dense attention's FLOPs at the full width d (the SFA notes quote
    speedups against it): 2 B H N^2 (d + d_v), halved if causal."""
    return 2.0 * B * H * N * N * (d + dv) * (0.5 if causal else 1.0)


def run_sfa(args, rank, world, local_rank):
    """The SFA row: Top-k (k = 16 of d = 128) of every query and key row, then
    the forward on the sparsified rows at scale 1/sqrt(d), on the C4 shape
    (B=1 H=32 N=32768 d=128 d_v=128 bf16, full attention); inputs resident.
    The Top-k kernel is also timed alone against the measured HBM bandwidth."""
    import torch
    import torch.distributed as dist

    import projected_feature_efficient_gb300 as spa
    import spa_inputs as si

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = si.WORKLOADS["C4"]
    if args.heads:
        w = w.scaled(H=args.heads)
    B, H, N, d, dv, topk = w.B, w.H, w.N, w.d, w.dv, 16
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + w.number + 7919 * rank)
    q = torch.randn((B, H, N, d), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((B, H, N, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((B, H, N, dv), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    ysel = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    W = max(3, args.warmup)
    for _ in range(W):
        spa.spa_sfa_attention_fwd(q, k, v, topk, out=out)
        spa.spa_topk_features(q, topk, out=ysel)
    barrier()
    K = args.steps
    R = repeats_for(lambda: spa.spa_sfa_attention_fwd(q, k, v, topk, out=out), K,
                    args.min_seconds, stream)
    sampler = ClockSampler(physical_device(local_rank))
    time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    barrier()
    sampler.mark_start()
    ev[0].record(stream)
    for _ in range(K * R):
        spa.spa_sfa_attention_fwd(q, k, v, topk, out=out)
    ev[1].record(stream)
    for _ in range(K):
        spa.spa_topk_features(q, topk, out=ysel)
    ev[2].record(stream)
    barrier()
    sampler.mark_end()
    clocks = sampler.summary()
    sampler.stop()
    t_ms = max_over_ranks(ev[0].elapsed_time(ev[1]), dist, dev)
    tk_ms = ev[1].elapsed_time(ev[2]) / K
    fl = sfa_flops(B, H, N, d, dv, w.causal)
    value = world * fl * K * R / (t_ms * 1e-3) / 1e12
    if spa.device_error() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait")
    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        # head 0 at the full N: Top-k of every key row, then query rows (each
        # against all N keys, with its own Top-k) until the budget is spent
        qh, kh, vh = (t[0:1, 0:1].cpu() for t in (q, k, v))
        eye = torch.eye(d, dtype=torch.bfloat16).unsqueeze(0)
        t0 = time.perf_counter()
        ks = torch.from_numpy(oracle.topk_features(kh, topk)).to(torch.bfloat16)
        qs = torch.from_numpy(oracle.topk_features(qh, topk)).to(torch.bfloat16)
        dt = time.perf_counter() - t0
        rows, step = 0, 256
        while rows < N and dt < args.cpu_seconds:
            t0 = time.perf_counter()
            oracle.attention(qs, ks, vh, eye, causal=w.causal, rows=list(range(rows, rows + step)))
            dt += time.perf_counter() - t0
            rows += step
        cpu = {"value": sfa_flops(1, 1, N, d, dv, w.causal) * rows / N / dt / 1e12, "unit": UNIT,
               "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"head 0: Top-k of all {N} key and query rows, then {rows} query rows "
                         f"against all keys; {dt:.1f} s"}
    if rank == 0:
        hbm = load_hbm_peak()
        tk_gbs = 2.0 * q.numel() * 2 / (tk_ms * 1e-3) / 1e9
        line = {
            "metric": SFA_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": t_ms / K, "ms_per_forward": t_ms / (K * R),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"SFA on the C4 shape: B={B} H={H} N={N} d={d} d_v={dv} "
                                   f"bf16, Top-k k={topk} of q and k rows, full attention",
                       "api": "spa_sfa_attention_fwd", "l2": "inputs (805 MB) exceed L2",
                       "repeats_per_step": R,
                       "parallelism": f"dp{world}"},
            "roofline": {"bound": "hbm", "achieved": tk_gbs, "peak": hbm[0], "unit": "GB/s",
                         "frac": tk_gbs / hbm[0],
                         "traffic": (recorded_traffic(profile="topk_rows_bf16_sfa_C4.md",
                                                      sources=TOPK_SOURCES) if H == 32 else None),
                         "kernel": "topk_rows_bf16_tma_kernel (reads and writes q: 2 x 2 bytes per value)",
                         "peak_source": hbm[1]},
            "kernels_ms_per_forward": {"topk_q": tk_ms, "rest": t_ms / (K * R) - tk_ms},
            "gpu_launches": 5 * K * R,  # Top-k of q and k, P = I, projection, attention
            "clocks": clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def load_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in pk and isinstance(pk[key], (int, float)):
                return float(pk[key]), "measured"
    except (OSError, ValueError):
        pass
    return 6800.0, "fallback"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workload (or the C3 backward) with fewer heads (smaller "
                         "case for profiler captures)")
    ap.add_argument("--config", default=None, choices=FWD_CONFIGS,
                    help="workload (forward default C4; --backward default C3)")
    ap.add_argument("--m", type=int, default=32, choices=(16, 32, 64),
                    help="projection width of the C4 sweep")
    ap.add_argument("--sweep", action="store_true",
                    help="measure every forward workload and C4 m point, one line each")
    ap.add_argument("--results", default=None,
                    help="append each line to this JSONL file and skip the workloads it "
                         "already holds for the current kernel source")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="shortest timed region (passes per step are repeated to reach it)")
    ap.add_argument("--decode", action="store_true",
                    help="measure the decode row (projected key cache, workload D1) instead")
    ap.add_argument("--sfa", action="store_true",
                    help="measure the Sparse Feature Attention row (C4 shape, k=16) instead")
    ap.add_argument("--backward", action="store_true",
                    help="measure the backward row instead (workload C3, or --config C4 "
                         "with --m)")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="decode with another batch size (smaller case for profiler captures)")
    args = ap.parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.decode:
        return run_decode(args, rank, world, local_rank)
    if args.backward:
        return run_backward(args, rank, world, local_rank)
    if args.sfa:
        return run_sfa(args, rank, world, local_rank)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
