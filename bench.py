"""Benchmark of the Positional LSH approximate-ALiBi hot path on one GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
redraw the s hashes per head and rebuild their bin records
(plsh_bins_resample: draw, bitmap, neighbour scans), then the fused block
attention with its in-kernel work queue and O / l epilogue (plsh_alibi_attn).
Inputs are resident in HBM when the timed region starts; L2 is flushed
(256 MiB write) between timed steps, outside the per-step events.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle
on a bounded sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from positional_lsh_approximation_gb300.inputs import WORKLOADS, make_qkv  # noqa: E402

METRIC = "approx-ALiBi attn tokens/s (n=8k, 32h, d=128, s=10) & % of bf16 TC roofline, 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {
            "hbm_gbs": float(d.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
            "bf16_tflops": float(d.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
            "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained",
                                                 FALLBACK_PEAKS["bf16_tflops_sustained"])),
            "source": "measured",
        }
    return dict(FALLBACK_PEAKS, source="fallback")


def work_counts(w, offsets, starts):
    """Algorithmic work of one launch from the actual bins.

    F_block = 4 d B sum_h sum_t sum_bins pairs(b), pairs(b) = b(b+1)/2 when
    causal else b^2 (QK^T and PV per (i, j) pair in a block); bytes = Q, K, V
    read once and O written once.  Also the tensor-core work the kernel
    executes: per (b, h, 128-row tile) every key tile of the union envelope,
    two 128x128x128 products (S in bf16, P V in f16)."""
    lens = np.diff(starts.astype(np.int64))
    # drop the terminal-to-next-hash differences: use per-hash slices
    pairs = 0
    H, s = w.Hq, w.s
    env_tiles = 0
    QT = (w.n + 127) // 128
    for h in range(H):
        lo_min = np.full(QT, np.iinfo(np.int64).max)
        for t in range(s):
            st = starts[offsets[h * s + t]:offsets[h * s + t + 1]].astype(np.int64)
            b = np.diff(st)
            pairs += int((b * (b + 1) // 2).sum() if w.causal else (b * b).sum())
            i0 = np.arange(QT) * 128
            lo = st[np.searchsorted(st, i0, side="right") - 1]
            lo_min = np.minimum(lo_min, lo)
        if w.causal:
            env_tiles += int((np.arange(QT) - lo_min // 128 + 1).sum())
        else:
            env_tiles += int(QT * QT)  # upper bound, not used for the headline
    f_block = 4.0 * w.d * w.B * pairs
    e = 2 if w.dtype == "bf16" else 4
    bytes_ = w.B * w.n * w.d * e * (2 * w.Hq + 2 * w.Hkv)
    mma = w.B * env_tiles * 2 * 2.0 * 128 * 128 * 128
    return f_block, bytes_, mma, env_tiles * w.B


class ClockSampler:
    """nvidia-smi samples during the timed region (clocks and throttle reasons)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_traffic():
    """dram bytes per launch of the fused kernel from the committed ncu summary,
    valid only for the exact kernel source it was taken from."""
    path = os.path.join(ROOT, "profiles", "attn_tc_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_sha256_16") != kernel_source_digest():
        return None
    return d.get("traffic_bytes_per_launch")


KERNEL_SOURCES = ("attn_tc.cu", "tc_ptx.cuh", "bins_dev.cuh", "plsh_internal.h")


def workload_config(w, world: int) -> dict:
    """The bench line's `config`: the workload and the timing protocol of the
    GPU arm; the oracle arm reports the same object, so that the two lines
    name one configuration."""
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "n": w.n,
            "d": w.d, "s": w.s, "causal": w.causal,
            "sigma": "ALiBi slopes sigma_h = 2^(8h/H)" if not w.sigma else list(w.sigma),
            "hashes": "redrawn on the device every step (same seed)",
            "l2": "flushed between timed steps (256 MiB write)",
            "parallelism": f"replicas x{world}"}


def kernel_source_digest() -> str:
    """sha256 (16 hex digits) over the fused kernel's source files."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "positional_lsh_approximation_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------ cross-rank timing
def max_over_ranks(x: float, device=None) -> float:
    """Largest x over the ranks of the default process group (x itself when
    there is none): the job is as slow as its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, steps: int, total_ms: float) -> float:
    """Units processed by all replicas per second over the slowest rank's time."""
    return units_per_rank * world * steps / (total_ms / 1e3)


# ------------------------------------------------------------- our arm
def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist

    import positional_lsh_approximation_gb300 as plsh

    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    plsh.build()
    Qn, Kn, Vn = make_qkv(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    Q = torch.from_numpy(Qn).to(tdt).to(dev)
    K = torch.from_numpy(Kn).to(tdt).to(dev)
    V = torch.from_numpy(Vn).to(tdt).to(dev)
    O = torch.empty_like(Q)
    sigma = w.sigmas()
    stream = torch.cuda.current_stream()
    bins = plsh.sample_bins(w.n, sigma, w.s, w.hash_seed)
    offsets, starts = bins.to_host()
    f_block, bytes_, mma_exec, tiles = work_counts(w, offsets, starts)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    seed = w.hash_seed   # the same draw every step, so F_block is exact for each

    for i in range(args.warmup):
        bins.resample(sigma, seed)
        plsh.alibi_attn(Q, K, V, bins, w.causal, out=O)
    plsh.stream_status()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # timed pass 1, the metric: whole steps with events only at the step
    # boundaries (an event between the sampler and the fused kernel would
    # stop the kernel from overlapping the sampler's tail, as it does in use)
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    # timed pass 2, the roofline: the same steps with events around each kernel
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            flush.zero_()
            a, c = ev_step[i]
            a.record(stream)
            bins.resample(sigma, seed)
            plsh.alibi_attn(Q, K, V, bins, w.causal, out=O)
            c.record(stream)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            e0, e1, e2 = ev[i]
            e0.record(stream)
            bins.resample(sigma, seed)
            e1.record(stream)
            plsh.alibi_attn(Q, K, V, bins, w.causal, out=O)
            e2.record(stream)
        torch.cuda.synchronize()
        # clock soak: the same steps back to back for ~1.5 s, so that the
        # clock record under load holds several samples (not part of value)
        soak_steps = 0
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        t_end = time.perf_counter() + args.soak_seconds
        while time.perf_counter() < t_end:
            for _ in range(64):
                bins.resample(sigma, seed)
                plsh.alibi_attn(Q, K, V, bins, w.causal, out=O)
            soak_steps += 64
            torch.cuda.synchronize()
        s1.record(stream)
        torch.cuda.synchronize()
    plsh.stream_status()
    soak_ms = s0.elapsed_time(s1) / max(1, soak_steps)
    step_ms = [a.elapsed_time(c) for a, c in ev_step]
    attn_ms = [b.elapsed_time(c) for a, b, c in ev]
    sample_ms = [a.elapsed_time(b) for a, b, c in ev]
    total_ms = max_over_ranks(sum(step_ms), dev)
    value = whole_job_rate(w.B * w.n, world, args.steps, total_ms)
    attn_avg_s = statistics.mean(attn_ms) / 1e3

    # end to end through the public API with host buffers (pinned)
    Qh, Kh, Vh = (x.cpu().pin_memory() for x in (Q, K, V))
    Oh = torch.empty(Q.shape, dtype=Q.dtype).pin_memory()
    for i in range(2):
        bins.resample(sigma, seed)
        plsh.alibi_attn(Qh, Kh, Vh, bins, w.causal, out=Oh)
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bins.resample(sigma, seed)
        plsh.alibi_attn(Qh, Kh, Vh, bins, w.causal, out=Oh)
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    h2d = sum(x.numel() * x.element_size() for x in (Q, K, V))
    d2h = O.numel() * O.element_size()

    # exact dense ALiBi on the same inputs, and the approximation error
    E = torch.empty_like(Q)
    plsh.alibi_exact(Q, K, V, sigma, w.causal, out=E)
    torch.cuda.synchronize()
    ex_ms = []
    for i in range(max(3, min(args.steps, 10))):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plsh.alibi_exact(Q, K, V, sigma, w.causal, out=E)
        b.record(stream)
        torch.cuda.synchronize()
        ex_ms.append(a.elapsed_time(b))
    plsh.stream_status()
    bins.resample(sigma, w.hash_seed)
    plsh.alibi_attn(Q, K, V, bins, w.causal, out=O)
    torch.cuda.synchronize()
    diff = (O.float() - E.float())
    approx_err = {
        "max_abs": float(diff.abs().max()),
        "mean_abs": float(diff.abs().mean()),
        "rel_fro": float(diff.norm() / E.float().norm()),
    }
    ex_avg_s = statistics.mean(ex_ms) / 1e3
    ex_flops = 4.0 * w.d * w.B * w.Hq * (w.n * (w.n + 1) / 2 if w.causal else w.n * w.n)

    pk = peaks()
    peak_tf = pk["bf16_tflops"]
    achieved_tf = f_block / attn_avg_s / 1e12
    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) Q/K/V of the workload's shape, no weights)",
        "config": workload_config(w, world),
        "roofline": {
            "bound": "tensor",
            "achieved": achieved_tf,
            "peak": peak_tf,
            "unit": "TFLOP/s",
            "frac": achieved_tf / peak_tf,
            "traffic": kernel_traffic(),
            "kernel": "attn_tc_kernel<false,true>",
            "flops_per_launch": f_block,
            "kernel_ms": attn_avg_s * 1e3,
            "peak_source": pk["source"] + " (burst, kernel timed alone)",
            "hbm_frac": bytes_ / attn_avg_s / 1e9 / pk["hbm_gbs"],
            "bytes_per_launch": bytes_,
            "mma_flops_executed": mma_exec,
            "mma_frac_executed": mma_exec / attn_avg_s / 1e12 / peak_tf,
            "tiles_executed": tiles,
        },
        "sample_ms": statistics.mean(sample_ms),
        "e2e": {"value": w.B * w.n * world / (statistics.mean(e2e_ms) / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": statistics.mean(e2e_ms)},
        "gpu_launches": 2 * args.steps,  # sample_kernel + attn_tc_kernel per step of the metric pass
        "exact": {"tokens_per_s": w.B * w.n / ex_avg_s, "ms": ex_avg_s * 1e3,
                  "tflops": ex_flops / ex_avg_s / 1e12,
                  "frac": ex_flops / ex_avg_s / 1e12 / peak_tf},
        "approx_error_vs_exact": approx_err,
        "clocks": dict(clocks.summary(), soak={"steps": soak_steps, "ms_per_step": soak_ms,
                                               "l2": "not flushed (back to back)"}),
    }
    result["decode"] = measure_decode(w, bins, sigma, flush, stream)
    result["fixed_blocks"] = measure_fixed(w, sigma, Q, K, V, E, flush, stream)
    result["shared_groups"] = measure_shared_groups(w, sigma, Q, K, V, E, flush, stream)
    result["backward"] = measure_backward(w, bins, Q, K, V, f_block, flush, stream)
    result["bias_error"] = measure_bias_error()
    if not args.no_configs:
        del E
        result["split"] = measure_split(flush, stream)
        result["configs"] = measure_configs(flush, stream)
        result["crossover"] = measure_crossover(flush, stream, result["configs"].get("scout"))
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(w, Qn, Kn, Vn, offsets, starts, args.cpu_seconds)
    return result


# ------------------------------------------------ the other workloads
CONFIG_NAMES = ["qwen_s10", "qwen_s20", "sweep_s1", "sweep_s5", "sweep_s10", "sweep_s20",
                "sweep_s40", "scout", "mistral_d64"]


def device_qkv(w, seed):
    """N(0,1) Q, K, V of the workload's shape drawn on the device (seeded;
    the timing lines do not need the oracle's host copies), with the peaky
    rows of the Qwen-shaped workload."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q = torch.randn(w.B, w.Hq, w.n, w.d, generator=g, device="cuda")
    k = torch.randn(w.B, w.Hkv, w.n, w.d, generator=g, device="cuda")
    v = torch.randn(w.B, w.Hkv, w.n, w.d, generator=g, device="cuda")
    if w.peaky_frac > 0:
        rows = torch.rand(w.B, w.n, generator=g, device="cuda") < w.peaky_frac
        sc = torch.where(rows, w.peaky_scale, 1.0)[:, None, :, None]
        q *= sc
        k *= sc
    return q.to(tdt), k.to(tdt), v.to(tdt)


def time_calls(fn, flush, stream, iters):
    import torch
    fn()
    torch.cuda.synchronize()
    ms = []
    for _ in range(iters):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    return statistics.median(ms)


def approx_vs_exact(w, flush, stream, iters=5, exact_iters=3, seed=77):
    """One workload: the fused kernel's time against its roofline (block
    FLOPs at the tensor peak, bytes at the HBM peak, whichever is slower), the
    exact kernel's time, and the approximation's error against exact ALiBi."""
    import torch
    import positional_lsh_approximation_gb300 as plsh
    q, k, v = device_qkv(w, seed)
    sigma = w.sigmas()
    bins = plsh.sample_bins(w.n, sigma, w.s, w.hash_seed)
    off, st = bins.to_host()
    f_block, bytes_, mma, tiles = work_counts(w, off, st)
    O = torch.empty_like(q)
    t_a = time_calls(lambda: plsh.alibi_attn(q, k, v, bins, w.causal, out=O), flush, stream,
                     iters)
    E = torch.empty_like(q)
    t_e = time_calls(lambda: plsh.alibi_exact(q, k, v, sigma, w.causal, out=E), flush, stream,
                     exact_iters)
    plsh.stream_status()
    diff = O.float() - E.float()
    err = float(diff.norm() / E.float().norm())
    del diff, O, E, q, k, v
    bins.free()
    pk = peaks()
    t_tc = f_block / (pk["bf16_tflops"] * 1e12)
    t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
    ex_flops = 4.0 * w.d * w.B * w.Hq * (w.n * (w.n + 1) / 2 if w.causal else w.n * w.n)
    sec = t_a / 1e3
    return {"n": w.n, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "s": w.s,
            "approx_ms": t_a, "tokens_per_s": w.B * w.n / sec,
            "bound": "tensor" if t_tc >= t_hbm else "hbm",
            "frac": max(t_tc, t_hbm) / sec,
            "tensor_frac": f_block / sec / 1e12 / pk["bf16_tflops"],
            "hbm_frac": bytes_ / sec / 1e9 / pk["hbm_gbs"],
            "mma_frac_executed": mma / sec / 1e12 / pk["bf16_tflops"],
            "flops_per_launch": f_block, "bytes_per_launch": bytes_,
            "exact_ms": t_e, "exact_frac": ex_flops / (t_e / 1e3) / 1e12 / pk["bf16_tflops"],
            "approx_over_exact_time": t_a / t_e,
            "approx_error_vs_exact_rel_fro": err}


def measure_split(flush, stream):
    """The key-range split of long work items on a case that needs it: one
    pair of heads of a long sequence with wide bins (few items, envelopes of
    up to ~100 key tiles), automatic split against none."""
    import torch
    import positional_lsh_approximation_gb300 as plsh
    from positional_lsh_approximation_gb300.inputs import Workload
    w = Workload("long_pair", 1, 2, 1, 16384, 128, "bf16", True, 10, (2000.0, 3000.0))
    q, k, v = device_qkv(w, 5)
    bins = plsh.sample_bins(w.n, w.sigmas(), w.s, w.hash_seed)
    O = torch.empty_like(q)
    out = {"workload": "B=1, 2 query heads / 1 KV head, n=16384, d=128, causal, s=10, "
                       "sigma 2000 and 3000"}
    for name, parts in (("unsplit", 1), ("automatic", 0)):
        plsh.set_split_parts(parts)
        out[name + "_ms"] = time_calls(lambda: plsh.alibi_attn(q, k, v, bins, True, out=O),
                                       flush, stream, 10)
    plsh.set_split_parts(0)
    plsh.stream_status()
    bins.free()
    out["speedup"] = out["unsplit_ms"] / out["automatic_ms"]
    return out


def measure_configs(flush, stream):
    """Every other workload's line, L2 flushed before each timed call."""
    out = {}
    for name in CONFIG_NAMES:
        w = WORKLOADS[name]
        out[name] = approx_vs_exact(w, flush, stream, exact_iters=2 if name == "scout" else 3)
    return out


def measure_crossover(flush, stream, scout=None):
    """Approximation against exact ALiBi in wall-clock on the Scout-shaped
    heads (40 query / 8 KV heads, d = 128, sigma = 256, s = 16) as n grows."""
    w0 = WORKLOADS["scout"]
    rows = []
    for n in (16384, 32768, 65536, 131072):
        if n == w0.n and scout is not None:
            r = scout
        else:
            r = approx_vs_exact(w0.with_(n=n), flush, stream, exact_iters=3)
        rows.append({"n": n, "approx_ms": r["approx_ms"], "exact_ms": r["exact_ms"],
                     "speedup_over_exact": r["exact_ms"] / r["approx_ms"],
                     "approx_error_vs_exact_rel_fro": r["approx_error_vs_exact_rel_fro"]})
    return rows


# ------------------------------------------------------------ backward
def measure_backward(w, bins, Q, K, V, f_block, flush, stream, iters=5):
    """Gradients of the workload's attention for a random dO: the tensor-core
    path (a forward pass in its row statistics mode, the backward kernel,
    the dQ conversion) against its roofline, the paper's block work of the
    backward (S, dP, dV, dK, dQ: 10 d per block pair, 2.5 x the forward's
    F_block) at the bf16 peak; the same from the forward's saved O and
    log-sum-exp (the rows' Delta from O instead of a forward recomputation),
    with the forward that writes them; and the CUDA-core path on the same
    call."""
    import torch
    import positional_lsh_approximation_gb300 as plsh
    g = torch.Generator(device=Q.device)
    g.manual_seed(99)
    dO = torch.randn(Q.shape, generator=g, device=Q.device).to(Q.dtype)
    run = lambda: plsh.alibi_attn_backward(Q, K, V, dO, bins, w.causal)
    t = time_calls(run, flush, stream, iters)
    plsh.stream_status()
    # from the forward's saved O and log-sum-exp, as a training step has them
    O, lse = plsh.alibi_attn_lse(Q, K, V, bins, w.causal)
    t_fwd_lse = time_calls(lambda: plsh.alibi_attn_lse(Q, K, V, bins, w.causal, out=O, lse=lse),
                           flush, stream, iters)
    t_saved = time_calls(lambda: plsh.alibi_attn_backward_lse(Q, K, V, O, lse, dO, bins, w.causal),
                         flush, stream, iters)
    plsh.stream_status()
    os.environ["PLSH_PATH"] = "simt"
    try:
        t_simt = time_calls(run, flush, stream, 2)
    finally:
        del os.environ["PLSH_PATH"]
    plsh.stream_status()
    pk = peaks()
    f_bwd = 2.5 * f_block
    return {"path": plsh.attn_path(Q, bins, w.causal), "ms": t,
            "tokens_per_s": w.B * w.n / (t / 1e3), "flops_per_call": f_bwd,
            "tensor_frac": f_bwd / (t / 1e3) / 1e12 / pk["bf16_tflops"],
            "from_saved_lse_ms": t_saved,
            "from_saved_lse_tensor_frac": f_bwd / (t_saved / 1e3) / 1e12 / pk["bf16_tflops"],
            "forward_with_lse_ms": t_fwd_lse,
            "cuda_core_ms": t_simt,
            "kernels": "attn_tc_kernel (row statistics) + bwd_tc_kernel + dq_convert_kernel"}


# ------------------------------------------- hashes shared across a group
def measure_shared_groups(w, sigma, Q, K, V, E, flush, stream, iters=10):
    """Hashes shared by the query heads of a KV group (one draw per group at
    the geometric mean of its heads' scales) against per-head hashes at equal
    s: attention time on the same kernel and error against exact ALiBi."""
    import torch
    import positional_lsh_approximation_gb300 as plsh
    G = w.Hq // w.Hkv
    sg = [float(np.exp(np.mean(np.log(sigma[g * G:(g + 1) * G])))) for g in range(w.Hkv)]
    src = plsh.sample_bins(w.n, sg, w.s, w.hash_seed)
    sh = plsh.bins_share_groups(src, w.Hq)
    O = torch.empty_like(Q)
    t = time_calls(lambda: plsh.alibi_attn(Q, K, V, sh, w.causal, out=O), flush, stream, iters)
    plsh.stream_status()
    diff = O.float() - E.float()
    err = float(diff.norm() / E.float().norm())
    sh.free()
    src.free()
    return {"sigma_per_group": "geometric mean of the group's sigma_h", "s": w.s,
            "attn_ms": t, "tokens_per_s": w.B * w.n / (t / 1e3), "rel_fro_vs_exact": err}


# ---------------------------------------------------- bias error at scale
def measure_bias_error(n=131072, sigma=256.0, ss=(4, 16, 64), iters=60):
    """||L* - M~|| in max and spectral norm for one head at n = 131072 (the
    Scout-shaped length, sigma = 256) as s grows: values, time per call (host
    clock: the call blocks) and the fitted slope of the spectral error in
    log s (the summary's O(1/sqrt(s)) convergence)."""
    import positional_lsh_approximation_gb300 as plsh
    rows = []
    for s_ in ss:
        b = plsh.sample_bins(n, [sigma], s_, 0)
        plsh.bias_error(b, sigma, 0, lanczos_iters=8, seed=1)     # warm-up
        t0 = time.perf_counter()
        mx, sp = plsh.bias_error(b, sigma, 0, lanczos_iters=iters, seed=1)
        dt = time.perf_counter() - t0
        b.free()
        rows.append({"s": s_, "max_abs": mx, "spectral": sp, "ms": dt * 1e3})
    slope = float(np.polyfit(np.log([r["s"] for r in rows]),
                             np.log([r["spectral"] for r in rows]), 1)[0])
    return {"n": n, "sigma": sigma, "lanczos_iters": iters, "rows": rows,
            "spectral_slope_vs_log_s": slope}


# ------------------------------------------------------- fixed blocks
def measure_fixed(w, sigma, Q, K, V, E, flush, stream, iters=10):
    """The fixed-blocks baseline at the workload's s: blocks of width
    round(2 sigma_h) (the mean width of the random bins), s evenly shifted
    grids; attention time on the same kernel and error against exact ALiBi."""
    import torch
    import positional_lsh_approximation_gb300 as plsh
    widths = [max(1, int(round(2.0 * sg))) for sg in sigma]
    t0 = time.perf_counter()
    fb = plsh.bins_fixed(w.n, widths, w.s)
    build_ms = (time.perf_counter() - t0) * 1e3
    O = torch.empty_like(Q)
    for _ in range(3):
        plsh.alibi_attn(Q, K, V, fb, w.causal, out=O)
    plsh.stream_status()
    ms = []
    for _ in range(iters):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plsh.alibi_attn(Q, K, V, fb, w.causal, out=O)
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    plsh.stream_status()
    diff = O.float() - E.float()
    fb.free()
    t = statistics.median(ms)
    return {"widths": "round(2 sigma_h)", "s": w.s, "build_ms": build_ms,
            "attn_ms": t, "tokens_per_s": w.B * w.n / (t / 1e3),
            "rel_fro_vs_exact": float(diff.norm() / E.float().norm())}


# ------------------------------------------------------------ decode step
DECODE_BATCH = 64


def measure_decode(w, bins, sigma, flush, stream, iters=20):
    """One decode step (plsh_alibi_decode) for a batch of DECODE_BATCH
    sequences whose caches hold the workload's n positions, the query at the
    last one; same heads, hashes and scales as the workload.  Bound by HBM:
    the algorithmic bytes are the K and V rows of each KV group's widest key
    envelope (every query head of a group reads inside it) plus q and o."""
    import torch
    import positional_lsh_approximation_gb300 as plsh
    if not w.causal:
        return None
    dev = stream.device
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    esz = 2 if w.dtype == "bf16" else 4
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    Bd, pos = DECODE_BATCH, w.n - 1
    K = torch.randn(Bd, w.Hkv, w.n, w.d, generator=g, device=dev).to(tdt)
    V = torch.randn(Bd, w.Hkv, w.n, w.d, generator=g, device=dev).to(tdt)
    q = torch.randn(Bd, w.Hq, 1, w.d, generator=g, device=dev).to(tdt)
    o = torch.empty_like(q)
    offsets, starts = bins.to_host()
    env = []
    for h in range(w.Hq):
        lo = pos
        for t in range(w.s):
            st = starts[offsets[h * w.s + t]:offsets[h * w.s + t + 1]]
            lo = min(lo, int(st[np.searchsorted(st, pos, side="right") - 1]))
        env.append(pos - lo + 1)
    per_group = w.Hq // w.Hkv
    widest = [max(env[g0 * per_group:(g0 + 1) * per_group]) for g0 in range(w.Hkv)]
    bytes_ = Bd * (sum(widest) * 2 * w.d * esz + 2 * w.Hq * w.d * esz)
    for _ in range(3):
        plsh.alibi_decode(q, K, V, bins, pos, out=o)
    plsh.stream_status()
    ms = []
    for _ in range(iters):
        # evict L2 by reading a buffer larger than it: a written flush would
        # leave ~129 MB of dirty lines whose write-back lands in this short step
        flush.sum()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plsh.alibi_decode(q, K, V, bins, pos, out=o)
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    plsh.stream_status()
    t = statistics.median(ms) / 1e3
    pk = peaks()
    return {"batch": Bd, "n_cache": w.n, "pos": pos, "tokens_per_s": Bd / t, "ms": t * 1e3,
            "envelope_keys_mean": float(np.mean(env)), "bytes": bytes_,
            "achieved_gbs": bytes_ / t / 1e9, "peak_gbs": pk["hbm_gbs"],
            "hbm_frac": bytes_ / t / 1e9 / pk["hbm_gbs"], "peak_source": pk["source"],
            "kernels": "decode_group_kernel + decode_merge_kernel",
            "l2": "evicted before each step (256 MiB read)"}


# ---------------------------------------------------------- oracle on CPU
def cpu_baseline(w, Qn, Kn, Vn, offsets, starts, budget_s):
    """The fp64 oracle as it stands, on every host core, over a bounded sample
    of token positions (all heads of batch element 0)."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    rng = np.random.default_rng(0)
    npos = 16
    elapsed = 0.0
    done = 0
    while True:
        pos = rng.integers(0, w.n, size=npos).astype(np.int32)
        rb = np.zeros(npos * w.Hq, np.int32)
        rh = np.repeat(np.arange(w.Hq, dtype=np.int32), npos)
        ri = np.tile(pos, w.Hq)
        t0 = time.perf_counter()
        oracle.plsh_attn_rows(Qn, Kn, Vn, offsets, starts, w.s, w.causal, (rb, rh, ri))
        dt = time.perf_counter() - t0
        elapsed += dt
        done += npos
        if elapsed >= budget_s or done >= w.B * w.n:
            break
        npos = int(min(4096, max(npos * 2, npos * (budget_s - elapsed) / max(dt, 1e-3) * 0.5)))
    all_cores = oracle.max_threads()
    # the same oracle on one core, over a smaller sample
    oracle.set_threads(1)
    pos = rng.integers(0, w.n, size=max(1, min(256, done // 16))).astype(np.int32)
    t0 = time.perf_counter()
    oracle.plsh_attn_rows(Qn, Kn, Vn, offsets, starts, w.s, w.causal,
                          (np.zeros(pos.size * w.Hq, np.int32),
                           np.repeat(np.arange(w.Hq, dtype=np.int32), pos.size),
                           np.tile(pos, w.Hq)))
    one_core = pos.size / (time.perf_counter() - t0)
    oracle.set_threads(cores)
    return {"value": done / elapsed, "unit": "tokens/s", "cores": all_cores,
            "kind": "oracle",
            "sample": f"{done} random token positions x all {w.Hq} heads of batch 0, "
                      f"fp64, {elapsed:.1f} s",
            "one_core": {"value": one_core, "unit": "tokens/s",
                         "sample": f"{pos.size} random token positions x all {w.Hq} heads"}}


def run_reference(args, rank, world):
    w = WORKLOADS[args.workload]
    import oracle
    Qn, Kn, Vn = make_qkv(w)
    offsets, starts = oracle.sample_bins(w.n, w.sigmas(), w.s, w.hash_seed)
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)
    rng = np.random.default_rng(1)
    per_step = args.ref_positions
    for i in range(args.warmup):
        pos = rng.integers(0, w.n, size=max(1, per_step // 4)).astype(np.int32)
        oracle.plsh_attn_rows(Qn, Kn, Vn, offsets, starts, w.s, w.causal,
                              (np.zeros(pos.size * w.Hq, np.int32),
                               np.repeat(np.arange(w.Hq, dtype=np.int32), pos.size),
                               np.tile(pos, w.Hq)))
    times = []
    for i in range(args.steps):
        pos = rng.integers(0, w.n, size=per_step).astype(np.int32)
        rows = (np.zeros(per_step * w.Hq, np.int32),
                np.repeat(np.arange(w.Hq, dtype=np.int32), per_step), np.tile(pos, w.Hq))
        t0 = time.perf_counter()
        oracle.plsh_attn_rows(Qn, Kn, Vn, offsets, starts, w.s, w.causal, rows)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = per_step * args.steps / total
    sample = (f"{per_step} random token positions x all {w.Hq} heads per step "
              f"(of {w.B * w.n} tokens), fp64 oracle")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) Q/K/V of the workload's shape, no weights)",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle",
                         "cores": oracle.max_threads(), "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mistral", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' lines and the crossover sweep")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-positions", type=int, default=96)
    ap.add_argument("--soak-seconds", type=float, default=1.5,
                    help="back-to-back steps after the timed ones, for the clock record")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
