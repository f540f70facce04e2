"""Benchmark of the GB300 fused attention forward: one JSON line on rank 0.

A step is one attn_fwd call (the whole fused forward: Q/K/V tile loads, QK^T,
online softmax, PV, epilogue) over one batch of seeded synthetic input.  The
default workload is the long-sequence throughput shape B=4, H=16, N=4096,
D=128, non-causal.  Value = algorithmic TFLOP/s (4*B*H*N^2*D, halved when
causal) measured with CUDA events on the launching stream, inputs resident in
device memory.  ``e2e`` repeats the measurement through the C ABI with pinned
host buffers (attn_fwd_from_host): each step copies Q, K, V in and O, LSE out,
overlapping the copies with the kernels chunk by chunk.

``--impl reference`` times the CPU oracle (plain C, fp64) on the host cores
instead: each step is a bounded sample of rows of the same workload.

Under torchrun every rank runs its own copy of the workload on its own GPU
(independent problems, no collective on the data path: weak scaling); rank 0
prints the line with value = total FLOPs of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tiled_attention_forward_fa2_gb300.inputs import BASED_WORKLOADS, WORKLOADS  # noqa: E402

METRIC = "attention fwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "b4h16n4096d128"
L2_BYTES = 129 * 2**20
FALLBACK_PEAK_TFLOPS = 1900.0
_CSRC = "tiled_attention_forward_fa2_gb300/csrc/"
# Sources that decide what each kernel family runs (kernel, launcher, PTX helpers);
# an ncu summary's traffic figure is used only while these are unchanged.
KERNEL_SOURCES = {
    "fwd": [_CSRC + f for f in ("attn_fwd_kernel.cuh", "attn_fwd_short_kernel.cuh", "sm103_ptx.cuh", "attn_fwd.cu")],
    "based": [_CSRC + f for f in ("based_fwd_kernel.cuh", "based_fwd_host.cuh", "sm103_ptx.cuh")],
    "bwd": [_CSRC + f for f in ("attn_bwd_kernel.cuh", "attn_bwd_host.cuh", "sm103_ptx.cuh")],
}


def kernel_source_hash(family: str = "fwd") -> str:
    """Hash of one kernel family's sources' code: comments and blank lines are
    left out, so editing a comment does not mark the committed ncu summaries stale."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()[:16]


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, dist_mod=None, device=None) -> float:
    """The largest `value` over all ranks (the job is as slow as its slowest rank)."""
    if dist_mod is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs its own replica, all within `ms_per_step`."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"bf16_tflops": FALLBACK_PEAK_TFLOPS, "hbm_gbs": 6800.0}, "fallback"


def ncu_traffic(workload: str, kernel: str = "attn_fwd_sm103", family: str = "fwd"):
    """DRAM bytes per launch from the committed ncu summary, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_src or not m_tr or m_src.group(1) != kernel_source_hash(family):
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) taken while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.marks = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc is not None and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, float("inf"))
        rows = [s for (t, s) in self.samples if t0 <= t <= t1]
        in_region = len(rows)
        if not rows:
            rows = [s for (_, s) in self.samples]
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons),
                "samples": in_region, "samples_total": len(self.samples)}


def to_dev(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def oracle_parity(w, o, lse, q, k, v):
    """Run the CPU oracle on the whole workload: (cpu_baseline, parity) objects.

    ``o``, ``lse`` are the device results of the timed workload (float64 copies).
    Parity compares every element: max and mean |dO| (with where the max is)
    and the LSE relative error |dLSE| / max(1e-2, |LSE|) (floored where a
    relative error is ill-posed), against the stated bounds."""
    import oracle

    t0 = time.perf_counter()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    secs = time.perf_counter() - t0
    cpu = {"value": w.flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
           "sample": f"the whole workload {w.name} (every query row, all visible keys), {secs:.1f} s wall"}
    if w.flops <= 5e9:
        # Small workloads: also the oracle on one core (a few seconds at most).
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v, w.causal, w.scale, nthreads=1)
        secs1 = time.perf_counter() - t0
        cpu["single_core"] = {"value": w.flops / secs1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "sample": f"the whole workload {w.name}, {secs1:.2f} s wall"}
    do = np.abs(o - o_ref)
    at = np.unravel_index(int(np.argmax(do)), do.shape)
    dl = np.abs(lse - lse_ref)
    parity = {"against": "CPU oracle (fp64 two-pass softmax attention), every element",
              "max_abs_dO": float(do.max()), "mean_abs_dO": float(do.mean()),
              "max_at_bhnd": [int(x) for x in at], "O_ref_at_max": float(o_ref[at]),
              "lse_err": float((dl / np.maximum(1e-2, np.abs(lse_ref))).max()), "lse_abs_max": float(dl.max()),
              "bounds": {"max_abs_dO": 2e-2, "mean_abs_dO": 2e-3, "lse_err": 1e-3}}
    parity["pass"] = bool(parity["max_abs_dO"] <= 2e-2 and parity["mean_abs_dO"] <= 2e-3 and parity["lse_err"] <= 1e-3)
    return cpu, parity


def time_backward(pkg, w, qd, kd, vd, o, lse, stream, dev, flush, scratch, steps, pg, world):
    """Device-timed backward (attn_bwd_qk: dQ, dK, dV; 2.5x the forward FLOPs) on the
    forward's own O and LSE with a seeded upstream gradient; same timing rules."""
    import torch

    from tiled_attention_forward_fa2_gb300.inputs import normal_bf16_bits

    dod = to_dev(normal_bf16_bits(w.B * w.H * w.N * w.D, w.seed, 3).reshape(w.B, w.H, w.N, w.D), dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    delta = torch.empty_like(lse)

    def step():
        st = pkg.attn_bwd_qk(qd, kd, vd, o, lse, dod, dq, dk, dv, delta, w.B, w.H, w.N, w.n_keys, w.D, w.causal,
                             w.scale, stream)
        if st != pkg.ATTN_OK:
            raise RuntimeError(pkg.attn_status_string(st))

    for _ in range(3):
        step()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    if flush:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            scratch.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
    else:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
    st = pkg.attn_last_status(stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(pkg.attn_status_string(st))
    ms = max_over_ranks(ms, pg, dev)
    flops = pkg.attn_bwd_qk_flops(w.B, w.H, w.N, w.n_keys, w.D, w.causal)
    return {"metric": "attention bwd TFLOP/s (dQ, dK, dV; 2.5x the forward FLOPs)", "value": job_tflops(flops, world, ms),
            "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps, "gpu_launches": 2 * steps,
            "kernels": "attn_bwd_dq_sm103 + attn_bwd_dkdv_sm103", "traffic": ncu_traffic(w.name, "attn_bwd", "bwd")}


def based_config(w, world=1):
    """The ``config`` of a Based line (the same dict for both arms)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "F": w.F, "D": w.D, "causal": True, "seed": w.seed,
            "q_std": w.q_std, "scale": w.scale, "layout": "q, k [B,H,N,F], v, y [B,H,N,D] bf16; z [B,H,N] fp32",
            "l2": f"working set {based_bytes(w) / 2**20:.0f} MiB > 2x 129 MiB L2, no flush",
            "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU"}


def based_bytes(w) -> float:
    """Algorithmic HBM bytes of one Based forward: q, k, v read, y written (bf16), z written (fp32)."""
    return float(w.B * w.H * w.N * (2 * 2 * w.F + 2 * 2 * w.D + 4))


BASED_METRIC = "Based linear attention fwd TFLOP/s (linear-form FLOPs, bf16, 1×GB300) and HBM roofline"


def run_reference_based(args, w):
    import oracle

    q, k, v = w.qkv()
    rng = np.random.default_rng(1)
    bh, ri = rng.integers(0, w.B * w.H, 32).astype(np.int64), rng.integers(0, w.N, 32).astype(np.int64)
    t0 = time.perf_counter()
    oracle.based_rows(q, k, v, w.scale, bh, ri)
    per_row = max((time.perf_counter() - t0) / 32, 1e-7)
    rows = int(max(8, min(8192, 60.0 / (args.steps + args.warmup) / per_row)))
    bh = rng.integers(0, w.B * w.H, rows).astype(np.int64)
    ri = rng.integers(0, w.N, rows).astype(np.int64)
    # The oracle's work is quadratic; the value is reported in the metric's own
    # units: linear-form FLOPs of the sampled rows (per token, as the GPU line counts).
    fs = 1 + w.F + w.F * (w.F + 1) // 2
    step_flops = 4.0 * fs * (w.D + 1) * rows
    for _ in range(args.warmup):
        oracle.based_rows(q, k, v, w.scale, bh, ri)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.based_rows(q, k, v, w.scale, bh, ri)
    dt = time.perf_counter() - t0
    value = step_flops * args.steps / dt / 1e12
    line = {"impl": "reference", "metric": BASED_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": based_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"{rows} sampled rows (all earlier tokens each) of {w.name} per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_based(args, w):
    """One JSON line for a Based workload: device-timed attn_based_fwd, e2e from pinned
    host buffers, HBM roofline, the oracle on the whole workload (parity, cpu_baseline)."""
    import torch

    import tiled_attention_forward_fa2_gb300 as pkg

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    pkg.library()
    q, k, v = w.qkv()
    qd, kd, vd = to_dev(q, dev), to_dev(k, dev), to_dev(v, dev)
    y = torch.empty_like(vd)
    z = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        st = pkg.attn_based_fwd(qd, kd, vd, y, z, w.B, w.H, w.N, w.F, w.D, w.scale, stream)
        if st != pkg.ATTN_OK:
            raise RuntimeError(pkg.attn_status_string(st))

    for _ in range(args.warmup):
        step()
    st = pkg.attn_last_status(stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(pkg.attn_status_string(st))
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.wait_first()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark()
    if pg:
        pg.barrier()
    st = pkg.attn_last_status(stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(pkg.attn_status_string(st))
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, dev)
    if sampler:
        sampler.stop()

    # End to end: pinned host q, k, v up, the kernel, y and z down, every step.
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()  # noqa: E731
    qh, kh, vh = pin(q), pin(k), pin(v)
    yh = torch.empty(y.shape, dtype=torch.bfloat16).pin_memory()
    zh = torch.empty(z.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        step()
        yh.copy_(y, non_blocking=True)
        zh.copy_(z, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(args.steps, 20))
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, pg, dev)
    y_host = y.float().cpu().numpy().astype(np.float64) if rank == 0 else None
    z_host = z.cpu().numpy().astype(np.float64) if rank == 0 else None
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    peaks, peak_src = measured_peaks()
    flops = pkg.attn_based_fwd_flops(w.B, w.H, w.N, w.F, w.D)
    alg = based_bytes(w)
    gbs = alg / (ms * 1e-3) / 1e9
    cpu, parity = None, None
    if not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        y_ref, z_ref = oracle.based_fwd(q, k, v, w.scale)
        secs = time.perf_counter() - t0
        fs = 1 + w.F + w.F * (w.F + 1) // 2
        cpu = {"value": 4.0 * fs * (w.D + 1) * w.tokens / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
               "kind": "oracle", "sample": f"the whole workload {w.name} (every row), {secs:.1f} s wall"}
        dy = np.abs(y_host - y_ref)
        zr = float((np.abs(z_host - z_ref) / z_ref).max())
        parity = {"against": "CPU oracle (fp64 quadratic definition), every element", "max_abs_dy": float(dy.max()),
                  "mean_abs_dy": float(dy.mean()), "z_rel_max": zr,
                  "bounds": {"max_abs_dy": 2e-2, "mean_abs_dy": 1e-3, "z_rel": 2.0 ** -6}}
        parity["pass"] = bool(dy.max() <= 2e-2 and dy.mean() <= 1e-3 and zr <= 2.0 ** -6)
    line = {
        "metric": BASED_METRIC, "value": job_tflops(flops, world, ms), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": based_config(w, world),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                     "frac": gbs / float(peaks["hbm_gbs"]), "traffic": ncu_traffic(w.name, "based_fwd_sm103", "based"),
                     "algorithmic_bytes": alg,
                     "peak_source": f"hbm_gbs of {peak_src}", "kernel": "based_fwd_sm103"},
        "cpu_baseline": cpu,
        "e2e": {"value": job_tflops(flops, world, e2e_ms), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(q.nbytes + k.nbytes + v.nbytes),
                "d2h_bytes_per_step": int(y.numel() * 2 + z.numel() * 4), "ms_per_step": e2e_ms, "steps": e2e_steps},
        "gpu_launches": args.steps, "clocks": sampler.summary() if sampler else None,
        "kernel_source": kernel_source_hash("based"), "parity": parity,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle

    if isinstance(w, type(next(iter(BASED_WORKLOADS.values())))):
        return run_reference_based(args, w)
    q, k, v = w.qkv()
    rng = np.random.default_rng(1)
    # Per step: a fixed sample of rows sized so that warm-up + timed steps take about a minute.
    bh, ri = rng.integers(0, w.B * w.H, 32).astype(np.int64), rng.integers(0, w.N, 32).astype(np.int64)
    t0 = time.perf_counter()
    oracle.attn_rows(q, k, v, w.causal, w.scale, bh, ri)
    per_row = max((time.perf_counter() - t0) / 32, 1e-7)
    rows = int(max(8, min(4096, 60.0 / (args.steps + args.warmup) / per_row)))
    bh = rng.integers(0, w.B * w.H, rows).astype(np.int64)
    ri = rng.integers(0, w.N, rows).astype(np.int64)
    vis = np.minimum(ri + 1 + w.n_keys - w.N, w.n_keys) if w.causal else np.full(ri.shape, w.n_keys)
    step_flops = float(4.0 * w.D * vis.sum())
    for _ in range(args.warmup):
        oracle.attn_rows(q, k, v, w.causal, w.scale, bh, ri)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attn_rows(q, k, v, w.causal, w.scale, bh, ri)
    dt = time.perf_counter() - t0
    value = step_flops * args.steps / dt / 1e12
    sample = f"{rows} sampled query rows (all keys each) of {w.name} per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def working_set_bytes(w) -> int:
    """Q, K, V read and O written (bf16)."""
    return 2 * w.B * w.H * w.D * (2 * w.N + 2 * w.n_keys)


def needs_flush(w) -> bool:
    """Working set below 2x L2: rewrite a 2x-L2 buffer between steps, each launch timed alone."""
    return working_set_bytes(w) < 2 * L2_BYTES


def rotating_sets(w) -> int:
    """Copies of the inputs and outputs the back-to-back forward leg rotates over: between two uses
    of one copy the other copies (at least 2x L2 of traffic) pass through L2."""
    ws = working_set_bytes(w)
    return 1 + -(-2 * L2_BYTES // ws)


def workload_config(w, world=1, extra=None):
    """The line's ``config``: the same dict for both arms (ours and --impl reference)."""
    in_bytes = 2 * w.B * w.H * w.D * (w.N + 2 * w.n_keys)
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "Nk": w.n_keys, "D": w.D, "causal": w.causal, "seed": w.seed,
           "q_std": w.q_std, "scale": w.scale, "layout": "[B,H,N,D] bf16, D innermost",
           "l2": ("working set < 2x L2: 2x-L2 buffer rewritten between steps, each launch timed alone"
                  if needs_flush(w) else f"inputs {in_bytes / 2**20:.0f} MiB > 129 MiB L2, no flush"),
           "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU"}
    if extra:
        cfg.update(extra)
    return cfg


def run_ours(args, w):
    import torch

    import tiled_attention_forward_fa2_gb300 as pkg

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    pkg.library()

    q, k, v = w.qkv()
    w_job = w
    if args.shard_heads and world > 1:
        # Strong scaling: each rank computes its contiguous block of the B*H
        # slices (independent problems, no collective on the data path).
        import dataclasses

        from tiled_attention_forward_fa2_gb300.sharding import head_range
        a, b = head_range(w.B * w.H, rank, world)
        cut = lambda t: np.ascontiguousarray(t.reshape(w.B * w.H, *t.shape[2:])[a:b][None])  # noqa: E731
        q, k, v = cut(q), cut(k), cut(v)
        w = dataclasses.replace(w, B=1, H=b - a)
    qd, kd, vd = to_dev(q, dev), to_dev(k, dev), to_dev(v, dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    in_bytes = q.nbytes + k.nbytes + v.nbytes
    flush = needs_flush(w)
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    if args.backward:
        # Inputs of the backward: the forward's O and LSE, and an upstream dO.
        assert pkg.attn_fwd_qk(qd, kd, vd, o, lse, w.B, w.H, w.N, w.n_keys, w.D, w.causal, w.scale, stream) == pkg.ATTN_OK
        dod = to_dev(w.qkv()[0][..., ::-1].copy(), dev)  # any bf16 tensor of O's shape
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        delta = torch.empty_like(lse)

    # Copies of the inputs and outputs (the same values) for the back-to-back leg
    # of a working set below 2x L2: rotating over them, every launch reads inputs
    # that are not in L2.  The timed steps use the first copy, after a flush.
    sets = [(qd, kd, vd, o, lse)]
    if flush and not args.backward:
        sets += [(qd.clone(), kd.clone(), vd.clone(), torch.empty_like(o), torch.empty_like(lse))
                 for _ in range(rotating_sets(w) - 1)]

    def step(i=0):
        if args.backward:
            st = pkg.attn_bwd_qk(qd, kd, vd, o, lse, dod, dq, dk, dv, delta, w.B, w.H, w.N, w.n_keys, w.D, w.causal,
                                 w.scale, stream)
        else:
            sq, sk, sv, so, sl = sets[i % len(sets)]
            if w.n_keys == w.N:
                st = pkg.attn_fwd(sq, sk, sv, so, sl, w.B, w.H, w.N, w.D, w.causal, w.scale, stream)
            else:
                st = pkg.attn_fwd_qk(sq, sk, sv, so, sl, w.B, w.H, w.N, w.n_keys, w.D, w.causal, w.scale, stream)
        if st != pkg.ATTN_OK:
            raise RuntimeError(pkg.attn_status_string(st))

    for i in range(args.warmup):
        step(i)
    st = pkg.attn_last_status(stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(pkg.attn_status_string(st))

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.wait_first()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark()
    if flush:
        # Working set below 2x L2: rewrite a 2x-L2 buffer between steps, time each launch alone.
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            scratch.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        elapsed_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        elapsed_ms = e0.elapsed_time(e1)
    if sampler:
        sampler.mark()
    if pg:
        pg.barrier()
    st = pkg.attn_last_status(stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(pkg.attn_status_string(st))
    elapsed_ms = max_over_ranks(elapsed_ms, pg, dev)
    if sampler:
        sampler.stop()
    l2_warm_ms = b2b_ms = None
    if flush and not args.backward:
        # Beside the line's value: the steps back to back between two events, over
        # copies of the inputs and outputs (every step's inputs out of L2).  Launch
        # latency then overlaps the previous step and the events' ~2 us timestamp
        # step is divided by the step count; each step's dirty O lines drain
        # during the next one, and the load is sustained.
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        for i in range(len(sets)):
            step(i)
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        b2b_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, dev)
        # The same launches back to back, without the buffer rewrite: inputs stay
        # resident in L2 between launches (reported beside the flushed number).
        n_warm = min(args.steps, 200)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_warm):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        l2_warm_ms = max_over_ranks(e0.elapsed_time(e1) / n_warm, pg, dev)

    flops = (pkg.attn_bwd_qk_flops if args.backward else pkg.attn_fwd_qk_flops)(w.B, w.H, w.N, w.n_keys, w.D,
                                                                                w.causal)
    ms_per_step = elapsed_ms / args.steps
    if w_job is w:
        value = job_tflops(flops, world, ms_per_step)
    else:  # the ranks share one problem: its FLOPs over the slowest rank's time
        value = (pkg.attn_bwd_qk_flops if args.backward else pkg.attn_fwd_qk_flops)(
            w_job.B, w_job.H, w_job.N, w_job.n_keys, w_job.D, w_job.causal) / (ms_per_step * 1e-3) / 1e12

    if args.backward:
        if rank == 0:
            peaks, peak_src = measured_peaks()
            peak = float(peaks["bf16_tflops"])
            achieved = flops / (ms_per_step * 1e-3) / 1e12
            line = {"metric": "attention bwd TFLOP/s (bf16, 1\u00d7GB300; 2.5x forward FLOPs)", "value": value,
                    "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "bf16", "data": "synthetic", "config": workload_config(w, world, {"pass": "backward"}),
                    "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                                 "frac": achieved / peak, "traffic": ncu_traffic(w.name, "attn_bwd", "bwd"),
                                 "peak_source": f"bf16_tflops (burst) of {peak_src}",
                                 "kernel": "attn_bwd_dq_sm103 + attn_bwd_dkdv_sm103"},
                    "gpu_launches": 2 * args.steps, "clocks": sampler.summary() if sampler else None,
                    "kernel_source": kernel_source_hash("bwd")}
            print(json.dumps(line), flush=True)
        if pg:
            pg.destroy_process_group()
        return

    # End to end through the C ABI with pinned host buffers (attn_fwd_from_host).
    e2e_steps = max(3, min(args.steps, 50))
    qh, kh, vh = (torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
                  for a in (q, k, v))
    oh = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        # One C-ABI call: copies of Q, K, V up and O, LSE down, overlapped with the
        # kernels chunk by chunk; the stream holds all of it.
        st = pkg.attn_fwd_from_host(qh, kh, vh, oh, lh, qd, kd, vd, o, lse, w.B, w.H, w.N, w.n_keys, w.D, w.causal,
                                    w.scale, stream)
        if st != pkg.ATTN_OK:
            raise RuntimeError(pkg.attn_status_string(st))

    for _ in range(2):
        e2e_step()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, pg, dev)

    backward = None
    if not args.no_backward and w.D <= 128:
        backward = time_backward(pkg, w, qd, kd, vd, o, lse, stream, dev, flush, scratch, max(3, min(args.steps, 100)),
                                 pg, world)
    o_host = o.float().cpu().numpy().astype(np.float64) if rank == 0 else None
    lse_host = lse.cpu().numpy().astype(np.float64) if rank == 0 else None

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    peaks, peak_src = measured_peaks()
    if backward is not None:
        bpeak = float(peaks["bf16_tflops"])
        backward.update({"peak": bpeak, "frac": backward["value"] / bpeak,
                         "peak_source": f"bf16_tflops (burst) of {peak_src}"})
    peak = float(peaks["bf16_tflops"])
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    kernel = pkg.attn_fwd_kernel_name(w.B, w.H, w.N, w.n_keys, w.D, w.causal)
    traffic = ncu_traffic(w.name, kernel.split("<")[0])
    # Below the ridge point (peak FLOP/s over HBM bytes/s) the kernel is bound by
    # HBM bandwidth: algorithmic bytes = Q, K, V read + O written (bf16) + LSE (fp32).
    alg_bytes = 2.0 * w.B * w.H * w.D * (2 * w.N + 2 * w.n_keys) + 4.0 * w.B * w.H * w.N
    ridge = peak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    if flops / alg_bytes < ridge:
        roofline = {"bound": "hbm", "achieved": alg_bytes / (ms_per_step * 1e-3) / 1e9, "peak": float(peaks["hbm_gbs"]),
                    "unit": "GB/s", "peak_source": f"hbm_gbs of {peak_src}"}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "peak_source": f"bf16_tflops (burst) of {peak_src}"}
    roofline["frac"] = roofline["achieved"] / roofline["peak"]
    roofline["traffic"] = traffic
    roofline["algorithmic_bytes"] = alg_bytes
    roofline["flop_per_byte"] = flops / alg_bytes
    roofline["kernel"] = kernel
    cpu, parity = None, None
    if not args.no_cpu_baseline:
        # The oracle on the whole workload: its wall time is the CPU baseline and
        # its output the parity check of the timed run's own output (every row).
        cpu, parity = oracle_parity(w, o_host, lse_host, q, k, v)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak" if w_job is w else "strong",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "pct_of_peak": 100.0 * achieved / peak,
        "config": workload_config(w_job, world, None if w_job is w else {
            "parallelism": f"B*H slices split over {world} ranks (contiguous blocks, no collective)"}),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": job_tflops(flops, world, e2e_ms) if w_job is w else value * ms_per_step / e2e_ms,
                "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(in_bytes), "d2h_bytes_per_step": int(o.numel() * 2 + lse.numel() * 4),
                "ms_per_step": e2e_ms, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": sampler.summary() if sampler else None,
        "kernel_source": kernel_source_hash(),
        "parity": parity,
        "backward": backward,
        # Working sets under 2x L2 (the line's value: each launch timed alone after
        # a 2x-L2 buffer rewrite): the launches back to back over copies of the
        # inputs, and back to back on one copy with the inputs resident in L2.
        "back_to_back": None if b2b_ms is None else {
            "value": job_tflops(flops, world, b2b_ms) if w_job is w else value * ms_per_step / b2b_ms,
            "unit": "TFLOP/s", "ms_per_step": b2b_ms, "steps": args.steps, "copies": len(sets)},
        "l2_resident": None if l2_warm_ms is None else {
            "value": job_tflops(flops, world, l2_warm_ms) if w_job is w else value * ms_per_step / l2_warm_ms,
            "unit": "TFLOP/s", "ms_per_step": l2_warm_ms, "steps": min(args.steps, 200)},
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(BASED_WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the CPU oracle (no cpu_baseline and no parity object)")
    ap.add_argument("--no-backward", action="store_true", help="leave the backward object out of the line")
    ap.add_argument("--shard-heads", action="store_true",
                    help="under torchrun: split the workload's B*H slices over the ranks (strong scaling) instead of "
                         "running one replica per rank (weak scaling, the default)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward (dQ, dK, dV; 2.5x the forward FLOPs) instead of the forward; device timing only")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = WORKLOADS.get(args.workload) or BASED_WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif args.workload in BASED_WORKLOADS:
        run_based(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
