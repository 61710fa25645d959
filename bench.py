"""Benchmark of the exact-attention hot path: one step = forward + backward
over one batch of synthetic bf16 inputs, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Default workload: B=1, H=16, N=32768, d=128, bf16, non-causal, scale
1/sqrt(d): the largest configuration of the fixed-token sweep (B*N = 32768)
and the long-context shape.  Reported beside it, each with its own kernel
rates: the causal variant of the same shape (its forward is the B1 H16 N32768
causal long-context forward), the B2 H16 N8192 causal backward, and the
B2 H16 N4096 step with the other entry points (deterministic backward, FP8
and CTA-pair forwards).  Algorithmic FLOPs: forward 4*B*H*N^2*d (halved when
causal), backward 2.5x that.

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs its
own replica on its own GPU (independent batches, no collective on the data
path: weak scaling); the step time is the max over ranks.

--impl reference times the fp64 CPU oracle on the host cores instead, each step
a bounded sample of the same workload (forward and backward rows of one head).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PAGES_PEAK_TFLOPS = 2250.0  # dense BF16 peak the pages quote for the GPU generation
METRIC = "attention fwd/bwd TFLOPs/s (bf16, d=128) and % of 2.25 PF dense BF16 peak"
WORKLOAD = dict(B=1, H=16, N=32768, d=128)
WORKLOAD_NAME = "attention fwd+bwd B1 H16 N32768 d128 non-causal"
BWD_CAUSAL = dict(B=2, H=16, N=8192, d=128)  # the B2 H16 N8192 causal backward
SMALL = dict(B=2, H=16, N=4096, d=128)  # the B2 H16 N4096 step and the other entry points


def flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    if causal:
        f *= 0.5
    return f, 2.5 * f


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: one JSON line per configuration of the "
                         "fixed-token sweep (B*N = 32768, H = 16, N = 1k..32k, d = 64/128, both masks)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (for profiler runs)")
    ap.add_argument("--loop", choices=sorted(LOOP_ENTRIES),
                    help="instead of the bench line: call one entry point warmup + steps times "
                         "on --shape (L2 flushed before each call) and print its median time; "
                         "the case a profiler captures")
    ap.add_argument("--shape", default="2,16,4096,128", help="B,H,N,d for --loop")
    ap.add_argument("--causal", action="store_true", help="causal mask for --loop")
    ap.add_argument("--poly", type=int, default=None,
                    help="exponentials per 8 on the FMA pipe in the forward (--loop)")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="instead of the bench line: the fp64 oracle timed on the host cores on "
                         "each configuration's oracle coverage (one JSON line each; no GPU)")
    return ap.parse_args()


# --loop entry points: name -> (forward or backward, call)
LOOP_ENTRIES = ("fwd", "fwd_2cta", "fwd_fp8", "bwd", "bwd_2cta", "bwd_deterministic")


def loop_arm(args):
    """One entry point called repeatedly on one shape, each call timed with
    CUDA events on the launching stream (L2 flushed before each call)."""
    import torch

    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N, d = (int(x) for x in args.shape.split(","))
    causal = bool(args.causal)
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", 0)
    if args.poly is not None:
        fa.fa_set_exp2_poly_share(args.poly)
    q, k, v, do = (t.to(dev) for t in attention_inputs(B, H, N, d, seed=1))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    wsf = fa.fwd_workspace_for(q, causal)
    ws = fa.workspace_for(q, deterministic=args.loop == "bwd_deterministic")
    ws8 = None
    if args.loop == "fwd_fp8":
        ws8 = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    calls = {
        "fwd": lambda: fa.fa_fwd(q, k, v, o, lse, scale, causal, wsf),
        "fwd_2cta": lambda: fa.fa_fwd_2cta(q, k, v, o, lse, scale, causal),
        "fwd_fp8": lambda: fa.fa_fwd_fp8(q, k, v, o, lse, scale, causal, True, ws8),
        "bwd": lambda: fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale, causal, ws),
        "bwd_2cta": lambda: fa.fa_bwd_2cta(q, k, v, o, lse, do, dq, dk, dv, scale, causal, ws),
        "bwd_deterministic": lambda: fa.fa_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv,
                                                             scale, causal, ws),
    }
    call = calls[args.loop]
    ms, kern_ms = [], []
    fa.fa_timing_enable(True)
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            ms.append(e0.elapsed_time(e1))
            if args.loop in ("fwd", "fwd_fp8"):
                kern_ms.append(fa.fa_timing_last_ms(fa.KERNEL_FWD))
    fa.fa_timing_enable(False)
    status = fa.fa_last_device_status()
    if status != fa.FA_OK:
        raise RuntimeError(f"device status {fa.status_string(status)}")
    f_fwd, f_bwd = flops(B, H, N, d, causal)
    f = f_fwd if args.loop.startswith("fwd") else f_bwd
    med = statistics.median(ms)
    print(json.dumps({"loop": args.loop, "shape": [B, H, N, d], "causal": causal,
                      "poly": fa.fa_get_exp2_poly_share(), "ms": med,
                      "tflops": f / med / 1e9, "calls": len(ms),
                      "kernel_ms": statistics.median(kern_ms) if kern_ms else None}), flush=True)


# DRAM traffic of one launch of the dominant kernel (the backward main kernel)
# on this workload: dram__bytes_read.sum + dram__bytes_write.sum from one
# `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum` capture (cold
# cache) of B1 H4 N32768 d128 (213259008 + 94483968 bytes), times 4 for the
# 16 independent heads of the headline (the full-size launch is too large to
# capture).  It describes the kernel built from the sources whose digest is
# recorded with it, and is reported as null as soon as any of them changes.
NCU_TRAFFIC = {
    "kernel": "fa_bwd_kernel<128>",
    "workload": WORKLOAD_NAME,
    "bytes": 4 * (213259008 + 94483968),
    "captured": "B1 H4 N32768 d128, scaled by 4",
    "sources_sha256": "2b438741862e2d8945ab4a5b3934dc9d3b119f45a14483163712c53cbaa60358",
}
KERNEL_SOURCES = ("fa_bwd.cu", "fa_device.cuh", "fa_kernels.h", "exp2_poly_coeffs.h")


def kernel_sources_sha256() -> str:
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "exact_attention_98_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def cpu_model() -> str:
    """The host CPU's model name as lscpu or /proc/cpuinfo give it ("" if
    neither does)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return ""


def oracle_fields(tf: float, threads: int, desc: str) -> dict:
    """The cpu_baseline object: the oracle's rate on its sample, the host it
    ran on and the time the whole fwd+bwd step of the workload would take at
    that rate."""
    B, H, N, d = WORKLOAD["B"], WORKLOAD["H"], WORKLOAD["N"], WORKLOAD["d"]
    f_fwd, f_bwd = flops(B, H, N, d, False)
    return {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc,
            "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "projected_full_step_s": (f_fwd + f_bwd) / (tf * 1e12) if tf > 0 else None}


def replica_seed(rank: int) -> int:
    """Seed of rank `rank`'s replica batch: each rank works on its own batch."""
    return rank


def max_over_ranks(x: float, device=None) -> float:
    """The max of a per-rank scalar over the process group (the job's time is
    its slowest rank's); x itself when there is no group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_replica: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank runs one replica of the workload."""
    return world * flops_per_replica / (ms * 1e-3) / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------- CPU oracle


def oracle_sample(seconds_target: float, steps: int = 1, warmup: int = 0):
    """Times the fp64 oracle on a bounded sample of the workload: forward and
    dQ-rows backward of R query rows of head 0 (R sized so one sample takes
    about `seconds_target`), `warmup` untimed samples then `steps` timed ones.
    Returns (TFLOP/s, threads, description, per-step seconds, FLOPs per step)."""
    import numpy as np

    import oracle
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N, d = WORKLOAD["B"], WORKLOAD["H"], WORKLOAD["N"], WORKLOAD["d"]
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = attention_inputs(1, 1, N, d, seed=0)
    q, k, v, do = (t.double().numpy()[0, 0] for t in (q, k, v, do))

    def run(rows):
        oracle.fwd_head(q, k, v, scale, False, rows=rows)
        oracle.bwd_head(q, k, v, do, scale, False, qrows=rows, krows=[])
        return len(rows)

    # warm up, calibrate on a few rows, then size the sample
    run(list(range(4)))
    t0 = time.perf_counter()
    run(list(range(32)))
    per_row = (time.perf_counter() - t0) / 32
    R = int(max(16, min(N, seconds_target / max(per_row, 1e-9))))
    rows = list(range(R))
    for _ in range(warmup):
        run(rows)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        run(rows)
        times.append(time.perf_counter() - t0)
    # algorithmic FLOPs of the sample, same convention as the GPU figure:
    # forward 4*R*N*d; of the backward only the dQ rows are computed, whose
    # share is S, dP and dS K for those rows: 6*R*N*d
    f = 10.0 * R * N * d
    tf = f / statistics.median(times) / 1e12
    desc = (f"forward + dQ rows of the backward for {R} of {N} query rows of one head "
            f"({WORKLOAD_NAME} workload), fp64, {oracle.num_threads()} threads")
    return tf, oracle.num_threads(), desc, times, f


def reference_arm(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    # seconds of oracle work per step: the whole warm-up + timed run stays
    # within about two and a half minutes
    per_step = min(4.0, max(0.25, 150.0 / max(1, args.steps + args.warmup)))
    tf, threads, desc, times, f = oracle_sample(per_step, steps=args.steps, warmup=args.warmup)
    ms = statistics.median(times) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME + " (bf16 inputs)", "sample": desc},
        "cpu_baseline": oracle_fields(tf, threads, desc),
        "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        import torch

        # nvidia-smi numbers GPUs without regard to CUDA_VISIBLE_DEVICES, so the
        # sampled GPU is named by its UUID where torch reports one
        uuid = getattr(torch.cuda.get_device_properties(gpu_index), "uuid", None)
        uuid = None if uuid is None else str(uuid)
        self.ids = [str(gpu_index)]
        if uuid:
            self.ids.insert(0, uuid if uuid.startswith("GPU-") else f"GPU-{uuid}")
        self.gpu = None
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"fa_clocks_{gpu_index}_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        return self.start()

    def __exit__(self, *exc):
        self.stop()

    def start(self):
        for gpu in self.ids:  # the UUID first; the index if nvidia-smi refuses it
            try:
                self.fh = open(self.path, "w")
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={gpu}", f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=self.fh, stderr=subprocess.DEVNULL)
                time.sleep(0.3)
            except Exception:
                self.proc = None
            if self.proc is not None and self.proc.poll() is None:
                self.gpu = gpu
                return self
            self.proc = None
            self.fh.close()
        return self

    def stop(self):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "gpu": self.gpu}


def kernel_rates(fa, shape, causal, flush, stream, reps=5, warmup=2, fwd=True, bwd=True):
    """Median forward-kernel and backward-main-kernel times (the library's
    CUDA events on the launch stream, L2 flushed before every step) of one
    shape; the step each rep runs is fa_fwd (with its workspace) then fa_bwd.
    Returns dict of ms and TFLOP/s."""
    import torch

    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N, d = shape["B"], shape["H"], shape["N"], shape["d"]
    dev = flush.device
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t.to(dev) for t in attention_inputs(B, H, N, d, seed=1))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = fa.workspace_for(q)
    wsf = fa.fwd_workspace_for(q, causal)
    f_fwd, f_bwd = flops(B, H, N, d, causal)
    fwd_ms, bwd_ms = [], []
    for i in range(warmup + reps):
        flush.zero_()
        fa.fa_timing_enable(i >= warmup)
        fa.fa_fwd(q, k, v, o, lse, scale, causal, wsf)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale, causal, ws)
        if i >= warmup:
            fwd_ms.append(fa.fa_timing_last_ms(fa.KERNEL_FWD))
            bwd_ms.append(fa.fa_timing_last_ms(fa.KERNEL_BWD_MAIN))
    fa.fa_timing_enable(False)
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status")
    fm, bm = statistics.median(fwd_ms), statistics.median(bwd_ms)
    out = {"workload": f"B{B} H{H} N{N} d{d} {'causal' if causal else 'non-causal'}"}
    if fwd:
        out.update(fwd_ms=fm, fwd_tflops=f_fwd / fm / 1e9)
    if bwd:
        out.update(bwd_main_ms=bm, bwd_main_tflops=f_bwd / bm / 1e9)
    del q, k, v, do, o, lse, dq, dk, dv, ws, wsf
    return out


def native_arm(args):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N, d = WORKLOAD["B"], WORKLOAD["H"], WORKLOAD["N"], WORKLOAD["d"]
    scale = 1.0 / math.sqrt(d)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
            torch.cuda.synchronize()

    # each rank: its own replica batch (different seed per rank)
    q, k, v, do = attention_inputs(B, H, N, d, seed=replica_seed(rank))
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    ws = fa.workspace_for(qd)
    wsf = {c: fa.fwd_workspace_for(qd, c) for c in (False, True)}
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 129 MB L2
    stream = torch.cuda.current_stream()

    def step(causal):
        fa.fa_fwd(qd, kd, vd, o, lse, scale, causal, wsf[causal])
        fa.fa_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, scale, causal, ws)

    def timed(causal, steps, warmup, kernel_times=False):
        for _ in range(warmup):
            step(causal)
        if fa.fa_last_device_status() != fa.FA_OK:
            raise RuntimeError("device status after warm-up")
        fa.fa_timing_enable(kernel_times)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        fwd_ms, bwd_ms = [], []
        barrier()
        launches0 = fa.fa_launch_count()
        wall0 = time.perf_counter()
        for i in range(steps):
            flush.zero_()  # L2 flush between steps, outside the step's events
            starts[i].record(stream)
            step(causal)
            ends[i].record(stream)
            if kernel_times:
                fwd_ms.append(fa.fa_timing_last_ms(fa.KERNEL_FWD))
                bwd_ms.append(fa.fa_timing_last_ms(fa.KERNEL_BWD_MAIN))
        barrier()
        wall = time.perf_counter() - wall0
        launches = fa.fa_launch_count() - launches0
        fa.fa_timing_enable(False)
        status = fa.fa_last_device_status()
        if status != fa.FA_OK:
            raise RuntimeError(f"device status {fa.status_string(status)}")
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return step_ms, fwd_ms, bwd_ms, wall, launches

    # headline: non-causal, with per-kernel events.  Clocks are sampled from
    # here to the end of the last GPU leg.
    clocks = ClockSampler(local).start()
    step_ms, fwd_ms, bwd_ms, wall, launches = timed(False, args.steps, args.warmup,
                                                     kernel_times=True)
    mean_ms = max_over_ranks(statistics.mean(step_ms), dev)
    f_fwd, f_bwd = flops(B, H, N, d, False)
    value = job_tflops(f_fwd + f_bwd, world, mean_ms)
    fwd_med, bwd_med = statistics.median(fwd_ms), statistics.median(bwd_ms)
    fwd_tf = f_fwd / (fwd_med * 1e-3) / 1e12
    bwd_main_tf = f_bwd / (bwd_med * 1e-3) / 1e12

    # causal variant of the same shape: its forward is the B1 H16 N32768
    # causal long-context forward
    c_ms, c_fwd, c_bwd, _, _ = timed(True, max(3, args.steps // 2), 2, kernel_times=True)
    cf_fwd, cf_bwd = flops(B, H, N, d, True)
    causal_extra = {
        "workload": "attention fwd+bwd B1 H16 N32768 d128 causal",
        "step_tflops": (cf_fwd + cf_bwd) / (statistics.mean(c_ms) * 1e-3) / 1e12,
        "fwd_tflops": cf_fwd / (statistics.median(c_fwd) * 1e-3) / 1e12,
        "fwd_ms": statistics.median(c_fwd),
        "bwd_main_tflops": cf_bwd / (statistics.median(c_bwd) * 1e-3) / 1e12,
        "bwd_main_ms": statistics.median(c_bwd),
    }

    # End to end through the public calls: every step copies its own inputs
    # Q, K, V, dO from pinned host memory and its gradients dQ, dK, dV back.
    # Two forms are timed.  Serial: copies and kernels one after another on
    # one stream.  Pipelined (the reported `e2e`): device tensors are double
    # buffered and the copies run on their own streams (one per direction),
    # so step k+1's inputs arrive and step k-1's gradients leave while step
    # k's kernels run, as a training loop that prefetches its next batch.
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    hdq, hdk, hdv = (torch.empty_like(t).pin_memory() for t in (q, q, q))
    # the pipeline's fill (first H2D) and drain (last D2H) are inside the timed
    # region and amortised over these steps
    e2e_steps = max(10, args.steps)

    def e2e_serial_step():
        qd.copy_(hq, non_blocking=True)
        kd.copy_(hk, non_blocking=True)
        vd.copy_(hv, non_blocking=True)
        dod.copy_(hdo, non_blocking=True)
        step(False)
        hdq.copy_(dq, non_blocking=True)
        hdk.copy_(dk, non_blocking=True)
        hdv.copy_(dv, non_blocking=True)

    def timed_e2e(run_steps, prepare=None, finish=None):
        for i in range(2):
            run_steps(i)
        if finish is not None:
            finish()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if prepare is not None:
            prepare(e0)
        for i in range(e2e_steps):
            run_steps(i)
        if finish is not None:
            finish()
        e1.record(stream)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)

    e2e_serial_ms = timed_e2e(lambda i: e2e_serial_step())

    # one copy stream per direction (two per direction measured no faster)
    h2d = [torch.cuda.Stream(dev)]
    d2h = [torch.cuda.Stream(dev)]
    slots = [dict(q=torch.empty_like(qd), k=torch.empty_like(qd), v=torch.empty_like(qd),
                  do=torch.empty_like(qd), dq=torch.empty_like(qd), dk=torch.empty_like(qd),
                  dv=torch.empty_like(qd), in_ready=[torch.cuda.Event() for _ in h2d],
                  in_free=torch.cuda.Event(), out_ready=torch.cuda.Event(),
                  out_free=[torch.cuda.Event() for _ in d2h], used=False)
             for _ in range(2)]

    def pipelined_step(i):
        sl = slots[i % 2]
        ins = ((sl["q"], hq), (sl["k"], hk), (sl["v"], hv), (sl["do"], hdo))
        for c, cs in enumerate(h2d):
            with torch.cuda.stream(cs):
                if sl["used"]:
                    cs.wait_event(sl["in_free"])
                for dst, src in ins[c::len(h2d)]:
                    dst.copy_(src, non_blocking=True)
                sl["in_ready"][c].record(cs)
            stream.wait_event(sl["in_ready"][c])
        if sl["used"]:
            for ev in sl["out_free"]:
                stream.wait_event(ev)
        fa.fa_fwd(sl["q"], sl["k"], sl["v"], o, lse, scale, False, wsf[False])
        fa.fa_bwd(sl["q"], sl["k"], sl["v"], o, lse, sl["do"], sl["dq"], sl["dk"], sl["dv"], scale,
                  False, ws)
        sl["in_free"].record(stream)
        sl["out_ready"].record(stream)
        outs = ((hdq, sl["dq"]), (hdk, sl["dk"]), (hdv, sl["dv"]))
        for c, cs in enumerate(d2h):
            with torch.cuda.stream(cs):
                cs.wait_event(sl["out_ready"])
                for dst, src in outs[c::len(d2h)]:
                    dst.copy_(src, non_blocking=True)
                sl["out_free"][c].record(cs)
        sl["used"] = True

    def pipelined_prepare(e0):
        for cs in h2d:  # the first copies start inside the timed region
            cs.wait_event(e0)

    def pipelined_finish():
        for sl in slots:  # the last gradients are back on the host
            for ev in sl["out_free"]:
                stream.wait_event(ev)

    e2e_ms = timed_e2e(pipelined_step, pipelined_prepare, pipelined_finish)
    e2e_value = job_tflops(f_fwd + f_bwd, world, e2e_ms)
    e2e_serial_value = job_tflops(f_fwd + f_bwd, world, e2e_serial_ms)
    tensor_bytes = q.numel() * q.element_size()
    del slots, hq, hk, hv, hdo, hdq, hdk, hdv, qd, kd, vd, dod, o, lse, dq, dk, dv, ws, wsf
    torch.cuda.empty_cache()

    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = peaks.get("bf16_tflops")
    peak_note = "measured burst cuBLAS bf16 (MEASURED_PEAKS.json bf16_tflops)"
    if peak is None:
        peak, peak_note = 1900.0, "fallback 1.9 PFLOP/s bf16"

    # the seconds-long power-capped cuBLAS figure, for kernels timed inside
    # steps long enough to reach the power cap (reported beside `frac`)
    peak_sustained = peaks.get("bf16_tflops_sustained")

    def roofline(kernel, achieved, **extra):
        r = {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak,
             "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_note}
        if peak_sustained:
            r.update(peak_sustained=peak_sustained, frac_of_sustained=achieved / peak_sustained)
        r.update(extra)
        return r

    # The B2 H16 N8192 causal backward, kernel events.
    bwd_causal = kernel_rates(fa, BWD_CAUSAL, True, flush, stream, fwd=False)
    # The B2 H16 N4096 step (non-causal) and the other entry points on it.
    small = kernel_rates(fa, SMALL, False, flush, stream)
    sB, sH, sN, sd = SMALL["B"], SMALL["H"], SMALL["N"], SMALL["d"]
    s_fwd, s_bwd = flops(sB, sH, sN, sd, False)
    sq, sk, sv, sdo = (t.to(dev) for t in attention_inputs(sB, sH, sN, sd, seed=2))
    so, slse = torch.empty_like(sq), torch.empty((sB, sH, sN), dtype=torch.float32, device=dev)
    sdq, sdk, sdv = torch.empty_like(sq), torch.empty_like(sq), torch.empty_like(sq)
    fa.fa_fwd(sq, sk, sv, so, slse, 1.0 / math.sqrt(sd), False, fa.fwd_workspace_for(sq, False))

    # The deterministic backward (all three of its kernels), L2 flushed
    # before each launch.
    ws_det = fa.workspace_for(sq, deterministic=True)
    det_ms = []
    for i in range(3 + 5):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fa.fa_bwd_deterministic(sq, sk, sv, so, slse, sdo, sdq, sdk, sdv, 1.0 / math.sqrt(sd),
                                False, ws_det)
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            det_ms.append(e0.elapsed_time(e1))
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status after the deterministic backward")
    del ws_det
    det_ms_med = statistics.median(det_ms)
    deterministic_extra = {"bwd_tflops": s_bwd / (det_ms_med * 1e-3) / 1e12, "bwd_ms": det_ms_med,
                           "workload": "B2 H16 N4096 d128 non-causal",
                           "note": "fa_bwd_deterministic, all kernels"}

    # The FP8 forward (rotation + e4m3 preparation, then the kernel); the
    # kernel alone from the library's events.
    ws8 = torch.empty(fa.fa_fwd_fp8_workspace_bytes(sB, sH, sN, sd), dtype=torch.uint8, device=dev)
    o8, lse8 = torch.empty_like(sq), torch.empty_like(slse)
    call_ms, kern_ms = [], []
    fa.fa_timing_enable(True)
    for i in range(3 + 5):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fa.fa_fwd_fp8(sq, sk, sv, o8, lse8, 1.0 / math.sqrt(sd), False, True, ws8)
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            call_ms.append(e0.elapsed_time(e1))
            kern_ms.append(fa.fa_timing_last_ms(fa.KERNEL_FWD))
    fa.fa_timing_enable(False)
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status after the FP8 forward")
    del ws8
    fp8_extra = {"call_tflops": s_fwd / (statistics.median(call_ms) * 1e-3) / 1e12,
                 "kernel_tflops": s_fwd / (statistics.median(kern_ms) * 1e-3) / 1e12,
                 "workload": "B2 H16 N4096 d128 non-causal",
                 "note": "fa_fwd_fp8 (rotate=1, e4m3): call = preparation + kernel"}

    # The CTA-pair forward (fa_fwd_2cta), kernel events.
    pair_ms = []
    fa.fa_timing_enable(True)
    for i in range(3 + 5):
        flush.zero_()
        fa.fa_fwd_2cta(sq, sk, sv, o8, lse8, 1.0 / math.sqrt(sd), False)
        if i >= 3:
            pair_ms.append(fa.fa_timing_last_ms(fa.KERNEL_FWD))
    fa.fa_timing_enable(False)
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status after the CTA-pair forward")
    two_cta_extra = {"kernel_tflops": s_fwd / (statistics.median(pair_ms) * 1e-3) / 1e12,
                     "workload": "B2 H16 N4096 d128 non-causal",
                     "note": "fa_fwd_2cta: CTA pairs sharing M = 256 products"}

    # The CTA-pair backward (fa_bwd_2cta), main kernel events.
    ws2 = fa.workspace_for(sq)
    pair_bwd_ms = []
    fa.fa_timing_enable(True)
    for i in range(3 + 5):
        flush.zero_()
        fa.fa_bwd_2cta(sq, sk, sv, so, slse, sdo, sdq, sdk, sdv, 1.0 / math.sqrt(sd), False, ws2)
        if i >= 3:
            pair_bwd_ms.append(fa.fa_timing_last_ms(fa.KERNEL_BWD_MAIN))
    fa.fa_timing_enable(False)
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status after the CTA-pair backward")
    del ws2
    pb = s_bwd / (statistics.median(pair_bwd_ms) * 1e-3) / 1e12
    two_cta_bwd_extra = {"kernel_tflops": pb, "workload": "B2 H16 N4096 d128 non-causal",
                         "roofline": roofline("fa_bwd_pair_kernel", pb),
                         "note": "fa_bwd_2cta: CTA pairs sharing cta_group::2 products, dQ "
                                 "added once per 256 keys"}
    del sq, sk, sv, sdo, so, slse, sdq, sdk, sdv, o8, lse8
    clocks.stop()
    clk = clocks.summary()

    traffic_ok = (NCU_TRAFFIC["bytes"] is not None and
                  kernel_sources_sha256() == NCU_TRAFFIC["sources_sha256"])
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": mean_ms,
        # this rank's step times (the headline uses the mean, max over ranks)
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                    "max": max(step_ms)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "B": B, "H": H, "N": N, "d": d, "causal": False,
                   "global_batch": B * world, "seq_len": N,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (256 MiB write outside the step events); "
                         "each input tensor (134 MB) is also larger than L2"},
        "pct_of_2250_tflops": 100.0 * value / PAGES_PEAK_TFLOPS,
        "fwd_tflops": fwd_tf,
        "bwd_main_tflops": bwd_main_tf,
        "fwd_ms": fwd_med,
        "bwd_main_ms": bwd_med,
        "fwd_pct_of_2250_tflops": 100.0 * fwd_tf / PAGES_PEAK_TFLOPS,
        "bwd_main_pct_of_2250_tflops": 100.0 * bwd_main_tf / PAGES_PEAK_TFLOPS,
        "causal": causal_extra,
        "bwd_b2h16n8192_causal": {
            **bwd_causal,
            "pct_of_2250_tflops": 100.0 * bwd_causal["bwd_main_tflops"] / PAGES_PEAK_TFLOPS,
            "roofline": roofline("fa_bwd_kernel<128>", bwd_causal["bwd_main_tflops"])},
        "b2h16n4096": {**small, "roofline_bwd": roofline("fa_bwd_kernel<128>",
                                                         small["bwd_main_tflops"])},
        "deterministic": deterministic_extra,
        "fp8_forward": fp8_extra,
        "two_cta_forward": two_cta_extra,
        "two_cta_backward": two_cta_bwd_extra,
        "roofline": roofline(
            "fa_bwd_kernel<128>", bwd_main_tf,
            traffic=NCU_TRAFFIC["bytes"] if traffic_ok else None,
            traffic_unit="bytes per launch (ncu, cold cache; " + NCU_TRAFFIC["captured"] + ")",
            algorithmic_bytes=(4 * 2 * B * H * N * d  # Q, K, V, dO read
                               + 2 * 2 * B * H * N * d  # dK, dV written
                               + 2 * 4 * B * H * N * d  # fp32 dQ accumulator read and written
                               + 2 * 4 * B * H * N)),  # LSE, D read
        "roofline_fwd": roofline("fa_fwd_kernel<128>", fwd_tf),
        "roofline_fwd_causal": roofline("fa_fwd_kernel<128>", causal_extra["fwd_tflops"]),
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": 4 * tensor_bytes, "d2h_bytes_per_step": 3 * tensor_bytes,
                "copies": "one stream per direction, overlapped with the kernels (double buffered)",
                "steps": e2e_steps,
                "serial": {"value": e2e_serial_value, "ms_per_step": e2e_serial_ms}},
        # the library's own launch counter across the timed steps: fa_fwd
        # (1, or 2 when it splits its last partial round) + fa_bwd (3)
        "gpu_launches": launches,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        tf, threads, desc, _, _ = oracle_sample(12.0, steps=1)
        line["cpu_baseline"] = oracle_fields(tf, threads, desc)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def sweep_arm(args):
    """Kernel-level throughput over the fixed-token sweep: forward kernel and
    backward main kernel, CUDA events recorded by the library around each
    launch, median of `steps` launches after `warmup`, L2 flushed in between."""
    import torch

    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    dev = torch.device("cuda", 0)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    steps, warmup = max(3, args.steps), max(3, args.warmup)
    for d in (128, 64):
        for N in (1024, 2048, 4096, 8192, 16384, 32768):
            B, H = 32768 // N, 16
            scale = 1.0 / math.sqrt(d)
            q, k, v, do = (t.to(dev) for t in attention_inputs(B, H, N, d, seed=0))
            o = torch.empty_like(q)
            lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            ws = fa.workspace_for(q)
            wsf = {c: fa.fwd_workspace_for(q, c) for c in (False, True)}
            for causal in (False, True):
                f_fwd, f_bwd = flops(B, H, N, d, causal)
                fwd_ms, bwd_ms = [], []
                for i in range(warmup + steps):
                    flush.zero_()
                    fa.fa_timing_enable(i >= warmup)
                    fa.fa_fwd(q, k, v, o, lse, scale, causal, wsf[causal])
                    fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale, causal, ws)
                    if i >= warmup:
                        fwd_ms.append(fa.fa_timing_last_ms(fa.KERNEL_FWD))
                        bwd_ms.append(fa.fa_timing_last_ms(fa.KERNEL_BWD_MAIN))
                fa.fa_timing_enable(False)
                if fa.fa_last_device_status() != fa.FA_OK:
                    raise RuntimeError("device status")
                fm, bm = statistics.median(fwd_ms), statistics.median(bwd_ms)
                print(json.dumps({"sweep": True, "B": B, "H": H, "N": N, "d": d, "causal": causal,
                                  "fwd_ms": fm, "fwd_tflops": f_fwd / fm / 1e9,
                                  "fwd_pct_of_2250": 100 * f_fwd / fm / 1e9 / PAGES_PEAK_TFLOPS,
                                  "bwd_main_ms": bm, "bwd_main_tflops": f_bwd / bm / 1e9,
                                  "bwd_pct_of_2250": 100 * f_bwd / bm / 1e9 / PAGES_PEAK_TFLOPS}),
                      flush=True)
            del q, k, v, do, o, lse, dq, dk, dv, ws, wsf


def oracle_configs_arm(args):
    """The oracle's own cost on the coverage the parity tests give it, per
    configuration: B1 H2 N128 d64 in full (fwd + bwd, both masks); head 0 of
    B2 H16 N4096 d128 in full (fwd); 512 sampled rows of head 0 of B1 H16
    N32768 d128 causal (fwd); 256 sampled rows of head 0 of B2 H16 N8192 d128
    causal (fwd + the dQ rows of the bwd).  Algorithmic FLOPs as on the GPU
    (causal rows count the keys they attend to).  Host cores only."""
    import numpy as np

    import oracle
    from exact_attention_98_gb300.inputs import attention_inputs, sampled_rows

    def head0(B, H, N, d, causal_seed=0):
        q, k, v, do = attention_inputs(B, H, N, d, seed=causal_seed)
        return tuple(t.double().numpy()[0, 0] for t in (q, k, v, do))

    def line(name, flop, secs, extra):
        print(json.dumps({"oracle_config": name, "gflop": flop / 1e9, "seconds": secs,
                          "gflop_per_s": flop / secs / 1e9, "threads": oracle.num_threads(),
                          "cpu_model": cpu_model(), "nproc": os.cpu_count(), **extra}), flush=True)

    # config 1 in full, both masks
    q, k, v, do = attention_inputs(1, 2, 128, 64, seed=0)
    q, k, v, do = (t.double().numpy() for t in (q, k, v, do))
    t0 = time.perf_counter()
    f = 0.0
    for causal in (False, True):
        oracle.fwd(q, k, v, 0.125, causal)
        oracle.bwd(q, k, v, do, 0.125, causal)
        ff, fb = flops(1, 2, 128, 64, causal)
        f += ff + fb
    line("1: B1 H2 N128 d64, fwd+bwd, both masks, full", f, time.perf_counter() - t0, {})

    # config 2, head 0 in full (forward)
    N, d = 4096, 128
    q, k, v, _ = head0(2, 16, N, d)
    t0 = time.perf_counter()
    oracle.fwd_head(q, k, v, 1.0 / math.sqrt(d), False)
    secs = time.perf_counter() - t0
    line("2: B2 H16 N4096 d128, head 0 in full, fwd", 4.0 * N * N * d, secs,
         {"projected_full_fwd_s": secs * 2 * 16})

    # config 3, sampled rows (causal forward)
    N = 32768
    q, k, v, _ = head0(1, 16, N, d)
    rows = sorted(set(int(x) for x in np.linspace(0, N - 1, 512)))
    t0 = time.perf_counter()
    oracle.fwd_head(q, k, v, 1.0 / math.sqrt(d), True, rows=rows)
    secs = time.perf_counter() - t0
    f = sum(4.0 * (r + 1) * d for r in rows)
    line("3: B1 H16 N32768 d128 causal, 512 rows of head 0, fwd", f, secs,
         {"projected_full_fwd_s": secs * (4.0 * 16 * N * N * d / 2) / f})

    # config 4, sampled rows (causal: forward and the dQ rows of the backward)
    N = 8192
    q, k, v, do = head0(2, 16, N, d)
    rows = sorted(set(int(x) for x in np.linspace(0, N - 1, 256)))
    t0 = time.perf_counter()
    oracle.fwd_head(q, k, v, 1.0 / math.sqrt(d), True, rows=rows)
    oracle.bwd_head(q, k, v, do, 1.0 / math.sqrt(d), True, qrows=rows, krows=[])
    secs = time.perf_counter() - t0
    f = sum(10.0 * (r + 1) * d for r in rows)
    line("4: B2 H16 N8192 d128 causal, 256 rows of head 0, fwd + dQ rows of bwd", f, secs,
         {"projected_full_fwd_bwd_s": secs * (14.0 * 2 * 16 * N * N * d / 2) / f})


def main():
    args = parse()
    if args.oracle_configs:
        oracle_configs_arm(args)
        return
    if args.loop:
        loop_arm(args)
        return
    if args.sweep:
        sweep_arm(args)
        return
    if args.impl == "reference":
        reference_arm(args)
    else:
        native_arm(args)


if __name__ == "__main__":
    main()
