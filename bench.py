"""Benchmark of the fused dynamic-LoRA linear on one or more GB300s.

One step = one fused forward of the Wan2.1-1.3B-shaped stacked q/k/v LoRA linear
(T = 32760 tokens, in = 1536, out = 3 x 1536 column groups, rank 32 per group, bf16,
no bias) over one batch of synthetic input, through the C ABI.  The metric is
TFLOP/s with FLOP = 2 T (in * out + sum_g r_g (in + out_g)), reported beside the
fraction of the measured BF16 tensor peak and the overhead over a bare base GEMM of
the same shape (cuBLAS through torch, and this library's own kernel with no adapter).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fused|reference]

N > 1 is launched by torchrun, one rank per GPU: every rank runs its own batch
(token-local op, no collective on the data path; weak scaling).  Rank 0 prints one
JSON line.  ``--impl reference`` times the CPU FP64 oracle on the host cores on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = ("wan2.1-1.3b stacked qkv: T=32760 (21x30x52 latent), in=1536, out=3x1536 as 3 "
            "column groups, rank=32 per group, bf16 X/W/A/B, alpha=32, strength=1, scale=1, no bias")
METRIC = "fused LoRA linear TFLOP/s & % BF16 roofline; overhead vs bare base GEMM"


def flops_of(lin) -> float:
    T, K = lin.X.rows, lin.X.cols
    out = lin.W.rows
    G = lin.groups
    og = out // G
    return 2.0 * T * (K * out + sum(p.rank * (K + og) for p in lin.patches))


# Kernels of this library per fused step on the bench workload: rank_pack_kernel (packs the
# adapters' A rows for the rank items, clears the row-block flags) and tc_fused_fwd_kernel.
LAUNCHES_PER_STEP = 2


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


def measured_sustained_bf16():
    """cuBLAS bf16 rate held for seconds under the power cap (the default timed loop runs
    about 0.3 s of back-to-back launches, long enough for the cap to act), or None."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        return json.load(f).get("bf16_tflops_sustained")


def captured_traffic():
    """DRAM bytes per launch of the fused kernel from the committed ncu summary, or None
    when the kernel source changed since that capture."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "tc_fused_fwd_c1_wan_qkv.md")
    src = os.path.join(ROOT, "weight_patches_gb300", "csrc", "wp_tc_fwd.cu")
    try:
        text = open(prof).read()
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    vals = dict(line.strip().split(": ", 1) for line in text.splitlines()
                if line.strip().startswith(("traffic_bytes_per_launch", "kernel_source_sha256_16")))
    if vals.get("kernel_source_sha256_16") != h:
        return None
    return int(vals["traffic_bytes_per_launch"])


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1])); smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip() == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------- GPU arm
def run_fused(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)

    import weight_patches_gb300 as wpg
    from weight_patches_gb300 import data_parallel as wdp
    import workloads

    lin = workloads.config1("full")
    X = lin.X.torch_cpu().to(dev)
    W = lin.W.torch_cpu().to(dev)
    ads = [wpg.Adapter(p.A.torch_cpu().to(dev), p.B.torch_cpu().to(dev), p.alpha, p.strength)
           for p in lin.patches]
    T, N = X.shape[0], W.shape[0]
    Y = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
    Y0 = torch.empty_like(Y)
    flops = flops_of(lin)
    stream = torch.cuda.current_stream(dev)

    def step():
        wpg.lora_linear_fwd_grouped(X, W, None, ads, lin.request_scale, out=Y)

    def barrier():
        if ws > 1:
            dist.barrier()

    def timed(fn, k, w):
        for _ in range(w):
            fn()
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        ms = e0.elapsed_time(e1)
        if ws > 1:
            ms = wdp.max_over_ranks(ms, device=dev)      # the whole job waits for its slowest rank
        return ms

    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    clocks = ClockSampler(vis[local] if local < len(vis) else str(local))
    clocks.start()
    time.sleep(0.3)
    total_ms = timed(step, args.steps, args.warmup)
    clk = clocks.stop()
    assert wpg.lora_device_status() == 0, "device wait timed out"
    ms_step = total_ms / args.steps

    # bare base GEMM of the same shape: cuBLAS via torch, and this library with no adapter
    kb = max(20, min(args.steps, 200))
    Wt = W.t()
    base_ms = timed(lambda: torch.matmul(X, Wt, out=Y0), kb, 5) / kb
    own_base_ms = timed(lambda: wpg.lora_linear_fwd(X, W, None, [], out=Y0), kb, 5) / kb

    # end to end through the public API with host buffers: pinned X in, Y out; the
    # host-buffer entry point moves row chunks in and out while it computes
    Xh = X.cpu().pin_memory()
    Yh = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    ws_host = torch.empty(wpg.lora_workspace_size(wpg.WP_OP_FWD_HOST, Xh, W, ads), dtype=torch.uint8,
                          device=dev)

    def e2e_step():
        wpg.lora_linear_fwd_host(Xh, W, None, ads, lin.request_scale, out=Yh, grouped=True,
                                 workspace=ws_host)

    ke = max(5, min(args.steps, 50))
    e2e_ms = timed(e2e_step, ke, 3) / ke
    h2d = X.numel() * X.element_size()
    d2h = Y.numel() * Y.element_size()

    peak, hbm, peak_kind = measured_peaks()
    sustained = measured_sustained_bf16()
    tflops = ws * flops / (ms_step * 1e-3) / 1e12
    per_launch_tflops = flops / (ms_step * 1e-3) / 1e12
    out = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T, "in": X.shape[1], "out": N, "groups": lin.groups,
                   "rank_per_group": lin.patches[0].rank, "gflop_per_step": round(flops / 1e9, 2),
                   "l2": "inputs larger than L2 (X 101 MB + W 14 MB + Y 302 MB per step > 129 MB)",
                   "parallelism": f"replicas x{ws} (token-local, no collective)"},
        "roofline": {"bound": "tensor", "achieved": round(per_launch_tflops, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(per_launch_tflops / peak, 4), "traffic": captured_traffic(),
                     "peak_source": f"{peak_kind} bf16 burst",
                     "frac_of_sustained": (round(per_launch_tflops / sustained, 4) if sustained else None),
                     "timing": "CUDA events over the timed steps; a step is the rank-operand pack "
                               "kernel plus the fused kernel, so this slightly understates the fused "
                               "kernel's own rate"},
        "overhead": {"vs_cublas_base_gemm": round(ms_step / base_ms - 1.0, 4),
                     "vs_own_base_kernel": round(ms_step / own_base_ms - 1.0, 4),
                     "cublas_base_ms": round(base_ms, 5), "own_base_ms": round(own_base_ms, 5)},
        "e2e": {"value": round(ws * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": args.steps * LAUNCHES_PER_STEP,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(lin, budget_s=args.cpu_seconds)
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


# ----------------------------------------------------------------------- CPU oracle
def cpu_baseline(lin, budget_s: float = 12.0, rows_per_call: int = 2048):
    """Time the FP64 oracle (as it stands) on a bounded sample of token rows."""
    from oracle import lora as olora
    T = lin.X.rows
    rng = np.random.default_rng(0)
    done_rows, t_total, calls = 0, 0.0, 0
    while t_total < budget_s and calls < 64:
        r0 = int(rng.integers(0, max(1, T - rows_per_call)))
        rows = np.arange(r0, min(T, r0 + rows_per_call))
        t0 = time.perf_counter()
        olora.reference_output(lin, rows)
        t_total += time.perf_counter() - t0
        done_rows += len(rows)
        calls += 1
    flops = flops_of(lin) * done_rows / T
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{done_rows} of {T} token rows ({calls} calls of {rows_per_call} rows), FP64 numpy, "
                      f"{t_total:.1f} s"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import workloads
    lin = workloads.config1("full")
    T = lin.X.rows
    from oracle import lora as olora
    rows_per_step = 512
    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        olora.reference_output(lin, np.arange(0, rows_per_step))
    t_steps = []
    for _ in range(args.steps):
        r0 = int(rng.integers(0, T - rows_per_step))
        t0 = time.perf_counter()
        olora.reference_output(lin, np.arange(r0, r0 + rows_per_step))
        t_steps.append(time.perf_counter() - t0)
    total = sum(t_steps)
    flops = flops_of(lin) * rows_per_step / T * len(t_steps)
    value = flops / total / 1e12
    out = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(t_steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{rows_per_step} token rows per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": f"{rows_per_step} of {T} token rows per step"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="fused", choices=["fused", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_fused(args)


if __name__ == "__main__":
    main()
