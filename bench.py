"""Benchmark of the fused dynamic-LoRA linear on one or more GB300s.

One step = one fused forward of the Wan2.1-1.3B-shaped stacked q/k/v LoRA linear
(T = 32760 tokens, in = 1536, out = 3 x 1536 column groups, rank 32 per group, bf16,
no bias) over one batch of synthetic input, through the C ABI.  The metric is
TFLOP/s with FLOP = 2 T (in * out + sum_g r_g (in + out_g)), reported beside the
fraction of the measured BF16 tensor peak and the overhead over a bare base GEMM of
the same shape (cuBLAS through torch, and this library's own kernel with no adapter).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fused|reference]

N > 1 runs one rank per GPU under torchrun (bench.py re-launches itself that way when it
is started without a torchrun environment): every rank runs its own batch (token-local op,
no collective on the data path; weak scaling).  Rank 0 prints one JSON line.  At N = 1 the
line also carries ``per_config``: every other workload of the library timed the same way
(forward and backward of each, the dense patch), each with its work, time, roofline
fraction, overheads and the clocks seen while it ran.  ``--impl reference`` times the CPU
FP64 oracle on the host cores on a bounded sample of the same workload (rank 0 only).
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


def bench_config(ws: int) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    import workloads
    f = workloads.FULL[1]
    return {"workload": WORKLOAD, "T": f["T"], "in": f["d_in"], "out": f["groups"] * f["d_out"],
            "groups": f["groups"], "rank_per_group": f["rank"],
            "gflop_per_step": round(2.0 * f["T"] * (f["d_in"] * f["groups"] * f["d_out"] + f["groups"] * f["rank"] *
                                                    (f["d_in"] + f["d_out"])) / 1e9, 2),
            "l2": "inputs larger than L2 (X 101 MB + W 14 MB + Y 302 MB per step > 129 MB)",
            "parallelism": f"replicas x{ws} (token-local, no collective)"}


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
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
            self.rows = []
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        return self.summary()

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and the throttle reasons of the samples taken between
        host times t0 and t1 (all samples when not given)."""
        from datetime import datetime
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in getattr(self, "rows", []):
            try:
                ts = datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                    continue
                sm.append(float(r[2])); smax.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[6:10]):
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

    # the overheads: the fused step, the bare base GEMM of the same shape by cuBLAS (via torch)
    # and this library's kernel with no adapter, each timed the same way (kb steps after the
    # same idle pause), so that no one of them runs in a hotter, power-capped stretch than the
    # others
    kb = max(20, min(args.steps, 50))
    Wt = W.t()
    time.sleep(0.5)
    fused_b_ms = timed(step, kb, 5) / kb
    time.sleep(0.5)
    base_ms = timed(lambda: torch.matmul(X, Wt, out=Y0), kb, 5) / kb
    time.sleep(0.5)
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
        "config": bench_config(ws),
        "roofline": {"bound": "tensor", "achieved": round(per_launch_tflops, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(per_launch_tflops / peak, 4), "traffic": captured_traffic(),
                     "peak_source": f"{peak_kind} bf16 burst",
                     "frac_of_sustained": (round(per_launch_tflops / sustained, 4) if sustained else None),
                     "timing": "CUDA events over the timed steps; a step is the rank-operand pack "
                               "kernel plus the fused kernel, so this slightly understates the fused "
                               "kernel's own rate"},
        "overhead": {"vs_cublas_base_gemm": round(fused_b_ms / base_ms - 1.0, 4),
                     "vs_own_base_kernel": round(fused_b_ms / own_base_ms - 1.0, 4),
                     "fused_ms": round(fused_b_ms, 5), "cublas_base_ms": round(base_ms, 5),
                     "own_base_ms": round(own_base_ms, 5),
                     "timing": f"{kb} steps of each after a 0.5 s idle pause (the same regime for all three)"},
        "e2e": {"value": round(ws * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": args.steps * LAUNCHES_PER_STEP,
        "clocks": clk,
    }
    if ws == 1 and not args.no_per_config:
        del Xh, Yh, ws_host, Y0
        torch.cuda.empty_cache()
        out["per_config"] = per_config(dev, args, peak, hbm)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(lin, budget_s=args.cpu_seconds)
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


# ----------------------------------------------------------------------- other workloads
CASES = ("c0_tiny_fp32", "f32_layer", "wan_qkv_rank128", "c2_ffn_up", "c2_ffn_down", "c3_nf4_gate_up_fwd",
         "c3_nf4_down_fwd", "c3_nf4_gate_up_bwd", "c3_nf4_down_bwd", "c3_swiglu_bwd", "c3_nf4_merge",
         "c3_nf4_gate_up_t1", "c3_nf4_gate_up_t16", "c4_sidecar", "c4_set_weight")


def per_config(dev, args, peak, hbm, only=None):
    """Every workload of the library besides the headline one, timed like it: CUDA events on
    the launching stream around back-to-back calls after warm-up (inputs larger than L2), and
    for the dense patch one call at a time after an L2 flush.  Each entry: its work (GFLOP or
    MB), ms per call, rate, fraction of the measured peak, overheads over cuBLAS's bf16 GEMM of
    the same shape and over this library's kernel without adapters, and the clocks seen."""
    import torch
    import weight_patches_gb300 as wpg
    import workloads

    stream = torch.cuda.current_stream(dev)
    want = lambda name: only is None or name in only
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    marks = {}
    k, w = max(10, min(args.steps, 50)), 5

    def timed(fn, kk=k, ww=w):
        # every measurement starts after the same short idle pause, so that none of them runs
        # in a hotter, power-capped stretch than the fused call it is compared with
        time.sleep(0.3)
        for _ in range(ww):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(kk):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / kk

    def d(mat):
        if mat.kind == "nf4":
            return wpg.NF4Weight(torch.from_numpy(mat.data).to(dev), torch.from_numpy(mat.absmax).to(dev),
                                 mat.rows, mat.cols)
        return mat.torch_cpu().to(dev)

    def ads_of(lin):
        return [wpg.Adapter(d(p.A), d(p.B), p.alpha, p.strength) for p in lin.patches]

    def fwd_flops(lin):
        T, K, N, G = lin.X.rows, lin.X.cols, lin.W.rows, lin.groups
        return 2.0 * T * (K * N + sum(p.rank * (K + N // G) for p in lin.patches))

    out = {}

    def fwd_entry(name, lin, note=""):
        t0 = time.time()
        X, W = d(lin.X), d(lin.W)
        bias = d(lin.bias).reshape(-1) if lin.bias is not None else None
        ads = ads_of(lin)
        N = lin.W.rows
        Y = torch.empty(lin.T, N, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(1, wpg.lora_workspace_size(wpg.WP_OP_FWD_GROUPED if lin.groups > 1 else wpg.WP_OP_FWD,
                                                        X, W, ads)), dtype=torch.uint8, device=dev)
        if lin.groups > 1:
            fn = lambda: wpg.lora_linear_fwd_grouped(X, W, bias, ads, lin.request_scale, out=Y, workspace=ws)
        else:
            fn = lambda: wpg.lora_linear_fwd(X, W, bias, ads, lin.request_scale, out=Y, workspace=ws)
        t_s = time.time()
        ms = timed(fn)
        own = timed(lambda: wpg.lora_linear_fwd(X, W, bias, [], out=Y))
        Wb = W if not isinstance(W, wpg.NF4Weight) else torch.randn(N, lin.X.cols, device=dev).to(torch.bfloat16)
        if bias is not None:
            cub = timed(lambda: torch.addmm(bias, X, Wb.t(), out=Y))
        else:
            cub = timed(lambda: torch.matmul(X, Wb.t(), out=Y))
        t_e = time.time()
        assert wpg.lora_device_status() == 0
        fl = fwd_flops(lin)
        tf = fl / (ms * 1e-3) / 1e12
        out[name] = {"gflop": round(fl / 1e9, 2), "ms": round(ms, 5), "tflops": round(tf, 1),
                     "frac": round(tf / peak, 4), "own_base_ms": round(own, 5), "cublas_base_ms": round(cub, 5),
                     "overhead_vs_cublas": round(ms / cub - 1, 4), "overhead_vs_own_base": round(ms / own - 1, 4),
                     "clocks": None, "setup_s": round(t_s - t0, 1)}
        if note:
            out[name]["note"] = note
        marks[name] = (t_s, t_e)

    def bwd_entry(name, lin):
        t0 = time.time()
        X, W, dY = d(lin.X), d(lin.W), d(lin.dY)
        ads = ads_of(lin)
        ws = torch.empty(wpg.lora_workspace_size(wpg.WP_OP_BWD, X, W, ads), dtype=torch.uint8, device=dev)
        fn = lambda: wpg.lora_linear_bwd(X, W, dY, ads, lin.request_scale, workspace=ws)
        t_s = time.time()
        ms = timed(fn, max(5, k // 2), 3)
        Wb = torch.randn(lin.W.rows, lin.X.cols, device=dev).to(torch.bfloat16)
        dX = torch.empty(lin.T, lin.X.cols, dtype=torch.bfloat16, device=dev)
        cub = timed(lambda: torch.matmul(dY, Wb, out=dX))
        t_e = time.time()
        assert wpg.lora_device_status() == 0
        T, K, N, G = lin.X.rows, lin.X.cols, lin.W.rows, lin.groups
        fl = 2.0 * T * (K * N + sum(2 * p.rank * (N // G + K) for p in lin.patches))
        tf = fl / (ms * 1e-3) / 1e12
        out[name] = {"gflop": round(fl / 1e9, 2), "ms": round(ms, 5), "tflops": round(tf, 1),
                     "frac": round(tf / peak, 4), "cublas_dX_gemm_ms": round(cub, 5),
                     "work": "dX, dA, dB (FLOP: 2T(in out + sum_g 2 r_g (out_g + in)))",
                     "clocks": None, "setup_s": round(t_s - t0, 1)}
        marks[name] = (t_s, t_e)

    ffma_peak = device_sm_count(dev) * 128 * 2 * 2.07e9 / 1e12

    def f32_entry(name, lin, note):
        X0, W0, b0 = d(lin.X), d(lin.W), d(lin.bias).reshape(-1)
        ads0 = ads_of(lin)
        Y0 = torch.empty(lin.T, lin.W.rows, dtype=torch.float32, device=dev)
        ws0 = torch.empty(max(1, wpg.lora_workspace_size(wpg.WP_OP_FWD, X0, W0, ads0)), dtype=torch.uint8,
                          device=dev)
        t_s = time.time()
        ms0 = timed(lambda: wpg.lora_linear_fwd(X0, W0, b0, ads0, lin.request_scale, out=Y0, workspace=ws0),
                    max(k, 20), 10)
        marks[name] = (t_s, time.time())
        fl0 = fwd_flops(lin)
        tf = fl0 / (ms0 * 1e-3) / 1e12
        out[name] = {"gflop": round(fl0 / 1e9, 5), "us": round(ms0 * 1e3, 2), "tflops": round(tf, 3),
                     "bound": "alu (fp32 FFMA)", "frac": round(tf / ffma_peak, 4), "note": note,
                     "peak": f"{ffma_peak:.1f} TFLOP/s fp32 FFMA (SMs x 128 lanes x 2 x 2.07 GHz)"}

    if want("c0_tiny_fp32"):
        f32_entry("c0_tiny_fp32", workloads.config0(), "the all-FP32 layer of the tiny workload: launch-bound")
    if want("f32_layer"):
        rng = np.random.default_rng(21)
        T, K, N, r = 4096, 1024, 1024, 16
        lf = workloads.Linear("f32_layer", workloads.draw(rng, T, K, 1.0, workloads.FP32),
                              workloads.draw(rng, N, K, (1.0 / K) ** 0.5, workloads.FP32),
                              workloads.draw(rng, 1, N, 0.01, workloads.FP32),
                              [workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5, workloads.FP32),
                                               workloads.draw(rng, N, r, 0.02, workloads.FP32), float(r), 0.8)])
        f32_entry("f32_layer", lf, "an all-FP32 layer large enough to fill the GPU: T=4096, 1024 -> 1024, rank 16 "
                                   "(rank_proj_kernel + f32_linear_kernel)")
    if want("wan_qkv_rank128"):
        fwd_entry("wan_qkv_rank128", workloads.wan_qkv_rank128("full"),
                  "the sglang PR's own Speed Tests shape: rank 128 on each of q/k/v (two rank passes)")
    if want("c2_ffn_up") or want("c2_ffn_down"):
        up, down, _ = workloads.config2("full")
        if want("c2_ffn_up"):
            fwd_entry("c2_ffn_up", up)
        del up
        if want("c2_ffn_down"):
            fwd_entry("c2_ffn_down", down)
        del down
        torch.cuda.empty_cache()
    c3 = ("c3_nf4_gate_up_fwd", "c3_nf4_down_fwd", "c3_nf4_gate_up_bwd", "c3_nf4_down_bwd")
    if any(want(n) for n in c3):
        gate_up, down3 = workloads.config3("full")
        for n, lin, fn in zip(c3, (gate_up, down3, gate_up, down3), (fwd_entry, fwd_entry, bwd_entry, bwd_entry)):
            if want(n):
                fn(n, lin)
        del gate_up, down3
        torch.cuda.empty_cache()
    if want("c3_swiglu_bwd"):
        # the SwiGLU backward step on the C3 shape: dH [T, F], e | g [T, 2F] -> de | dg and h
        rng = np.random.default_rng(22)
        T, F = workloads.FULL[3]["T"], workloads.FULL[3]["d_ff"]
        dH = workloads.draw(rng, T, F, 1.0).torch_cpu().to(dev)
        EG = workloads.draw(rng, T, 2 * F, 1.0).torch_cpu().to(dev)
        dEG = torch.empty_like(EG)
        Hh = torch.empty_like(dH)
        t_s = time.time()
        ms = timed(lambda: wpg.lora_swiglu_bwd(dH, EG, deg=dEG, h=Hh, want_h=True))
        marks["c3_swiglu_bwd"] = (t_s, time.time())
        nbytes = T * F * (2 + 4 + 4 + 2)
        out["c3_swiglu_bwd"] = {"mb": round(nbytes / 1e6, 1), "ms": round(ms, 5),
                                "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bound": "hbm",
                                "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                                "work": "read dH, e, g; write de, dg, h (12 B per element of F)"}
    def flushed(fn):
        # one call at a time after an L2 flush, CUDA events around the call; the median
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        times = []
        for i in range(k + 3):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 3:
                times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    if want("c3_nf4_merge"):
        # the rank-16 patch baked into the 4-bit C3 down weight in place (dequantise, add,
        # requantise); a small request scale keeps the repeated merges near the seeded weight
        down3 = workloads.config3("full")[1]
        W3, ads3 = d(down3.W), ads_of(down3)
        ws3 = torch.empty(max(1, wpg.lora_workspace_size(wpg.WP_OP_MERGE, None, W3, ads3)), dtype=torch.uint8,
                          device=dev)
        t_s = time.time()
        ms = flushed(lambda: wpg.lora_merge(W3, ads3, 1e-4, workspace=ws3))
        seeds = iter(range(1, 1 << 20))
        ms_st = flushed(lambda: wpg.lora_merge(W3, ads3, 1e-4, workspace=ws3, rounding_seed=next(seeds)))
        marks["c3_nf4_merge"] = (t_s, time.time())
        assert wpg.lora_device_status() == 0
        nbytes = 2 * (W3.packed.numel() + W3.absmax.numel() * 4)
        out["c3_nf4_merge"] = {"mb": round(nbytes / 1e6, 1), "ms": round(ms, 5),
                               "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bound": "hbm",
                               "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                               "stochastic": {"ms": round(ms_st, 5),
                                              "frac": round(nbytes / (ms_st * 1e-3) / 1e9 / hbm, 4)},
                               "work": "codes and scales read and written once (the adapter's 0.3 MB aside); "
                                       "stochastic: the same with the Philox-sampled codes",
                               "timing": "one call after an L2 flush, launch included, median"}
        del W3, ads3, ws3
        torch.cuda.empty_cache()
    for name, T_few in (("c3_nf4_gate_up_t1", 1), ("c3_nf4_gate_up_t16", 16)):
        if not want(name):
            continue
        # a few tokens through the 4-bit gate/up layer: the weight-streaming paths (the CUDA-core
        # GEMV up to 4 tokens, the tensor-core small-token kernel above); bound by reading the
        # 4-bit weight once
        g3 = workloads.config3("full")[0]
        lf = workloads.Linear(g3.name, g3.X.slice_rows(0, T_few), g3.W, g3.bias, g3.patches, g3.request_scale,
                              g3.groups)
        Xf, Wf, adsf = d(lf.X), d(lf.W), ads_of(lf)
        Yf = torch.empty(T_few, lf.W.rows, dtype=torch.bfloat16, device=dev)
        wsf = torch.empty(max(1, wpg.lora_workspace_size(wpg.WP_OP_FWD_GROUPED, Xf, Wf, adsf)), dtype=torch.uint8,
                          device=dev)
        t_s = time.time()
        ms = flushed(lambda: wpg.lora_linear_fwd_grouped(Xf, Wf, None, adsf, lf.request_scale, out=Yf, workspace=wsf))
        marks[name] = (t_s, time.time())
        assert wpg.lora_device_status() == 0
        nbytes = Wf.packed.numel() + Wf.absmax.numel() * 4
        out[name] = {"tokens": T_few, "mb": round(nbytes / 1e6, 1), "ms": round(ms, 5),
                     "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bound": "hbm",
                     "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                     "work": "the 4-bit weight (codes and scales) read once; the call's kernels and launches",
                     "timing": "one call after an L2 flush, launch included, median"}
        del Xf, Wf, adsf, Yf, wsf
        torch.cuda.empty_cache()
    if want("c4_sidecar") or want("c4_set_weight"):
        lin4, payload = workloads.config4("full")
        if want("c4_sidecar"):
            fwd_entry("c4_sidecar", lin4, "three patches (ranks 16 fp32 / 32 / 128 bf16)")
        if want("c4_set_weight"):
            P = d(payload)
            param = torch.empty_like(P)
            t_s = time.time()
            ms = flushed(lambda: wpg.lora_dense_patch(param, P, wpg.WP_PATCH_SET, 1.0))
            marks["c4_set_weight"] = (t_s, time.time())
            nbytes = 2 * P.numel() * P.element_size()
            out["c4_set_weight"] = {"mb": round(nbytes / 1e6, 1), "ms": round(ms, 5),
                                    "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bound": "hbm",
                                    "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                                    "timing": "one call after an L2 flush, launch included, median"}
    clocks.stop()
    for name, (a, b) in marks.items():
        out[name]["clocks"] = clocks.summary(a, b)
    return out


def run_case(args):
    """One workload of per_config on its own (for profiling a single kernel's launches)."""
    import torch
    if args.case not in CASES:
        sys.exit(f"bench.py: unknown case {args.case!r}; cases: {', '.join(CASES)}")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, hbm, _ = measured_peaks()
    res = per_config(dev, args, peak, hbm, only={args.case})
    print(json.dumps({"case": args.case, **res[args.case]}))


def device_sm_count(dev):
    import torch
    return torch.cuda.get_device_properties(dev).multi_processor_count


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
        "config": bench_config(ws),
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
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--case", default=None, help="time one workload of per_config alone: " + ", ".join(CASES))
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, _, _ = dist_env()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one rank per GPU: re-launch this command under torchrun
        import socket
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
        sys.exit(subprocess.call(cmd))
    if ws != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={ws}")
    if args.impl == "reference":
        run_reference(args)
    elif args.case:
        run_case(args)
    else:
        run_fused(args)


if __name__ == "__main__":
    main()
