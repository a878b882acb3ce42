"""Shared helpers for the GPU parity tests: storage -> device tensors, calls through the
binding, decoding of outputs for the oracle comparison."""
import numpy as np
import torch

import weight_patches_gb300 as wpg
from oracle import lora as olora
from oracle.numerics import bf16_bits_to_f64, relative_rms

DEV = torch.device("cuda:0")


def dev(mat):
    """workloads.Mat -> device tensor (bf16/fp32) or NF4Weight."""
    if mat.kind == "nf4":
        return wpg.NF4Weight(torch.from_numpy(np.ascontiguousarray(mat.data)).to(DEV),
                             torch.from_numpy(np.ascontiguousarray(mat.absmax)).to(DEV),
                             mat.rows, mat.cols)
    return mat.torch_cpu().to(DEV)


def adapters(lin):
    return [wpg.Adapter(dev(p.A), dev(p.B), p.alpha, p.strength,
                        dev(p.bias_B).reshape(-1) if getattr(p, "bias_B", None) is not None else None)
            for p in lin.patches]


def run_fwd(lin, out_dtype=torch.bfloat16, with_base=True, request_scale=None):
    X = dev(lin.X)
    W = dev(lin.W) if (with_base and lin.W is not None) else None
    bias = dev(lin.bias).reshape(-1) if lin.bias is not None else None
    rs = lin.request_scale if request_scale is None else request_scale
    ads = adapters(lin)
    if lin.groups > 1:
        Y = wpg.lora_linear_fwd_grouped(X, W, bias, ads, rs, out_dtype=out_dtype)
    else:
        Y = wpg.lora_linear_fwd(X, W, bias, ads, rs, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return Y


def to_f64(Y: torch.Tensor) -> np.ndarray:
    if Y.dtype == torch.bfloat16:
        return bf16_bits_to_f64(Y.cpu().view(torch.int16).numpy().view(np.uint16))
    return Y.cpu().numpy().astype(np.float64)


def errors(lin, Y, rows=None):
    """(fused rel-RMS, simulated unfused-chain rel-RMS) against the FP64 definition."""
    got = to_f64(Y)
    if rows is not None:
        got = got[rows]
    want = olora.reference_output(lin, rows)
    chain = olora.reference_chain(lin, rows)
    return relative_rms(got, want), relative_rms(chain, want)


def torch_unfused_chain(lin):
    """The pre-PR chain in torch eager bf16 on the GPU (test harness only)."""
    X = dev(lin.X)
    W = dev(lin.W)
    bias = dev(lin.bias).reshape(-1) if lin.bias is not None else None
    Y = torch.nn.functional.linear(X, W, bias)
    G = lin.groups
    og = Y.shape[1] // G if G > 1 else Y.shape[1]
    for i, p in enumerate(lin.patches):
        A, B = dev(p.A), dev(p.B)
        t = X.to(A.dtype) @ A.t()
        d = t @ B.t()
        for c in (p.alpha / p.rank, p.strength, lin.request_scale):
            if c != 1.0:
                d = d * c
        sl = slice(i * og, (i + 1) * og) if G > 1 else slice(None)
        Y[:, sl] = (Y[:, sl].to(d.dtype) + d).to(Y.dtype)
    torch.cuda.synchronize()
    return Y
