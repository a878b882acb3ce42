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


# ----------------------------------------------------------------- element-wise bounds
# Every output element of the single-rounding design obeys
#
#   |y - y*| <= ulp_out(|y*| + e) + e,
#   e = 2^-8 sum_p |s_p| (|X| |A_p|^T) |B_p|^T            (bf16 adapters: s X A^T rounded once)
#     + 4 (K + R + 16) 2^-24 S,                             (fp32 sums of K + R terms)
#   S = |X| |W|^T + |bias| + sum_p |s_p| ((|X| |A_p|^T) |B_p|^T + |bias_B,p|),
#
# with y* the FP64 definition, K the inner size, R the adapters' total rank.  The first term
# of e is the one bf16 rounding of s X A^T (unit roundoff 2^-8) carried through B; the second
# is the fp32 accumulation: a tensor-core K step adds 16 exact products to the accumulator
# aligned to the largest and truncated, at most 17 units of 2^-23 of the running magnitude,
# which is at most S, per 16 terms (about 2.1 K 2^-24 S in all; a sequential fp32 sum of n
# terms is within n 2^-24 S), doubled for margin.  FP32 adapters on the tensor cores travel as
# bf16 pieces whose dropped terms are below 2^-24 of their product, inside the same term.
# ulp_out is one unit in the last place of the output type at that magnitude (the final
# round-to-nearest costs half of one; the other half covers the accumulator sitting in a
# higher binade than y*).  An element that is wrong by anything near its own size fails.

def ulp_bf16(v: np.ndarray) -> np.ndarray:
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return np.exp2(np.maximum(e - 7, -133))


def ulp_f32(v: np.ndarray) -> np.ndarray:
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return np.exp2(np.maximum(e - 23, -149))


def linear_error_bound(X, W, bias, patches, request_scale, groups=1, out_f32=False, y_ref=None,
                       cols=None, out_features=None):
    """Element-wise bound of the fused forward (see above) on decoded FP64 inputs.  cols
    optionally restricts the output columns (W's rows); y_ref is the FP64 result on them."""
    aX = np.abs(X)
    K = X.shape[1]
    n_out = W.shape[0] if W is not None else (out_features if out_features is not None else
                                              sum(p.B.shape[0] for p in patches) if groups > 1 else
                                              patches[0].B.shape[0])
    og = n_out // groups
    colv = np.arange(n_out) if cols is None else np.asarray(cols)
    S = np.zeros((X.shape[0], len(colv)))
    if W is not None:
        S += aX @ np.abs(W[colv]).T
    if bias is not None:
        S += np.abs(np.asarray(bias, dtype=np.float64).reshape(-1)[colv])[None, :]
    lora_round = np.zeros_like(S)
    R = 0
    for i, p in enumerate(patches):
        R += p.rank
        s = abs(olora.combined_scale(p.alpha, p.rank, p.strength, request_scale))
        g = i if groups > 1 else 0
        sel = (colv >= g * og) & (colv < (g + 1) * og) if groups > 1 else np.ones(len(colv), bool)
        if not sel.any():
            continue
        local = colv[sel] - g * og if groups > 1 else colv[sel]
        mag = s * ((aX @ np.abs(p.A).T) @ np.abs(p.B[local]).T)
        if p.bias_B is not None:
            mag = mag + s * np.abs(np.asarray(p.bias_B, dtype=np.float64).reshape(-1)[local])[None, :]
        S[:, sel] += mag
        if not p.fp32_adapter:
            lora_round[:, sel] += 2.0 ** -8 * mag
    e = lora_round + 4.0 * (K + R + 16) * 2.0 ** -24 * S
    mag_y = np.abs(y_ref) + e
    return (ulp_f32(mag_y) if out_f32 else ulp_bf16(mag_y)) + e


def fwd_bound(lin, rows=None, out_f32=False, y_ref=None, with_base=True, request_scale=None):
    X, W, bias, patches = olora.decode_linear(lin, rows)
    rs = lin.request_scale if request_scale is None else request_scale
    if y_ref is None:
        y_ref = olora.reference_output(lin, rows)
    return linear_error_bound(X, W if with_base else None, bias, patches, rs, lin.groups, out_f32, y_ref,
                              out_features=lin.out_features)


def assert_elementwise(got, want, bound, what=""):
    got = np.asarray(got, dtype=np.float64)
    bad = ~(np.abs(got - want) <= bound)          # NaN in got fails too
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(int(v) for v in i), float(got[tuple(i)]), float(want[tuple(i)]), float(bound[tuple(i)]))
                  for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside the element-wise "
                             f"bound (index, got, want, bound): {detail}")


def errors(lin, Y, rows=None, elementwise=True):
    """(fused rel-RMS, simulated unfused-chain rel-RMS) against the FP64 definition; also
    asserts the element-wise bound of every output element."""
    got = to_f64(Y)
    if rows is not None:
        got = got[rows]
    want = olora.reference_output(lin, rows)
    chain = olora.reference_chain(lin, rows)
    if elementwise:
        bound = fwd_bound(lin, rows, out_f32=Y.dtype == torch.float32, y_ref=want)
        assert_elementwise(got, want, bound, lin.name)
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


def swiglu_bound(e_ref, g_ref, be, bg):
    """Element-wise bound of h = bf16(silu(e) g) where e and g are the bf16 outputs of the
    gate/up linear (within be, bg of their FP64 values e*, g*): silu is 1.1-Lipschitz
    (|silu'(x)| = |sigma(x) (1 + x (1 - sigma(x)))| < 1.1), the fp32 evaluation of silu and
    of the product adds at most 2^-18 relative, and the final rounding one ulp."""
    from oracle import swiglu as osw
    sil = np.abs(osw.silu(e_ref))
    ag = np.abs(g_ref) + bg
    d = 1.1 * be * ag + (sil + 1.1 * be) * bg + 2.0 ** -18 * (sil + 1.1 * be) * ag
    h_ref = osw.swiglu(e_ref, g_ref)
    return ulp_bf16(np.abs(h_ref) + d) + d


def bwd_bounds(X, W, dY, patches, request_scale, dX_ref, dA_ref, dB_ref, dX_f32=False):
    """Element-wise bounds of dX, dA_g, dB_g of the closed-form backward on decoded FP64
    inputs (X [T, K], W [N, K], dY [T, N]).  dX = dY W + sum_g s_g (dY_g B_g) A_g is the
    forward's structure with dY as the tokens and W^T as the weight (inner size N); dA_g and
    dB_g take s G_g (G_g = dY_g B_g, an fp32 sum over the group's columns) and H_g = X A_g^T
    (an fp32 sum over K) as two bf16 pieces each (2^-16 relative) and sum over the T tokens
    in fp32."""
    G = len(patches)
    N = W.shape[0]
    og = N // G
    T, K = X.shape
    aX, adY = np.abs(X), np.abs(dY)
    pats_t = []
    for g, p in enumerate(patches):
        Bhat = np.zeros((p.rank, N))
        Bhat[:, g * og:(g + 1) * og] = p.B.T
        pats_t.append(olora.DecodedPatch(Bhat, p.A.T, p.alpha, p.strength))
    b_dX = linear_error_bound(dY, W.T, None, pats_t, request_scale, 1, dX_f32, dX_ref)
    b_dA, b_dB = [], []
    for g, p in enumerate(patches):
        s = abs(olora.combined_scale(p.alpha, p.rank, p.strength, request_scale))
        dyg = adY[:, g * og:(g + 1) * og]
        magA = s * ((dyg @ np.abs(p.B)).T @ aX)
        magB = s * (dyg.T @ (aX @ np.abs(p.A).T))
        eA = (4.0 * (og + T + 32) * 2.0 ** -24 + 2.0 ** -16) * magA
        eB = (4.0 * (K + T + 32) * 2.0 ** -24 + 2.0 ** -16) * magB
        b_dA.append(ulp_f32(np.abs(dA_ref[g]) + eA) + eA)
        b_dB.append(ulp_f32(np.abs(dB_ref[g]) + eB) + eB)
    return b_dX, b_dA, b_dB
