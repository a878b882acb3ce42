"""The dynamic, unmerged LoRA linear in FP64 (oracle side).

Test infrastructure only; see the package docstring.

Notation (PyTorch / PEFT convention): X [T, in], W [out, in], A_p [r_p, in],
B_p [out, r_p], bias [out], Y [T, out], all row-major, and

    Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T,
    s_p = alpha_p / r_p * strength_p * request_scale.

Sources:
  * sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM",
    Motivation: the update is scaled by alpha/rank, by the adapter strength and by the
    request's LoRA scale, and added to the base output; Modifications: the combined
    scale multiplies the rank-wide intermediate x @ A^T, the second GEMM accumulates
    onto the base output, stacked q/k/v (gate/up) adapters take one update per column
    group, the bias belongs to the base GEMM's epilogue, an FP32 adapter on BF16
    activations keeps FP32 GEMMs and adds once.
  * InvokeAI sidecar-patch article, sections 三 and 四: several patches on one layer
    each contribute their own weighted term and the contributions are summed.
  * Unsloth fast_lora walkthrough, section 2: the forward is linear,
    out = X (W + s A B)^T in its transposed naming, and the backward has closed forms
    for dX, dA, dB (section 4, ``LoRA_MLP`` / ``LoRA_QKV``).
  * piper-offload docs, "LoRA merge": older PEFT/Wan adapters may carry a vector beside A
    and B (their lora_B.bias); routed mode applies it as part of the output residual, merge
    mode adds it to the module's bias with the same adapter strength.  Reading: the vector
    is scaled by the adapter's own s, so a patch contributes s ((X A^T) B^T + bias_B), as
    the second factor's bias of a PEFT adapter does.

Everything is exact FP64 on exactly decoded inputs; ``numpy.matmul`` is the only
library step.  ``unfused_bf16_chain`` is not the definition: it simulates the
pre-PR chain (each pass rounded to bf16) and is the baseline of the "error no worse
than the reference chain" gate.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from .numerics import f64_to_bf16_value


@dataclass
class DecodedPatch:
    A: np.ndarray          # [r, in] float64
    B: np.ndarray          # [out, r] float64
    alpha: float
    strength: float
    fp32_adapter: bool = False
    bias_B: Optional[np.ndarray] = None   # [out] float64: the legacy vector, or None

    @property
    def rank(self) -> int:
        return self.A.shape[0]


def combined_scale(alpha: float, rank: int, strength: float, request_scale: float) -> float:
    """s = alpha / rank * strength * request_scale (sglang PR, Motivation and
    Modifications), in float64."""
    return alpha / rank * strength * request_scale


def lora_delta(X: np.ndarray, p: DecodedPatch, request_scale: float) -> np.ndarray:
    """s ((X A^T) B^T + bias_B) for one patch (bias_B, the legacy vector, if it has one)."""
    s = combined_scale(p.alpha, p.rank, p.strength, request_scale)
    H = X @ p.A.T
    D = H @ p.B.T
    if p.bias_B is not None:
        D = D + np.asarray(p.bias_B, dtype=np.float64).reshape(1, -1)
    return s * D


def linear_fwd(X: np.ndarray, W: Optional[np.ndarray], bias: Optional[np.ndarray],
               patches: Sequence[DecodedPatch], request_scale: float,
               out_features: Optional[int] = None) -> np.ndarray:
    """Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T.  W may be None (delta only)."""
    if W is not None:
        Y = X @ W.T
    else:
        n = out_features if out_features is not None else patches[0].B.shape[0]
        Y = np.zeros((X.shape[0], n), dtype=np.float64)
    if bias is not None:
        Y = Y + np.asarray(bias, dtype=np.float64).reshape(1, -1)
    for p in patches:
        Y = Y + lora_delta(X, p, request_scale)
    return Y


def linear_fwd_grouped(X: np.ndarray, W_stacked: np.ndarray, bias: Optional[np.ndarray],
                       group_patches: Sequence[DecodedPatch], request_scale: float) -> np.ndarray:
    """Stacked column groups: W_stacked is the row-stack of G equal groups; group g's
    output columns get X W_g^T + s_g (X A_g^T) B_g^T (sglang PR, Modifications:
    one update per group on column views of the output)."""
    G = len(group_patches)
    out = W_stacked.shape[0]
    if out % G:
        raise ValueError("stacked weight rows must split evenly into groups")
    og = out // G
    Y = X @ W_stacked.T
    if bias is not None:
        Y = Y + np.asarray(bias, dtype=np.float64).reshape(1, -1)
    for g, p in enumerate(group_patches):
        Y[:, g * og:(g + 1) * og] += lora_delta(X, p, request_scale)
    return Y


@dataclass
class Grads:
    dX: np.ndarray
    dA: list
    dB: list


def linear_bwd(X: np.ndarray, W: np.ndarray, dY: np.ndarray,
               group_patches: Sequence[DecodedPatch], request_scale: float) -> Grads:
    """Closed-form backward of Y = X W^T + s (X A^T) B^T for one or more column groups
    (Unsloth fast_lora walkthrough, sections 2 and 4), with G_g = dY_g B_g:

        dX   = sum_g dY_g W_g + s_g G_g A_g
        dA_g = s_g G_g^T X
        dB_g = s_g dY_g^T (X A_g^T)
    """
    dX = grad_X(X, W, dY, group_patches, request_scale)
    dA, dB = grad_AB(X, dY, group_patches, request_scale)
    return Grads(dX, dA, dB)


def grad_X(X: np.ndarray, W: np.ndarray, dY: np.ndarray, group_patches: Sequence[DecodedPatch],
           request_scale: float) -> np.ndarray:
    """dX = sum_g dY_g W_g + s_g (dY_g B_g) A_g (rows of dX depend only on the same rows of
    dY, so it may be evaluated on any subset of token rows)."""
    G = len(group_patches)
    og = W.shape[0] // G
    dX = np.zeros((dY.shape[0], W.shape[1]))
    for g, p in enumerate(group_patches):
        s = combined_scale(p.alpha, p.rank, p.strength, request_scale)
        dYg = dY[:, g * og:(g + 1) * og]
        dX = dX + dYg @ W[g * og:(g + 1) * og] + s * ((dYg @ p.B) @ p.A)
    return dX


def grad_AB(X: np.ndarray, dY: np.ndarray, group_patches: Sequence[DecodedPatch],
            request_scale: float):
    """dA_g = s_g (dY_g B_g)^T X and dB_g = s_g dY_g^T (X A_g^T).  Both are sums over token
    rows, so the results of disjoint row sets add up to the result of their union."""
    G = len(group_patches)
    og = dY.shape[1] // G
    dA, dB = [], []
    for g, p in enumerate(group_patches):
        s = combined_scale(p.alpha, p.rank, p.strength, request_scale)
        dYg = dY[:, g * og:(g + 1) * og]
        dA.append(s * ((dYg @ p.B).T @ X))
        dB.append(s * (dYg.T @ (X @ p.A.T)))
    return dA, dB


def unfused_bf16_chain(X: np.ndarray, W: Optional[np.ndarray], bias: Optional[np.ndarray],
                       patches: Sequence[DecodedPatch], request_scale: float,
                       column_slices: Optional[Sequence[slice]] = None,
                       out_features: Optional[int] = None,
                       bf16_tensors: bool = True) -> np.ndarray:
    """Simulation of the pre-PR dynamic chain (sglang PR, Motivation): every tensor the
    chain materialises is rounded to bf16.

        base = bf16(X W^T + bias)                 (bias in the base GEMM, one GPU)
        t    = bf16(X A^T);  d = bf16(t B^T)      (d = bf16(t B^T + bias_B) for a legacy
                                                   vector: the second factor's own bias)
        d    = bf16(d * alpha/r); d = bf16(d * strength); d = bf16(d * request_scale)
        Y    = bf16(Y + d)                        (patch after patch, in order)

    A multiplication by exactly 1.0 is exact, so skipping it changes nothing (the PR's
    ``exact`` tier).  An FP32 adapter keeps its two GEMMs and its scaling in FP32 and is
    added once.  ``column_slices[p]`` restricts patch p to a column range (stacked
    groups).  With ``bf16_tensors=False`` (an all-FP32 layer) nothing is rounded and the
    chain equals the definition."""
    rnd = f64_to_bf16_value if bf16_tensors else (lambda v: v)
    if W is not None:
        acc = X @ W.T
    else:
        n = out_features if out_features is not None else patches[0].B.shape[0]
        acc = np.zeros((X.shape[0], n))
    if bias is not None:
        acc = acc + np.asarray(bias, dtype=np.float64).reshape(1, -1)
    Y = rnd(acc)
    for i, p in enumerate(patches):
        sl = column_slices[i] if column_slices is not None else slice(None)
        scales = [np.float64(np.float32(p.alpha / p.rank)), np.float64(np.float32(p.strength)),
                  np.float64(np.float32(request_scale))]
        vb = 0.0 if p.bias_B is None else np.asarray(p.bias_B, dtype=np.float64).reshape(1, -1)
        if p.fp32_adapter:
            d = (X @ p.A.T) @ p.B.T + vb
            for c in scales:
                d = d * c
        else:
            t = rnd(X @ p.A.T)
            d = rnd(t @ p.B.T + vb)
            for c in scales:
                if c != 1.0:
                    d = rnd(d * c)
        Y[:, sl] = rnd(Y[:, sl] + d)
    return Y


def decode_patch(p) -> DecodedPatch:
    """A ``workloads.Patch`` decoded to exact float64."""
    from .numerics import to_f64
    vb = getattr(p, "bias_B", None)
    return DecodedPatch(to_f64(p.A), to_f64(p.B), float(p.alpha), float(p.strength),
                        fp32_adapter=(p.A.kind == "fp32" and p.B.kind == "fp32"),
                        bias_B=None if vb is None else to_f64(vb).reshape(-1))


def decode_linear(lin, rows=None):
    """(X, W, bias, patches) of a ``workloads.Linear`` as float64; ``rows`` optionally
    selects token rows of X (spot checks at full size)."""
    from .numerics import to_f64
    X = to_f64(lin.X) if rows is None else to_f64_rows(lin.X, rows)
    W = to_f64(lin.W) if lin.W is not None else None
    bias = to_f64(lin.bias).reshape(-1) if lin.bias is not None else None
    return X, W, bias, [decode_patch(p) for p in lin.patches]


def to_f64_rows(mat, rows) -> np.ndarray:
    from .numerics import bf16_bits_to_f64
    if mat.kind == "bf16":
        return bf16_bits_to_f64(mat.data[rows])
    if mat.kind == "fp32":
        return np.asarray(mat.data[rows], dtype=np.float32).astype(np.float64)
    raise ValueError(mat.kind)


def reference_output(lin, rows=None) -> np.ndarray:
    """The FP64 definition's Y for a ``workloads.Linear`` (grouped or not)."""
    X, W, bias, patches = decode_linear(lin, rows)
    if lin.groups > 1:
        return linear_fwd_grouped(X, W, bias, patches, lin.request_scale)
    return linear_fwd(X, W, bias, patches, lin.request_scale, out_features=lin.out_features)


def reference_chain(lin, rows=None) -> np.ndarray:
    """The simulated unfused bf16 chain's Y for a ``workloads.Linear``."""
    X, W, bias, patches = decode_linear(lin, rows)
    slices = None
    if lin.groups > 1:
        og = W.shape[0] // lin.groups
        slices = [slice(g * og, (g + 1) * og) for g in range(lin.groups)]
    return unfused_bf16_chain(X, W, bias, patches, lin.request_scale, slices,
                              out_features=lin.out_features, bf16_tensors=(lin.X.kind == "bf16"))
