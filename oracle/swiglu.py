"""SwiGLU around the LoRA MLP, in FP64 (oracle side).

Test infrastructure only; see the package docstring.

Unsloth fast_lora walkthrough, section 4 (``LoRA_MLP``): the gate and up projections are
two LoRA linears, e = X G'^T and g = X U'^T (``matmul_lora``), the activation is SwiGLU,
h = f(e) g with the SiLU gate f(e) = e sigmoid(e), and the down projection takes h,
y = h D'^T.  The forward keeps X, e and g for the backward.  The backward receives the
gradient DW at h (the down projection's dX) and produces, in one kernel, h again (for the
down adapter's gradients), the gradient at g and the gradient at e; the gate/up
linears' backward then takes those two as the gradient of their stacked output.

Readings (the pages name the kernels but print no formula):
  * SwiGLU is the standard gated unit silu(e) * g, silu(e) = e / (1 + exp(-e)).
  * The gradient at g is DW * f(e); the gradient at e is DW * g * f'(e) with
    f'(e) = sigmoid(e) (1 + e (1 - sigmoid(e))), the derivative of e sigmoid(e).
  * ``lora_mlp_fwd`` / ``lora_mlp_bwd`` compose the linear oracle (``lora``) with these
    steps exactly, in FP64, with no intermediate rounding.

Pinned by ``tests/test_oracle_swiglu.py``: closed-form values of the sigmoid
(sigmoid(ln 3) = 3/4), the identities silu(x) - silu(-x) = x and
sigmoid(x) + sigmoid(-x) = 1 out to |x| = 800, and central finite differences of
sum(DW * h) and of the whole MLP's sum(dY * y) for every gradient.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .lora import DecodedPatch, combined_scale, grad_AB, linear_fwd, linear_fwd_grouped


def sigmoid(x: np.ndarray) -> np.ndarray:
    """1 / (1 + exp(-x)), evaluated on the side where the exponential cannot overflow."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    ex = np.exp(x[~pos])
    out[~pos] = ex / (1.0 + ex)
    return out


def silu(e: np.ndarray) -> np.ndarray:
    """The SiLU gate f(e) = e sigmoid(e)."""
    e = np.asarray(e, dtype=np.float64)
    return e * sigmoid(e)


def swiglu(e: np.ndarray, g: np.ndarray) -> np.ndarray:
    """h = f(e) g."""
    return silu(e) * np.asarray(g, dtype=np.float64)


def swiglu_bwd(dh: np.ndarray, e: np.ndarray, g: np.ndarray):
    """(h, dg, de) from the gradient dh at h: dg = dh f(e), de = dh g f'(e)."""
    dh = np.asarray(dh, dtype=np.float64)
    e = np.asarray(e, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    s = sigmoid(e)
    f = e * s
    fprime = s * (1.0 + e * (1.0 - s))
    return f * g, dh * f, dh * g * fprime


def lora_mlp_fwd(X: np.ndarray, W_gate_up: np.ndarray, bias_gate_up: Optional[np.ndarray],
                 gate_up_patches: Sequence[DecodedPatch], W_down: np.ndarray,
                 bias_down: Optional[np.ndarray], down_patches: Sequence[DecodedPatch],
                 request_scale: float):
    """(e, g, h, y) of the SwiGLU LoRA MLP: [e | g] is the grouped gate/up linear (one patch
    per group), h = swiglu(e, g), y the down linear of h."""
    eg = linear_fwd_grouped(X, W_gate_up, bias_gate_up, gate_up_patches, request_scale)
    F = W_gate_up.shape[0] // 2
    e, g = eg[:, :F], eg[:, F:]
    h = swiglu(e, g)
    y = linear_fwd(h, W_down, bias_down, down_patches, request_scale)
    return e, g, h, y


def lora_mlp_bwd(X: np.ndarray, W_gate_up: np.ndarray, bias_gate_up: Optional[np.ndarray],
                 gate_up_patches: Sequence[DecodedPatch], W_down: np.ndarray,
                 bias_down: Optional[np.ndarray], down_patches: Sequence[DecodedPatch],
                 request_scale: float, dY: np.ndarray) -> dict:
    """Closed-form gradients of sum(dY * y) for the SwiGLU LoRA MLP, in the order the
    walkthrough's LoRA_MLP.backward takes them: DW = dY through the down projection
    (with its LoRA), h / dg / de by the SwiGLU step, then the down adapter's dA/dB from
    h, and dX plus the gate/up adapters' dA/dB from [de | dg].  Returns a dict with keys
    dX, dH, dE, dG, h, and lists of (dA, dB) pairs for 'gate_up' (gate, up) and 'down'."""
    e, g, h, _ = lora_mlp_fwd(X, W_gate_up, bias_gate_up, gate_up_patches, W_down, bias_down,
                              down_patches, request_scale)
    # gradient at h: through the down projection W_d + sum_p s_p B_p A_p
    dH = dY @ W_down
    for p in down_patches:
        s = combined_scale(p.alpha, p.rank, p.strength, request_scale)
        dH = dH + s * ((dY @ p.B) @ p.A)
    h2, dG, dE = swiglu_bwd(dH, e, g)
    down_AB = []
    for p in down_patches:
        dA, dB = grad_AB(h2, dY, [p], request_scale)
        down_AB.append((dA[0], dB[0]))
    F = W_gate_up.shape[0] // 2
    dEG = np.concatenate([dE, dG], axis=1)
    dX = np.zeros_like(X)
    gu_AB = []
    for k, p in enumerate(gate_up_patches):
        sl = slice(k * F, (k + 1) * F)
        dYk = dEG[:, sl]
        s = combined_scale(p.alpha, p.rank, p.strength, request_scale)
        dX = dX + dYk @ W_gate_up[sl] + s * ((dYk @ p.B) @ p.A)
        dA, dB = grad_AB(X, dYk, [p], request_scale)
        gu_AB.append((dA[0], dB[0]))
    return dict(dX=dX, dH=dH, dE=dE, dG=dG, h=h2, gate_up=gu_AB, down=down_AB)
