"""LoRA merge into the base weight (oracle side).

Test infrastructure only; see the package docstring.

piper-offload docs, "LoRA merge" and "Quantized weight support": merging bakes the
adapters into the weight in place -- a plain floating-point weight takes an ``addmm_``
update, a bitsandbytes NF4 weight is dequantised, takes every LoRA of the target as one
staged low-rank update and is re-encoded once; the re-encoding is stochastic by default
and deterministic round-to-nearest on request (both forms are here).
The update of one adapter is s (B A) with s = alpha / r * strength * scale (the PEFT
convention the rest of the library uses).

Readings (the pages fix the flow, not the arithmetic):
  * every adapter of a call is one update, accumulated exactly and rounded once:
    W' = round(W + sum_p s_p B_p A_p);
  * bf16 weight: round to nearest even;
  * NF4 weight: W_eff = bf16(fl32(level[q]) * absmax) as in the forward; u = W_eff + update;
    per 64-element block absmax' = max |u|, and each element's code is the nearest level of
    u / absmax' -- decided, like the kernel, in float32: x = fl32(fl32(u) / absmax'), code =
    the number of midpoints fl32((level[k] + level[k+1]) / 2) below x (a value on a midpoint
    takes the lower code); an all-zero block keeps scale 0 and the code of level 0 (index 7).

Stochastic re-encoding (piper-offload docs, "LoRA merge": the final scales come from the
deterministic recipe, then only the terminal code is sampled "between the two neighboring
values on that finalized grid"; "exact endpoints and saturation retain the upstream code";
samples are keyed by logical element index).  Reading, with x = fl32(u / absmax') as above:
x equal to a level keeps that level's code; otherwise lo < x < hi are the neighbouring levels
and hi is chosen with probability (x - lo) / (hi - lo), decided in float32 as
U * w < d * 2^23 with d = fl32(x - lo), w = fl32(hi - lo) and U the element's 23-bit uniform
draw (``rng.element_uniform23``; U * w and d * 2^23 are exact, so the comparison is too).
An all-zero block keeps scale 0 and the zero level's code, as in the deterministic form.

Legacy adapter bias vectors (the lora_B.bias older adapters carry; piper-offload docs,
"LoRA merge": merge mode adds the vector to the module's dense bias with the same adapter
strength) follow the dense bias patch's arithmetic (FastVideo DenseLoRAPatch.apply_to:
cast(fp32(param) + fp32(payload) * k)) with k = s_p, all of a call's vectors summed in
float32 in call order and the sum cast once (one update, as for the weight).

Pinned by ``tests/test_oracle_merge.py``: brute force (exhaustive argmin over the 16
levels), the dequantise-requantise round trip on blocks that hold level +-1, merge and
unmerge returning the weight within one rounding, zero strength leaving it unchanged,
and the merged weight reproducing the unmerged forward (the forward is linear, Unsloth
fast_lora walkthrough, section 2).
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

from . import nf4 as onf4
from . import rng as orng
from .lora import DecodedPatch, combined_scale
from .numerics import f64_to_bf16_value


def update(patches: Sequence[DecodedPatch], scale: float) -> np.ndarray:
    """sum_p s_p B_p A_p in float64."""
    U = None
    for p in patches:
        s = combined_scale(p.alpha, p.rank, p.strength, scale)
        d = s * (p.B @ p.A)
        U = d if U is None else U + d
    return U


def merge_bf16_values(W: np.ndarray, patches: Sequence[DecodedPatch], scale: float) -> np.ndarray:
    """The merged bf16 weight (as float64 values) from the float64 values of the old one."""
    return f64_to_bf16_value(W + update(patches, scale))


def merge_bias_values(bias: np.ndarray, patches: Sequence[DecodedPatch], scale: float,
                      bf16: bool) -> np.ndarray:
    """The merged bias (float64 values) from the old one: v = fl32(bias), then for each
    patch with a legacy vector v = fl32(v + fl32(fl32(s_p) * fl32(vec))), then the bias's
    own dtype (bf16 round to nearest even, or float32 as is)."""
    v = np.asarray(bias, dtype=np.float64).astype(np.float32)
    for p in patches:
        if p.bias_B is None:
            continue
        s = np.float32(combined_scale(p.alpha, p.rank, p.strength, scale))
        if s == 0:
            continue
        term = (s * np.asarray(p.bias_B, dtype=np.float64).astype(np.float32)).astype(np.float32)
        v = (v + term).astype(np.float32)
    v = v.astype(np.float64)
    return f64_to_bf16_value(v) if bf16 else v


def midpoints_f32() -> np.ndarray:
    """The 15 decision points between consecutive levels, in float32."""
    lv = onf4.codebook_f32()
    return ((lv[:-1] + lv[1:]).astype(np.float32) * np.float32(0.5)).astype(np.float32)


def quantize_blocks(u: np.ndarray):
    """float32 [rows, cols] (cols % 64 == 0) -> (codes uint8 [rows, cols], absmax float32
    [rows * cols / 64], x float32 [rows, cols]): the requantisation rule of the module
    docstring, in float32."""
    u = np.asarray(u, dtype=np.float32)
    rows, cols = u.shape
    b = u.reshape(-1, onf4.BLOCK)
    m = np.max(np.abs(b), axis=1).astype(np.float32)
    safe = np.where(m > 0, m, np.float32(1.0)).astype(np.float32)
    x = (b / safe[:, None]).astype(np.float32)
    mid = midpoints_f32()
    codes = np.sum(x[:, :, None] > mid[None, None, :], axis=2).astype(np.uint8)
    codes[m == 0] = 7
    return codes.reshape(rows, cols), m, x.reshape(rows, cols)


def quantize_blocks_stochastic(u: np.ndarray, seed: int):
    """The stochastic re-encoding of the module docstring: float32 [rows, cols] -> (codes
    uint8 [rows, cols], absmax float32 [rows * cols / 64], x float32 [rows, cols], slack
    float64 [rows, cols]).  slack is how far the element's decision lies from flipping, in
    units of x: min(|U w - d 2^23| / 2^23, the distance from x to the nearest level); an
    element whose x moved by less than that would keep its code."""
    u = np.asarray(u, dtype=np.float32)
    rows, cols = u.shape
    b = u.reshape(-1, onf4.BLOCK)
    m = np.max(np.abs(b), axis=1).astype(np.float32)
    safe = np.where(m > 0, m, np.float32(1.0)).astype(np.float32)
    x = (b / safe[:, None]).astype(np.float32).reshape(rows, cols)
    lv = onf4.codebook_f32()
    below = np.sum(x[..., None] > lv, axis=-1)                  # levels strictly below x
    at = np.minimum(below, 15)
    exact = lv[at] == x
    hi_i = np.clip(below, 1, 15)
    lo_v, hi_v = lv[hi_i - 1], lv[hi_i]
    d = (x - lo_v).astype(np.float32)
    w = (hi_v - lo_v).astype(np.float32)
    e = np.arange(rows * cols, dtype=np.int64).reshape(rows, cols)
    U = orng.element_uniform23(e, seed).astype(np.float64)
    lhs, rhs = U * w.astype(np.float64), d.astype(np.float64) * 2.0 ** 23
    up = lhs < rhs
    codes = np.where(exact, at, np.where(up, hi_i, hi_i - 1)).astype(np.uint8)
    zero = np.repeat(m == 0, onf4.BLOCK).reshape(rows, cols)
    codes[zero] = 7
    near_level = np.min(np.abs(x[..., None].astype(np.float64) - lv.astype(np.float64)), axis=-1)
    slack = np.minimum(np.abs(lhs - rhs) / 2.0 ** 23, np.where(exact, np.inf, near_level))
    slack[zero] = np.inf
    return codes, m, x, slack


def nearest_level_brute(x: np.ndarray) -> np.ndarray:
    """argmin_k |x - level[k]| over the 16 float32 levels (ties to the lower index), by
    exhaustive comparison; the pin of the midpoint rule."""
    lv = onf4.codebook_f32().astype(np.float64)
    d = np.abs(np.asarray(x, dtype=np.float64)[..., None] - lv)
    return np.argmin(d, axis=-1).astype(np.uint8)


def merge_nf4(packed: np.ndarray, absmax: np.ndarray, rows: int, cols: int,
              patches: Sequence[DecodedPatch], scale: float, rounding_seed=None):
    """(codes uint8 [rows, cols], absmax' float32, x float32): the requantised merge, with
    u = fl32(W_eff + update) taken to float32 once before the float32 decisions.  With a
    rounding seed, the stochastic re-encoding, which also returns each element's slack."""
    W = onf4.dequant_f64(packed, absmax, rows, cols)
    u = (W + update(patches, scale)).astype(np.float32)
    if rounding_seed is None:
        return quantize_blocks(u)
    return quantize_blocks_stochastic(u, rounding_seed)
