"""Exact decoding of stored values and round-to-nearest-even encodings (oracle side).

Test infrastructure only; see the package docstring.

bf16 is the upper half of an IEEE binary32: 1 sign, 8 exponent, 7 fraction bits.
Rounding to bf16 is round-to-nearest, ties to even, the rule torch's ``.to(bfloat16)``
applies (the sglang PR "Add the dynamic LoRA delta inside the second GEMM" keeps its
tensors in BF16 and its accuracy gate is stated against FP64 math, Accuracy Tests).
"""
from __future__ import annotations

import numpy as np

BF16_MAX = float(np.uint32(0x7F7F0000).view(np.float32))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the exact float32 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even; NaN stays NaN (quiet)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, ((u >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040)), r)
    return r


def f64_to_bf16_value(x: np.ndarray) -> np.ndarray:
    """Round float64 values straight to the nearest bf16 value (ties to even), with
    no intermediate float32 step.  Returns float64 holding bf16 values.

    A bf16 number has 8 significant bits; with x = m * 2**e (0.5 <= |m| < 1) its
    quantum is 2**(e - 8), floored at the subnormal quantum 2**-133.  Values past
    the largest finite bf16 after rounding become infinities."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    m, e = np.frexp(x[fin])
    q = np.maximum(e - 8, -133).astype(np.float64)
    scaled = np.ldexp(x[fin], (-q).astype(np.int64))
    r = np.ldexp(np.rint(scaled), q.astype(np.int64))
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)
    out[fin] = r
    return out


def to_f64(mat) -> np.ndarray:
    """Decode a ``workloads.Mat`` of bf16 / fp32 storage to exact float64."""
    if mat.kind == "bf16":
        return bf16_bits_to_f64(mat.data)
    if mat.kind == "fp32":
        return np.asarray(mat.data, dtype=np.float32).astype(np.float64)
    if mat.kind == "nf4":
        from .nf4 import dequant_f64
        return dequant_f64(mat.data, mat.absmax, mat.rows, mat.cols)
    raise ValueError(mat.kind)


def relative_rms(y: np.ndarray, y_ref: np.ndarray) -> float:
    """sqrt(sum (y - y*)^2 / sum y*^2) over the whole tensor: the RMS error measure of
    the sglang PR's accuracy gate (Accuracy Tests), read as relative to the FP64
    result's own RMS."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    den = float(np.sum(y_ref * y_ref))
    num = float(np.sum((y - y_ref) ** 2))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return (num / den) ** 0.5
