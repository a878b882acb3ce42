"""4-bit NormalFloat (NF4) base weights, oracle side.

Test infrastructure only; see the package docstring.

The pages use NF4 base weights without printing the code table: the InvokeAI
sidecar-patch article (section 五, the quantised layer) and the Unsloth fast_lora
walkthrough (section 3, ``matmul_lora``: 4-bit -> bf16 before the matmul) both
dequantise bitsandbytes' 4-bit weights.  The table is the published QLoRA NormalFloat
construction (Dettmers et al., 2023, "4-bit NormalFloat Quantization"):

  * take quantiles of N(0, 1) at evenly spaced probabilities between 1/2 and an
    upper probability delta (the normal's 1-quantile is infinite);
  * the positive half uses 2**(k-1) + 1 = 9 points, the negative half 2**(k-1) = 8
    points, each including the zero at probability 1/2;
  * merge the halves, keep a single zero, and divide by the largest value so the
    16 levels span [-1, 1] exactly.

Readings where the definition leaves a choice (each listed in the design notes):
  * delta = ((1 - 1/(2*15)) + (1 - 1/(2*16))) / 2, the mean of the symmetric
    endpoint for 15 and for 16 levels;
  * the table is computed in float64 (``statistics.NormalDist.inv_cdf``) and rounded
    once to float32;
  * dequantisation: W_eff = bf16_rne(fl32(code[q] * absmax)), one float32 product
    rounded to bf16 (the walkthrough dequantises to bf16 before the GEMM);
  * storage: blocks of 64 consecutive row-major elements, one fp32 absmax each;
    byte k holds element 2k in the high nibble, 2k+1 in the low nibble.

Parity unpinned: bit-identity of this table with the one bitsandbytes ships (its
checkpoints are not in reach); interoperability is left for later.
"""
from __future__ import annotations

from statistics import NormalDist

import numpy as np

from .numerics import bf16_bits_to_f64, f32_to_bf16_bits

BLOCK = 64


def upper_probability() -> float:
    return 0.5 * ((1.0 - 1.0 / (2 * 15)) + (1.0 - 1.0 / (2 * 16)))


def codebook_f64() -> np.ndarray:
    """The 16 NormalFloat levels in float64, ascending."""
    nd = NormalDist()
    delta = upper_probability()
    pos = [nd.inv_cdf(delta - j * (delta - 0.5) / 8.0) for j in range(8)]   # 8 > 0
    neg = [-nd.inv_cdf(delta - j * (delta - 0.5) / 7.0) for j in range(7)]  # 7 < 0
    top = nd.inv_cdf(delta)
    levels = sorted(v / top for v in pos + neg + [0.0])
    return np.array(levels, dtype=np.float64)


def codebook_f32() -> np.ndarray:
    return codebook_f64().astype(np.float32)


def unpack_codes(packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """uint8 [rows, cols/2] -> uint8 codes [rows, cols]; element 2k is the high nibble."""
    p = np.asarray(packed, dtype=np.uint8).reshape(rows, cols // 2)
    codes = np.empty((rows, cols), dtype=np.uint8)
    codes[:, 0::2] = p >> 4
    codes[:, 1::2] = p & 0x0F
    return codes


def pack_codes(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    return ((c[:, 0::2] << 4) | c[:, 1::2]).astype(np.uint8)


def dequant_bf16_bits(packed: np.ndarray, absmax: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """The effective bf16 weight as bit patterns [rows, cols]."""
    codes = unpack_codes(packed, rows, cols)
    cb = codebook_f32()
    scale = np.asarray(absmax, dtype=np.float32).reshape(rows, cols // BLOCK)
    scale = np.repeat(scale, BLOCK, axis=1)
    prod = (cb[codes] * scale).astype(np.float32)   # one IEEE float32 product
    return f32_to_bf16_bits(prod)


def dequant_f64(packed: np.ndarray, absmax: np.ndarray, rows: int, cols: int) -> np.ndarray:
    return bf16_bits_to_f64(dequant_bf16_bits(packed, absmax, rows, cols))
