"""Seeded synthetic inputs for the LoRA-linear workloads.

This module only draws random numbers and stores them in the storage formats the
library reads (bf16 bit patterns, fp32, packed 4-bit codes with fp32 block
scales).  It holds none of the method's arithmetic: no products, no scales, no
dequantisation.  Both the CPU oracle (through the tests) and the CUDA path (through
the tests and the benchmark) take their inputs from here, so the two sides see the
same bits.

Recipe (every tensor, every workload):
  * a ``numpy.random.default_rng(seed)`` stream, seed = the workload's index, drawn in a
    fixed order;
  * X ~ N(0, 1), W ~ N(0, 1/in), A ~ N(0, 1/in), B ~ N(0, 0.02), bias ~ N(0, 0.01),
    dY ~ N(0, 1); draws in float32 (``Generator.standard_normal(dtype=float32)``),
    scaled, then rounded to nearest-even into bf16 by torch's cast;
  * 4-bit weights: every byte uniform in 0..255 (two independent uniform codes),
    per-64-block absmax = |N(0, 1)| in fp32;
  * dense-patch payloads: RMSNorm vector 1 + N(0, 0.02), ``.diff`` ~ N(0, 1e-3),
    ``.diff_b`` ~ N(0, 1e-5), ``.set_weight`` ~ N(0, 1/in).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

BF16, FP32, NF4 = "bf16", "fp32", "nf4"
NF4_BLOCK = 64


@dataclass
class Mat:
    """A row-major matrix in storage form.

    bf16: ``data`` is uint16 bit patterns [rows, cols].
    fp32: ``data`` is float32 [rows, cols].
    nf4:  ``data`` is uint8 [rows, cols // 2]; byte k of a row holds element 2k in its
          high nibble and element 2k + 1 in its low nibble; ``absmax`` is float32
          [rows * cols // 64], one scale per 64 consecutive elements of the row-major
          matrix.
    """

    kind: str
    data: np.ndarray
    rows: int
    cols: int
    absmax: Optional[np.ndarray] = None

    @property
    def shape(self):
        return (self.rows, self.cols)

    def slice_rows(self, r0: int, r1: int) -> "Mat":
        if self.kind == NF4:
            per_row = self.cols // NF4_BLOCK
            return Mat(NF4, self.data[r0:r1], r1 - r0, self.cols,
                       self.absmax[r0 * per_row:r1 * per_row])
        return Mat(self.kind, self.data[r0:r1], r1 - r0, self.cols)

    def torch_cpu(self) -> torch.Tensor:
        """The storage bits as a CPU torch tensor (bf16 / fp32 / uint8)."""
        if self.kind == BF16:
            return torch.from_numpy(np.ascontiguousarray(self.data).view(np.int16)).view(torch.bfloat16)
        if self.kind == FP32:
            return torch.from_numpy(np.ascontiguousarray(self.data))
        return torch.from_numpy(np.ascontiguousarray(self.data))


def _normal(rng: np.random.Generator, shape, std: float, mean: float = 0.0) -> np.ndarray:
    z = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    if mean != 0.0:
        z += np.float32(mean)
    return z


def _to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def draw(rng: np.random.Generator, rows: int, cols: int, std: float, kind: str = BF16,
         mean: float = 0.0) -> Mat:
    z = _normal(rng, (rows, cols), std, mean)
    if kind == BF16:
        return Mat(BF16, _to_bf16_bits(z), rows, cols)
    if kind == FP32:
        return Mat(FP32, z, rows, cols)
    raise ValueError(kind)


def draw_nf4(rng: np.random.Generator, rows: int, cols: int) -> Mat:
    if cols % NF4_BLOCK:
        raise ValueError("4-bit weights need cols % 64 == 0")
    packed = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    absmax = np.abs(rng.standard_normal(size=rows * cols // NF4_BLOCK, dtype=np.float32))
    return Mat(NF4, packed, rows, cols, absmax)


@dataclass
class Patch:
    """One low-rank patch: A [r, in], B [out, r], alpha, strength (the patch weight), and
    optionally the legacy vector older adapters carry beside A and B (bias_B, [1, out])."""

    A: Mat
    B: Mat
    alpha: float
    strength: float
    bias_B: Optional[Mat] = None

    @property
    def rank(self) -> int:
        return self.A.rows


@dataclass
class Linear:
    """One LoRA linear problem: Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T.

    ``groups`` > 1 means W is the row-stack of ``groups`` equal column groups and
    ``patches[g]`` belongs to group g (stacked q/k/v or gate/up).
    """

    name: str
    X: Mat
    W: Optional[Mat]
    bias: Optional[Mat]           # [1, out]
    patches: list
    request_scale: float = 1.0
    groups: int = 1
    dY: Optional[Mat] = None      # for the backward
    extra: dict = field(default_factory=dict)

    @property
    def T(self):
        return self.X.rows

    @property
    def in_features(self):
        return self.X.cols

    @property
    def out_features(self):
        if self.W is not None:
            return self.W.rows
        return sum(p.B.rows for p in self.patches) if self.groups > 1 else self.patches[0].B.rows


# --------------------------------------------------------------------------------------
# The five workloads.  ``scale="full"`` gives the sizes the benchmark times; ``"small"``
# keeps the structure (ranks, groups, dtypes, bias, 4-bit base) at sizes the FP64 oracle
# finishes in seconds while still spanning several 128x256 tiles and ragged tails.
# --------------------------------------------------------------------------------------

FULL = {
    0: dict(T=64, d_in=128, d_out=256, rank=8),
    1: dict(T=32760, d_in=1536, d_out=1536, groups=3, rank=32),
    2: dict(T=32760, d_model=1536, d_ff=8960, rank=64),
    3: dict(T=8192, d_model=4096, d_ff=14336, rank=16),
    4: dict(T=16384, d=5120, ranks=(16, 32, 128)),
}

SMALL = {
    0: dict(T=64, d_in=128, d_out=256, rank=8),
    1: dict(T=300, d_in=320, d_out=320, groups=3, rank=32),
    2: dict(T=300, d_model=192, d_ff=520, rank=64),
    3: dict(T=200, d_model=256, d_ff=320, rank=16),
    4: dict(T=260, d=384, ranks=(16, 32, 128)),
}


def config0(scale: str = "full") -> Linear:
    """Tiny all-fp32 LoRA linear (T=64, 128 -> 256, rank 8, alpha 16, strength 0.8)."""
    p = (FULL if scale == "full" else SMALL)[0]
    rng = np.random.default_rng(0)
    T, di, do, r = p["T"], p["d_in"], p["d_out"], p["rank"]
    X = draw(rng, T, di, 1.0, FP32)
    W = draw(rng, do, di, (1.0 / di) ** 0.5, FP32)
    A = draw(rng, r, di, (1.0 / di) ** 0.5, FP32)
    B = draw(rng, do, r, 0.02, FP32)
    bias = draw(rng, 1, do, 0.01, FP32)
    return Linear("c0_tiny_fp32", X, W, bias, [Patch(A, B, 16.0, 0.8)], request_scale=1.0)


def config1(scale: str = "full") -> Linear:
    """Wan2.1-1.3B stacked q/k/v: 3 column groups of 1536, rank 32 each, bf16, no bias."""
    p = (FULL if scale == "full" else SMALL)[1]
    rng = np.random.default_rng(1)
    T, di, do, G, r = p["T"], p["d_in"], p["d_out"], p["groups"], p["rank"]
    X = draw(rng, T, di, 1.0)
    W = draw(rng, G * do, di, (1.0 / di) ** 0.5)
    patches = []
    for _ in range(G):
        A = draw(rng, r, di, (1.0 / di) ** 0.5)
        B = draw(rng, do, r, 0.02)
        patches.append(Patch(A, B, 32.0, 1.0))
    return Linear("c1_wan_qkv", X, W, None, patches, request_scale=1.0, groups=G)


def config2(scale: str = "full") -> tuple:
    """FFN pair with bias (up d_model -> d_ff, down d_ff -> d_model), rank 64, alpha 64,
    strength 0.7, request scale 0.5; plus the dense patches (.diff_b on both biases,
    .diff on an RMSNorm vector of d_model).  Returns (up, down, dense) where dense is a
    dict name -> (param Mat, payload Mat, kind)."""
    p = (FULL if scale == "full" else SMALL)[2]
    rng = np.random.default_rng(2)
    T, dm, dff, r = p["T"], p["d_model"], p["d_ff"], p["rank"]
    X1 = draw(rng, T, dm, 1.0)
    W1 = draw(rng, dff, dm, (1.0 / dm) ** 0.5)
    b1 = draw(rng, 1, dff, 0.01)
    A1 = draw(rng, r, dm, (1.0 / dm) ** 0.5)
    B1 = draw(rng, dff, r, 0.02)
    X2 = draw(rng, T, dff, 1.0)
    W2 = draw(rng, dm, dff, (1.0 / dff) ** 0.5)
    b2 = draw(rng, 1, dm, 0.01)
    A2 = draw(rng, r, dff, (1.0 / dff) ** 0.5)
    B2 = draw(rng, dm, r, 0.02)
    up = Linear("c2_ffn_up", X1, W1, b1, [Patch(A1, B1, 64.0, 0.7)], request_scale=0.5)
    down = Linear("c2_ffn_down", X2, W2, b2, [Patch(A2, B2, 64.0, 0.7)], request_scale=0.5)
    norm = draw(rng, 1, dm, 0.02, mean=1.0)
    dense = {
        "ffn.up.bias.diff_b": (b1, draw(rng, 1, dff, 1e-5), "add"),
        "ffn.down.bias.diff_b": (b2, draw(rng, 1, dm, 1e-5), "add"),
        "norm.weight.diff": (norm, draw(rng, 1, dm, 1e-3), "add"),
    }
    return up, down, dense


def config3(scale: str = "full") -> tuple:
    """4-bit SwiGLU base: gate/up d_model -> d_ff as 2 groups, down d_ff -> d_model,
    4-bit W (64-blocks, fp32 absmax), rank 16 bf16 LoRA (alpha = rank, strength 1),
    with dY ~ N(0, 1) for the closed-form backward.  Returns (gate_up, down)."""
    p = (FULL if scale == "full" else SMALL)[3]
    rng = np.random.default_rng(3)
    T, dm, dff, r = p["T"], p["d_model"], p["d_ff"], p["rank"]
    X = draw(rng, T, dm, 1.0)
    Wgu = draw_nf4(rng, 2 * dff, dm)
    patches = []
    for _ in range(2):
        patches.append(Patch(draw(rng, r, dm, (1.0 / dm) ** 0.5), draw(rng, dff, r, 0.02),
                             float(r), 1.0))
    dY_gu = draw(rng, T, 2 * dff, 1.0)
    gate_up = Linear("c3_nf4_gate_up", X, Wgu, None, patches, groups=2, dY=dY_gu)
    X2 = draw(rng, T, dff, 1.0)
    Wd = draw_nf4(rng, dm, dff)
    pd = Patch(draw(rng, r, dff, (1.0 / dff) ** 0.5), draw(rng, dm, r, 0.02), float(r), 1.0)
    dY_d = draw(rng, T, dm, 1.0)
    down = Linear("c3_nf4_down", X2, Wd, None, [pd], dY=dY_d)
    return gate_up, down


def config4(scale: str = "full") -> tuple:
    """Multi-patch sidecar: d -> d, three summed patches (ranks 16/32/128, weights
    1.0/0.6/-0.3, alpha = rank); the rank-16 patch is an fp32 adapter on bf16
    activations; plus a d x d ``.set_weight`` replacement payload.  Returns
    (linear, set_weight_payload)."""
    p = (FULL if scale == "full" else SMALL)[4]
    rng = np.random.default_rng(4)
    T, d, ranks = p["T"], p["d"], p["ranks"]
    weights = (1.0, 0.6, -0.3)
    X = draw(rng, T, d, 1.0)
    W = draw(rng, d, d, (1.0 / d) ** 0.5)
    patches = []
    for i, (r, wgt) in enumerate(zip(ranks, weights)):
        kind = FP32 if i == 0 else BF16
        A = draw(rng, r, d, (1.0 / d) ** 0.5, kind)
        B = draw(rng, d, r, 0.02, kind)
        patches.append(Patch(A, B, float(r), wgt))
    lin = Linear("c4_sidecar", X, W, None, patches, request_scale=1.0)
    payload = draw(rng, d, d, (1.0 / d) ** 0.5)
    return lin, payload


def wan_qkv_rank128(scale: str = "full") -> Linear:
    """The sglang PR's own Speed Tests shape for Wan2.1 1.3B 480p: stacked q/k/v of the
    1536-wide attention (T = 32760 = 21 x 30 x 52 latent tokens) with a rank-128 adapter
    per group (alpha = 128, strength 1, scale 1), bf16, no bias.  "small" keeps the three
    rank-128 groups at T = 600, in = 256, out = 3 x 320."""
    T, di, do = (32760, 1536, 1536) if scale == "full" else (600, 256, 320)
    G, r = 3, 128
    rng = np.random.default_rng(11)
    X = draw(rng, T, di, 1.0)
    W = draw(rng, G * do, di, (1.0 / di) ** 0.5)
    patches = []
    for _ in range(G):
        A = draw(rng, r, di, (1.0 / di) ** 0.5)
        B = draw(rng, do, r, 0.02)
        patches.append(Patch(A, B, float(r), 1.0))
    return Linear("wan_qkv_rank128", X, W, None, patches, request_scale=1.0, groups=G)


def combined_scale_inputs(lin: Linear):
    """(alpha, rank, strength, request_scale) per patch, as stored (no arithmetic)."""
    return [(p.alpha, p.rank, p.strength, lin.request_scale) for p in lin.patches]


def sample_rows(T: int, n: int, seed: int = 12345) -> np.ndarray:
    """Sorted row indices for spot checks at full size: n random rows plus the first
    and the last 8 rows (the ragged tail of the last 128-row tile)."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    rows.update(range(min(8, T)))
    rows.update(range(max(0, T - 8), T))
    return np.array(sorted(rows), dtype=np.int64)
