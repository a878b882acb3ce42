"""GPU parity of the fused forward against the CPU FP64 oracle, through the C ABI.

Tolerances (from the method's accuracy gate): bf16 outputs within relative RMS 4e-3 and
no worse than the unfused bf16 chain that materialises the delta; FP32 cases within
1e-5.  Every output element is also held to the element-wise bound of the single-rounding
design (tests/gpu_util.py), so a single wrong element fails."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import lora as olora
from oracle.numerics import relative_rms
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

BF16_TOL = 4e-3
FP32_TOL = 1e-5


def _gate(err, chain):
    assert err <= BF16_TOL, err
    assert err <= chain, (err, chain)


def test_c0_tiny_fp32():
    lin = workloads.config0()
    Y = gu.run_fwd(lin, out_dtype=torch.float32)
    want = olora.reference_output(lin)
    err = relative_rms(gu.to_f64(Y), want)
    assert err <= FP32_TOL, err
    gu.assert_elementwise(gu.to_f64(Y), want, gu.fwd_bound(lin, out_f32=True, y_ref=want), lin.name)


def test_c1_grouped_small():
    lin = workloads.config1("small")
    Y = gu.run_fwd(lin)
    _gate(*gu.errors(lin, Y))
    assert wpg.lora_device_status() == 0


def test_c2_ffn_small_with_bias():
    up, down, _ = workloads.config2("small")
    for lin in (up, down):
        Y = gu.run_fwd(lin)
        _gate(*gu.errors(lin, Y))


def test_c4_multipatch_small():
    lin, _ = workloads.config4("small")
    Y = gu.run_fwd(lin)
    _gate(*gu.errors(lin, Y))


def test_c4_fp32_adapter_fp32_output():
    lin, _ = workloads.config4("small")
    lin.patches = lin.patches[:1]            # the fp32 adapter alone, on the bf16 layer
    Y = gu.run_fwd(lin, out_dtype=torch.float32)
    want = olora.reference_output(lin)
    err = relative_rms(gu.to_f64(Y), want)
    assert err <= FP32_TOL, err
    gu.assert_elementwise(gu.to_f64(Y), want, gu.fwd_bound(lin, out_f32=True, y_ref=want), "fp32 adapter")
    # delta only (no base weight): the fp32 adapter's contribution by itself
    Yd = gu.run_fwd(lin, out_dtype=torch.float32, with_base=False)
    X, _, _, patches = olora.decode_linear(lin)
    want = olora.linear_fwd(X, None, None, patches, lin.request_scale, out_features=lin.out_features)
    err = relative_rms(gu.to_f64(Yd), want)
    assert err <= FP32_TOL, err
    gu.assert_elementwise(gu.to_f64(Yd), want, gu.fwd_bound(lin, out_f32=True, y_ref=want, with_base=False),
                          "fp32 adapter, delta only")


@pytest.mark.parametrize("T,K,N,r,xkind", [(77, 70, 40, 5, workloads.FP32), (131, 200, 96, 24, workloads.FP32),
                                           (300, 200, 264, 20, workloads.BF16), (70, 64, 48, 40, workloads.BF16)])
def test_fp32_adapter_odd_shapes(T, K, N, r, xkind):
    """FP32 adapters with ragged K (partial chunks, unaligned rows) and rank widths that
    span one or two column blocks of the rank projection; all-fp32 and bf16 layers."""
    rng = np.random.default_rng(T + K + r)
    X = workloads.draw(rng, T, K, 1.0, xkind)
    W = workloads.draw(rng, N, K, (1.0 / K) ** 0.5, xkind)
    A = workloads.draw(rng, r, K, (1.0 / K) ** 0.5, workloads.FP32)
    B = workloads.draw(rng, N, r, 0.02, workloads.FP32)
    lin = workloads.Linear("odd32", X, W, None, [workloads.Patch(A, B, float(r), 0.8)], request_scale=1.3)
    Y = gu.run_fwd(lin, out_dtype=torch.float32)
    want = olora.reference_output(lin)
    err = relative_rms(gu.to_f64(Y), want)
    assert err <= FP32_TOL, err
    gu.assert_elementwise(gu.to_f64(Y), want, gu.fwd_bound(lin, out_f32=True, y_ref=want), lin.name)


def test_fp32_output_bf16_adapters():
    lin = workloads.config1("small")
    Y = gu.run_fwd(lin, out_dtype=torch.float32)
    err, _ = gu.errors(lin, Y)
    # one bf16 rounding of s * X A^T remains; the base is exact to fp32 accumulation
    assert err <= 2e-3, err


def test_zero_scale_equals_no_adapter_bitwise():
    lin = workloads.config1("small")
    X, W = gu.dev(lin.X), gu.dev(lin.W)
    ads = gu.adapters(lin)
    y0 = wpg.lora_linear_fwd_grouped(X, W, None, ads, 0.0)
    zero = [wpg.Adapter(a.A, a.B, a.alpha, 0.0) for a in ads]
    y1 = wpg.lora_linear_fwd_grouped(X, W, None, zero, 1.0)
    # base only, through the plain entry with no adapters
    y2 = wpg.lora_linear_fwd(X, W, None, [])
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_delta_linear_in_scale():
    lin = workloads.config1("small")
    X, W = gu.dev(lin.X), gu.dev(lin.W)
    ads = gu.adapters(lin)
    base = wpg.lora_linear_fwd(X, W, None, [], out_dtype=torch.float32)
    y1 = wpg.lora_linear_fwd_grouped(X, W, None, ads, 0.25, out_dtype=torch.float32)
    y2 = wpg.lora_linear_fwd_grouped(X, W, None, ads, 0.5, out_dtype=torch.float32)
    d1, d2 = (y1 - base).double(), (y2 - base).double()
    # s * H is rounded to bf16 once, so doubling s doubles the delta exactly up to fp32 sums
    assert float(((d2 - 2 * d1).norm() / d2.norm()).item()) < 1e-5


def test_multi_patch_is_sum_of_single_patches():
    lin, _ = workloads.config4("small")
    lin.patches = lin.patches[1:]           # the two bf16 patches
    X, W = gu.dev(lin.X), gu.dev(lin.W)
    ads = gu.adapters(lin)
    base = wpg.lora_linear_fwd(X, W, None, [], out_dtype=torch.float32).double()
    both = wpg.lora_linear_fwd(X, W, None, ads, out_dtype=torch.float32).double() - base
    one = sum(wpg.lora_linear_fwd(X, W, None, [a], out_dtype=torch.float32).double() - base for a in ads)
    assert float(((both - one).norm() / both.norm()).item()) < 1e-5


@pytest.mark.parametrize("T,K,N,r", [(1, 64, 256, 8), (127, 200, 520, 16), (129, 64, 8, 8),
                                     (300, 72, 264, 24), (640, 1024, 768, 96), (256, 128, 256, 256)])
def test_edge_shapes(T, K, N, r):
    rng = np.random.default_rng(T * 7 + K)
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    A = workloads.draw(rng, r, K, (1.0 / K) ** 0.5)
    B = workloads.draw(rng, N, r, 0.02)
    bias = workloads.draw(rng, 1, N, 0.01)
    lin = workloads.Linear("edge", X, W, bias, [workloads.Patch(A, B, float(2 * r), 0.9)], request_scale=0.7)
    Y = gu.run_fwd(lin)
    _gate(*gu.errors(lin, Y))


@pytest.mark.parametrize("ranks", [(128, 64, 48), (136, 32, 8), (8, 8, 8, 8, 8), (120,), (40, 24)])
def test_rank_mixes(ranks):
    """Rank mixes that place whole adapters on either CTA of the pair (lopsided or even
    halves) and ones that must split every adapter between the two halves."""
    rng = np.random.default_rng(sum(ranks))
    T, K, N = 520, 192, 384
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    patches = [workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5), workloads.draw(rng, N, r, 0.02),
                               float(r), 0.5 + 0.1 * i) for i, r in enumerate(ranks)]
    lin = workloads.Linear("mix", X, W, None, patches, request_scale=1.1)
    Y = gu.run_fwd(lin)
    _gate(*gu.errors(lin, Y))


@pytest.mark.parametrize("ranks,nf4", [((200, 200, 48), False), ((256, 64), False), ((256, 256, 256, 256), False),
                                       ((128, 128, 64), True), ((104, 32, 88, 48, 72), False)])
def test_rank_passes(ranks, nf4):
    """Adapters whose rank columns exceed one 256-column accumulator: s X A^T comes from
    several rank passes per row block (adapters grouped whole, first-fit), with a 4-bit
    weight too."""
    rng = np.random.default_rng(sum(ranks) + nf4)
    T, K, N = 600, 256, 384
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw_nf4(rng, N, K) if nf4 else workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    bias = workloads.draw(rng, 1, N, 0.01)
    patches = [workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5), workloads.draw(rng, N, r, 0.02),
                               float(r), 0.3 + 0.2 * i) for i, r in enumerate(ranks)]
    lin = workloads.Linear("passes", X, W, bias, patches, request_scale=0.9)
    Y = gu.run_fwd(lin)
    assert wpg.lora_device_status() == 0
    _gate(*gu.errors(lin, Y))


def test_rank_passes_with_fp32_adapter():
    """An FP32 adapter beside bf16 adapters of more than 256 rank columns: the bf16 ones take
    two rank passes, the FP32 one the CUDA-core route; fp32 output to 1e-5."""
    rng = np.random.default_rng(31)
    T, K, N = 300, 192, 264
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    patches = [workloads.Patch(workloads.draw(rng, 16, K, (1.0 / K) ** 0.5, workloads.FP32),
                               workloads.draw(rng, N, 16, 0.02, workloads.FP32), 16.0, 1.0)]
    patches += [workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5), workloads.draw(rng, N, r, 0.02),
                                float(r), 0.6) for r in (160, 128)]
    lin = workloads.Linear("passes32", X, W, None, patches, request_scale=1.0)
    Y = gu.run_fwd(lin)
    _gate(*gu.errors(lin, Y))
    Y32 = gu.run_fwd(lin, out_dtype=torch.float32)
    gu.errors(lin, Y32)                       # element-wise bound at fp32 output


def test_wan_rank128_small():
    """The pages' Wan2.1 adapter shape (rank 128 on each of q, k, v: 384 rank columns, two
    rank passes) at a small size."""
    lin = workloads.wan_qkv_rank128("small")
    Y = gu.run_fwd(lin)
    assert wpg.lora_device_status() == 0
    _gate(*gu.errors(lin, Y))


def test_rank_without_aligned_pitch_is_rejected():
    X = torch.zeros(16, 64, dtype=torch.bfloat16, device=gu.DEV)
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device=gu.DEV)
    A = torch.zeros(3, 64, dtype=torch.bfloat16, device=gu.DEV)
    B = torch.zeros(64, 3, dtype=torch.bfloat16, device=gu.DEV)   # row pitch 3: not TMA-able
    with pytest.raises(wpg.WeightPatchesError) as e:
        wpg.lora_linear_fwd(X, W, None, [wpg.Adapter(A, B, 3.0)])
    assert e.value.status == -4
    # the same adapter with a padded pitch works
    Bp = torch.zeros(64, 8, dtype=torch.bfloat16, device=gu.DEV)[:, :3]
    Ap = torch.zeros(3, 64, dtype=torch.bfloat16, device=gu.DEV)
    wpg.lora_linear_fwd(X, W, None, [wpg.Adapter(Ap, Bp, 3.0)])
    torch.cuda.synchronize()


def test_no_worse_than_torch_unfused_chain():
    lin = workloads.config1("small")
    Y = gu.run_fwd(lin)
    want = olora.reference_output(lin)
    gu.assert_elementwise(gu.to_f64(Y), want, gu.fwd_bound(lin, y_ref=want), lin.name)
    err = relative_rms(gu.to_f64(Y), want)
    chain = relative_rms(gu.to_f64(gu.torch_unfused_chain(lin)), want)
    assert err <= chain, (err, chain)


# ----------------------------------------------------------------- full sizes (spot checks)
def test_c1_full_sampled_rows():
    lin = workloads.config1("full")
    Y = gu.run_fwd(lin)
    rows = workloads.sample_rows(lin.T, 192)
    _gate(*gu.errors(lin, Y, rows))


def test_c2_full_sampled_rows():
    up, down, _ = workloads.config2("full")
    for lin in (up, down):
        Y = gu.run_fwd(lin)
        rows = workloads.sample_rows(lin.T, 96)
        _gate(*gu.errors(lin, Y, rows))


def test_c4_full_sampled_rows():
    lin, _ = workloads.config4("full")
    Y = gu.run_fwd(lin)
    rows = workloads.sample_rows(lin.T, 96)
    _gate(*gu.errors(lin, Y, rows))


def test_c4_fp32_adapter_full_sampled_rows():
    """The FP32 adapter of C4 at full size (T = 8192, 5120 -> 5120, rank 16, fp32 A and B on
    bf16 activations; three bf16 pieces on the tensor cores): fp32 output, with and without the
    base weight, on sampled rows against the FP64 definition -- the same 1e-5 gate as the small
    case, and every element within its bound."""
    lin, _ = workloads.config4("full")
    lin.patches = lin.patches[:1]
    rows = workloads.sample_rows(lin.T, 64)
    Y = gu.run_fwd(lin, out_dtype=torch.float32)
    want = olora.reference_output(lin, rows)
    got = gu.to_f64(Y)[rows]
    assert relative_rms(got, want) <= FP32_TOL
    gu.assert_elementwise(got, want, gu.fwd_bound(lin, rows, out_f32=True, y_ref=want), "fp32 adapter, full size")
    Yd = gu.run_fwd(lin, out_dtype=torch.float32, with_base=False)
    X, _, _, patches = olora.decode_linear(lin, rows)
    want = olora.linear_fwd(X, None, None, patches, lin.request_scale, out_features=lin.out_features)
    got = gu.to_f64(Yd)[rows]
    assert relative_rms(got, want) <= FP32_TOL
    gu.assert_elementwise(got, want, gu.fwd_bound(lin, rows, out_f32=True, y_ref=want, with_base=False),
                          "fp32 adapter, full size, delta only")


def test_wan_rank128_full_sampled_rows():
    """The sglang PR's Wan2.1 1.3B 480p Speed Tests shape: T = 32760, 1536 -> 3 x 1536, rank
    128 per group."""
    lin = workloads.wan_qkv_rank128("full")
    Y = gu.run_fwd(lin)
    assert wpg.lora_device_status() == 0
    rows = workloads.sample_rows(lin.T, 128)
    _gate(*gu.errors(lin, Y, rows))
