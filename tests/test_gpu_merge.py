"""LoRA merge on the GPU against the FP64 oracle (piper-offload docs, "LoRA merge" and
"Quantized weight support").

bf16 weight: the kernel rounds fl32(s * acc + W) (fp32 accumulation of B A, one fused
multiply-add) to bf16, the oracle rounds the exact W + s B A: the two agree except where the
exact value lies within float32 noise of a bf16 rounding boundary, so nearly every element is
bit-equal and none is further apart than one bf16 ulp plus that float32 noise -- r
accumulation roundings of at most 2^-24 of sum |s B_oj A_ji|, and the rounding of the fused
sum with W (it matters only where W and the update cancel and the result's own ulp is tiny).
4-bit weight: the new block scales agree to float32 accuracy, and the codes agree except where
the oracle's normalised value lies within float32 noise of a decision midpoint (there either
neighbour is valid)."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import merge as om
from oracle import nf4 as onf4
from oracle.lora import decode_patch
from oracle.numerics import bf16_bits_to_f64, to_f64
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _patches(rng, ranks, out, d_in, strengths=None):
    strengths = strengths or [0.8] * len(ranks)
    return [workloads.Patch(workloads.draw(rng, r, d_in, (1.0 / d_in) ** 0.5), workloads.draw(rng, out, r, 0.05),
                            float(r) * 0.5, st) for r, st in zip(ranks, strengths)]


def _bf16_check(W0, got_bits, patches, scale):
    dp = [decode_patch(p) for p in patches]
    W = to_f64(W0)
    want = om.merge_bf16_values(W, dp, scale)
    got = bf16_bits_to_f64(got_bits)
    big = np.maximum(np.abs(got), np.abs(want)).astype(np.float32)
    ulp = np.maximum(np.spacing(big).astype(np.float64) * 2 ** 16, 2.0 ** -133)
    # float32 noise of the kernel's intermediates (see the module docstring)
    terms = sum(abs(p.alpha / p.rank * p.strength * scale) * (np.abs(p.B) @ np.abs(p.A)) for p in dp)
    r = max(p.rank for p in dp)
    noise = 2.0 ** -24 * ((r + 2) * terms + 2 * np.abs(W))
    assert np.all(np.abs(got - want) <= ulp + noise)
    assert np.mean(got == want) >= 0.999


@pytest.mark.parametrize("out,d_in,ranks,scale", [
    (300, 264, [8], 1.0),
    (256, 512, [5], -0.5),          # B rows of 5 elements: the library copies B to a padded buffer
    (520, 1024, [128], 0.5),
    (384, 256, [4, 16, 64], 1.0),   # several adapters: one fp32 update, rounded once
])
def test_merge_bf16(out, d_in, ranks, scale):
    rng = np.random.default_rng(out + d_in)
    W0 = workloads.draw(rng, out, d_in, (1.0 / d_in) ** 0.5)
    ps = _patches(rng, ranks, out, d_in)
    W = gu.dev(W0)
    ads = [wpg.Adapter(gu.dev(p.A), gu.dev(p.B), p.alpha, p.strength) for p in ps]
    wpg.lora_merge(W, ads, scale)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    _bf16_check(W0, _bits(W), ps, scale)


def test_merge_zero_strength_and_unmerge():
    rng = np.random.default_rng(7)
    W0 = workloads.draw(rng, 256, 384, 0.05)
    ps = _patches(rng, [16, 32], 256, 384)
    W = gu.dev(W0)
    ads = [wpg.Adapter(gu.dev(p.A), gu.dev(p.B), p.alpha, 0.0) for p in ps]
    wpg.lora_merge(W, ads, 1.0)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(W), W0.data)                  # nothing to add: untouched
    ads = [wpg.Adapter(gu.dev(p.A), gu.dev(p.B), p.alpha, p.strength) for p in ps]
    wpg.lora_merge(W, ads, 1.0)
    merged = _bits(W).copy()
    wpg.lora_merge(W, ads, -1.0)
    torch.cuda.synchronize()
    back = bf16_bits_to_f64(_bits(W))
    orig = bf16_bits_to_f64(W0.data)
    big = np.maximum(np.abs(orig), np.abs(bf16_bits_to_f64(merged))).astype(np.float32)
    assert np.all(np.abs(back - orig) <= np.spacing(big).astype(np.float64) * 2 ** 16 + 2.0 ** -133)
    assert not np.array_equal(merged, W0.data)


@pytest.mark.parametrize("rows,cols,scale,ranks", [
    (256, 512, 1.0, [16]),
    (200, 320, 40.0, [16]),                 # columns not a multiple of 256: 64-column tiles
    (200, 768, 30.0, [16]),                 # ragged row tile, three 256-column tiles a row
    (384, 1024, 20.0, [16, 100, 8]),        # three adapters, two K blocks: one operand stage
    (128, 256, 20.0, [256]),                # four K blocks: the 64-column form again
    (2560, 4096, 10.0, [32]),               # more tiles than SMs: each CTA takes two or three
])
def test_merge_nf4(rows, cols, scale, ranks):
    rng = np.random.default_rng(rows + cols)
    W0 = workloads.draw_nf4(rng, rows, cols)
    ps = _patches(rng, ranks, rows, cols)
    W = gu.dev(W0)
    ads = [wpg.Adapter(gu.dev(p.A), gu.dev(p.B), p.alpha, p.strength) for p in ps]
    wpg.lora_merge(W, ads, scale)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    got_codes = onf4.unpack_codes(W.packed.cpu().numpy(), rows, cols)
    got_am = W.absmax.cpu().numpy()
    want_codes, want_am, x = om.merge_nf4(W0.data, W0.absmax, rows, cols, [decode_patch(p) for p in ps], scale)
    np.testing.assert_allclose(got_am, want_am, rtol=1e-5, atol=0)
    lv = onf4.codebook_f64()
    mids = (lv[:-1] + lv[1:]) / 2
    near = np.min(np.abs(x[..., None].astype(np.float64) - mids), axis=-1) <= 1e-5
    assert np.array_equal(got_codes[~near], want_codes[~near])
    assert np.all(np.abs(got_codes.astype(int) - want_codes.astype(int)) <= 1)
    if scale > 1:
        orig = onf4.unpack_codes(W0.data, rows, cols)
        assert np.mean(got_codes != orig) > 0.01                # the update moved codes


@pytest.mark.parametrize("rows,cols,scale,ranks", [
    (256, 512, 1.0, [16]),                  # 256-column tiles
    (200, 320, 40.0, [16]),                 # 64-column tiles
    (384, 1024, 20.0, [16, 100, 8]),        # several adapters
    (128, 256, 20.0, [300]),                # a rank above 256: the three-kernel route
    (2560, 4096, 10.0, [32]),               # more tiles than SMs
])
def test_merge_nf4_stochastic(rows, cols, scale, ranks):
    """The stochastic re-encoding against the oracle's, element by element: equal codes
    wherever the oracle's decision is further than float32 noise from flipping (its slack),
    equal scales; the same seed gives the same codes, another seed others."""
    rng = np.random.default_rng(rows + cols + 1)
    W0 = workloads.draw_nf4(rng, rows, cols)
    ps = _patches(rng, ranks, rows, cols)
    ads = [wpg.Adapter(gu.dev(p.A), gu.dev(p.B), p.alpha, p.strength) for p in ps]
    seed = 0x9E3779B97F4A7C15 + rows
    got = []
    for sd in (seed, seed, seed + 1):
        W = gu.dev(W0)
        wpg.lora_merge(W, ads, scale, rounding_seed=sd)
        torch.cuda.synchronize()
        assert wpg.lora_device_status() == 0
        got.append((onf4.unpack_codes(W.packed.cpu().numpy(), rows, cols), W.absmax.cpu().numpy()))
    want_codes, want_am, x, slack = om.merge_nf4(W0.data, W0.absmax, rows, cols, [decode_patch(p) for p in ps],
                                                 scale, rounding_seed=seed)
    codes, am = got[0]
    np.testing.assert_allclose(am, want_am, rtol=1e-5, atol=0)
    sure = slack > 1e-5
    assert sure.mean() > 0.99
    assert np.array_equal(codes[sure], want_codes[sure])
    assert np.all(np.abs(codes.astype(int) - want_codes.astype(int)) <= 1)
    assert np.array_equal(codes, got[1][0])                    # the same seed, the same codes
    other = om.merge_nf4(W0.data, W0.absmax, rows, cols, [decode_patch(p) for p in ps], scale,
                         rounding_seed=seed + 1)[0]
    moved = np.mean(want_codes != other)                       # another seed samples anew
    assert moved > 0 and np.mean(codes != got[2][0]) > 0.5 * moved


def test_merge_full_size_sidecar():
    """The 5120 x 5120 sidecar weight with its rank-128 patch (bf16), every element checked."""
    lin, _ = workloads.config4("full")
    W0 = lin.W
    p = lin.patches[2]                                           # rank 128, bf16
    W = gu.dev(W0)
    wpg.lora_merge(W, [wpg.Adapter(gu.dev(p.A), gu.dev(p.B), p.alpha, p.strength)], 1.0)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    _bf16_check(W0, _bits(W), [p], 1.0)
