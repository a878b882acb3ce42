"""Pins of the merge oracle (piper-offload docs, "LoRA merge"): the requantisation rule
against brute force, the 4-bit round trip, zero strength, merge/unmerge, and the merged
weight reproducing the unmerged forward."""
import numpy as np

from oracle import merge as om
from oracle import nf4 as onf4
from oracle.lora import DecodedPatch, linear_fwd
from oracle.numerics import bf16_bits_to_f64, f32_to_bf16_bits, f64_to_bf16_value


def _patch(rng, r, d_in, d_out, alpha=8.0, strength=0.7):
    A = f64_to_bf16_value(rng.normal(0, (1.0 / d_in) ** 0.5, (r, d_in)))
    B = f64_to_bf16_value(rng.normal(0, 0.05, (d_out, r)))
    return DecodedPatch(A, B, alpha, strength)


def test_midpoint_rule_is_nearest_level():
    rng = np.random.default_rng(0)
    x = rng.uniform(-1.0, 1.0, 200000).astype(np.float32)
    mid = om.midpoints_f32()
    x = np.concatenate([x, mid, np.nextafter(mid, np.float32(2)), np.nextafter(mid, np.float32(-2)),
                        np.array([-1, 1, 0], dtype=np.float32)]).astype(np.float32)
    # one block per value, its absmax forced to 1 by a 1.0 entry
    n = len(x)
    blocks = np.zeros((n, 64), dtype=np.float32)
    blocks[:, 0] = 1.0
    blocks[:, 1] = x
    codes, m, xs = om.quantize_blocks(blocks)
    assert np.all(m == 1.0)
    got = codes[:, 1]
    want = om.nearest_level_brute(x)
    # the two rules can differ only within one float32 ulp of a midpoint (the midpoint itself
    # is rounded to float32); everywhere else they agree
    lv = onf4.codebook_f64()
    exact_mid = (lv[:-1] + lv[1:]) / 2
    near = np.min(np.abs(x[:, None].astype(np.float64) - exact_mid[None, :]), axis=1) <= \
        np.spacing(np.abs(x).astype(np.float32)).astype(np.float64)
    assert np.array_equal(got[~near], want[~near])
    assert np.all(np.abs(got.astype(int) - want.astype(int)) <= 1)
    # a value exactly on a (float32) midpoint takes the lower code
    on_mid = np.isin(x, mid)
    assert np.array_equal(got[on_mid], np.searchsorted(mid, x[on_mid], side="left").astype(np.uint8))


def test_requantise_round_trip():
    # blocks that hold level +1 (code 15): dequantise then requantise gives the same codes and
    # absmax' = bf16(absmax)
    rng = np.random.default_rng(1)
    rows, cols = 8, 256
    codes = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
    codes[:, ::64] = 15
    absmax = np.abs(rng.normal(0, 1, rows * cols // 64)).astype(np.float32) + np.float32(0.01)
    packed = onf4.pack_codes(codes)
    W = onf4.dequant_f64(packed, absmax, rows, cols).astype(np.float32)
    c2, m2, _ = om.quantize_blocks(W)
    assert np.array_equal(c2, codes)
    # the new scale is the block's largest |value|: level 15 is 1, so bf16(absmax)
    assert onf4.codebook_f32()[15] == 1.0
    np.testing.assert_array_equal(m2, bf16_bits_to_f64(f32_to_bf16_bits(absmax)).astype(np.float32))


def test_zero_block_and_zero_update():
    c, m, _ = om.quantize_blocks(np.zeros((2, 128), dtype=np.float32))
    assert np.all(c == 7) and np.all(m == 0)
    rng = np.random.default_rng(2)
    W = f64_to_bf16_value(rng.normal(0, 0.1, (40, 64)))
    p = _patch(rng, 4, 64, 40, strength=0.0)
    assert np.array_equal(om.merge_bf16_values(W, [p], 1.0), W)


def test_merge_then_unmerge_within_one_rounding():
    rng = np.random.default_rng(3)
    W = f64_to_bf16_value(rng.normal(0, 0.1, (96, 128)))
    ps = [_patch(rng, 8, 128, 96), _patch(rng, 16, 128, 96, alpha=16.0, strength=-0.4)]
    W1 = om.merge_bf16_values(W, ps, 1.0)
    W2 = om.merge_bf16_values(W1, ps, -1.0)
    # two roundings: |W2 - W| is at most one bf16 ulp at the larger of |W| and |W1|
    big = np.maximum(np.abs(W), np.abs(W1)).astype(np.float32)
    ulp = np.spacing(big).astype(np.float64) * 2 ** 16
    assert np.all(np.abs(W2 - W) <= ulp)
    assert np.any(W1 != W)


def test_merged_weight_reproduces_the_forward():
    # the forward is linear (Unsloth walkthrough, section 2): X (W + sum s B A)^T equals the
    # unmerged X W^T + sum s (X A^T) B^T exactly in float64
    rng = np.random.default_rng(4)
    X = rng.normal(0, 1, (5, 48))
    W = rng.normal(0, 0.2, (32, 48))
    ps = [_patch(rng, 4, 48, 32), _patch(rng, 6, 48, 32, alpha=3.0, strength=1.3)]
    merged = X @ (W + om.update(ps, 0.9)).T
    np.testing.assert_allclose(merged, linear_fwd(X, W, None, ps, 0.9), rtol=1e-12, atol=1e-12)


def test_nf4_merge_small_update_keeps_codes():
    # an update far below every decision margin leaves the codes as they were (blocks holding
    # level +1 keep their scale up to the update)
    rng = np.random.default_rng(5)
    rows, cols = 16, 128
    codes = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
    codes[:, ::64] = 15
    absmax = (np.abs(rng.normal(0, 1, rows * cols // 64)) + 0.5).astype(np.float32)
    p = DecodedPatch(np.full((1, cols), 1e-6), np.full((rows, 1), 1e-6), 1.0, 1.0)
    c2, m2, _ = om.merge_nf4(onf4.pack_codes(codes), absmax, rows, cols, [p], 1.0)
    assert np.array_equal(c2, codes)
