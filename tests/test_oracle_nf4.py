"""Pins for the oracle's 4-bit NormalFloat table and dequantisation.

The table is checked against the properties the QLoRA NormalFloat construction fixes
(16 levels, one exact zero, endpoints +-1, 8 positive and 7 negative levels) and
against the normal distribution through the forward CDF (scipy), which the oracle does
not use: mapped back to probabilities, the levels must be evenly spaced."""
import struct

import numpy as np
import pytest
import torch
from scipy.special import ndtr, ndtri

from oracle import nf4
from oracle.numerics import bf16_bits_to_f64


def test_codebook_shape_and_order():
    cb = nf4.codebook_f64()
    assert cb.shape == (16,)
    assert np.all(np.diff(cb) > 0)
    assert cb[0] == -1.0 and cb[-1] == 1.0
    assert np.count_nonzero(cb == 0.0) == 1
    assert np.count_nonzero(cb > 0) == 8 and np.count_nonzero(cb < 0) == 7
    assert cb[7] == 0.0


def test_codebook_levels_are_evenly_spaced_normal_quantiles():
    cb = nf4.codebook_f64()
    delta = nf4.upper_probability()
    z_top = ndtri(delta)                 # scipy's inverse, not the oracle's
    pos = cb[cb > 0][::-1]               # descending: delta, delta - step, ...
    neg = -cb[cb < 0]                    # descending magnitudes
    p_pos = ndtr(pos * z_top)
    p_neg = ndtr(neg * z_top)
    assert np.allclose(p_pos, delta - np.arange(8) * (delta - 0.5) / 8, atol=1e-13, rtol=0)
    assert np.allclose(p_neg, delta - np.arange(7) * (delta - 0.5) / 7, atol=1e-13, rtol=0)
    # the first step below 1/2 is not a level (the zero is shared once)
    assert abs(delta - 0.9677083333333333) < 1e-15


def test_codebook_f32_is_the_float32_rounding():
    assert np.array_equal(nf4.codebook_f32(), nf4.codebook_f64().astype(np.float32))


def test_nibble_order_and_pack_roundtrip():
    packed = np.array([[0xA3, 0x0F]], dtype=np.uint8)
    codes = nf4.unpack_codes(packed, 1, 4)
    assert codes.tolist() == [[10, 3, 0, 15]]
    rng = np.random.default_rng(0)
    c = rng.integers(0, 16, size=(5, 128), dtype=np.uint8)
    assert np.array_equal(nf4.unpack_codes(nf4.pack_codes(c), 5, 128), c)


def _scalar_dequant_bits(code_value_f32: float, absmax: float) -> int:
    """One element by hand: float32 product via struct, bf16 rounding via torch."""
    prod = struct.unpack("f", struct.pack("f", code_value_f32 * absmax))[0]
    return int(torch.tensor([prod], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


def test_dequant_brute_force_all_codes():
    cb = nf4.codebook_f32()
    absmaxes = np.array([1.0, 0.3712, 2.5e-3, 7.75, 1e-20, 3.1e4], dtype=np.float32)
    rows, cols = len(absmaxes), 64
    codes = np.tile(np.arange(16, dtype=np.uint8), (rows, 4))
    packed = nf4.pack_codes(codes)
    bits = nf4.dequant_bf16_bits(packed, absmaxes, rows, cols)
    for r in range(rows):
        for c in range(cols):
            # the float32 product of two float32 values is exact in float64, so
            # struct's float32 rounding of the f64 product is the IEEE float32 product
            want = _scalar_dequant_bits(float(cb[codes[r, c]]) * float(absmaxes[r]), 1.0)
            assert int(bits[r, c]) == want


def test_dequant_endpoints_and_block_index():
    rows, cols = 3, 192                   # 3 blocks per row
    absmax = np.arange(1, 10, dtype=np.float32) * np.float32(0.5)  # distinct per block
    codes = np.full((rows, cols), 15, dtype=np.uint8)                # level +1
    w = nf4.dequant_f64(nf4.pack_codes(codes), absmax, rows, cols)
    for o in range(rows):
        for i in range(cols):
            blk = (o * cols + i) // 64
            assert w[o, i] == float(absmax[blk])  # multiples of 0.5 are exact in bf16
    codes[:] = 7                                  # the zero level
    assert np.all(nf4.dequant_f64(nf4.pack_codes(codes), absmax, rows, cols) == 0.0)
    codes[:] = 0                                  # level -1
    w = nf4.dequant_f64(nf4.pack_codes(codes), absmax, rows, cols)
    assert w[2, 191] == -float(absmax[8])


def test_dequant_values_are_bf16():
    rng = np.random.default_rng(5)
    packed = rng.integers(0, 256, size=(4, 64), dtype=np.uint8)
    absmax = np.abs(rng.standard_normal(8).astype(np.float32))
    bits = nf4.dequant_bf16_bits(packed, absmax, 4, 128)
    w = bf16_bits_to_f64(bits)
    assert np.array_equal(w.astype(np.float32).astype(np.float64), w)
    with pytest.raises(Exception):
        nf4.dequant_bf16_bits(packed, absmax[:3], 4, 128)
