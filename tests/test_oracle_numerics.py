"""Pins for the oracle's bf16 encodings: a library routine (torch's cast) and hand
worked ties."""
import numpy as np
import pytest
import torch

from oracle import numerics as nm

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _torch_bits(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_f32_to_bf16_matches_torch_cast_random():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    assert np.array_equal(nm.f32_to_bf16_bits(x), _torch_bits(x))


def test_f32_to_bf16_specials():
    specials = np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0, 3.3895314e38, 3.4028235e38,
                         1e-40, -1e-45, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-23],
                        dtype=np.float32)
    assert np.array_equal(nm.f32_to_bf16_bits(specials), _torch_bits(specials))
    nan = nm.f32_to_bf16_bits(np.array([np.nan], dtype=np.float32))
    assert np.isnan(nm.bf16_bits_to_f32(nan)[0])


def test_bf16_decode_roundtrip_all_patterns():
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = nm.bf16_bits_to_f32(allb)
    fin = np.isfinite(f)
    assert np.array_equal(nm.f32_to_bf16_bits(f[fin]), allb[fin])
    ref = torch.from_numpy(allb.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(f[fin], ref[fin])


def test_f64_to_bf16_ties_and_no_double_rounding():
    one = 1.0
    # bf16 spacing at 1 is 2**-7: 1 + 2**-8 is a tie -> even (1.0);
    # 1 + 3*2**-8 is a tie between 1+2**-7 (odd) and 1+2**-6 (even) -> 1+2**-6
    assert nm.f64_to_bf16_value(np.array([one + 2**-8]))[0] == 1.0
    assert nm.f64_to_bf16_value(np.array([one + 3 * 2**-8]))[0] == 1.0 + 2**-6
    # just above the tie: direct rounding goes up, while a float32 detour would round to
    # the tie first and then to even
    assert nm.f64_to_bf16_value(np.array([one + 2**-8 + 2**-30]))[0] == 1.0 + 2**-7
    assert nm.f64_to_bf16_value(np.array([-(one + 2**-8 + 2**-30)]))[0] == -(1.0 + 2**-7)
    # overflow past the largest finite bf16 after rounding
    assert np.isinf(nm.f64_to_bf16_value(np.array([3.4e38]))[0])


def test_f64_to_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100_000) * np.exp(rng.uniform(-30, 30, 100_000))).astype(np.float32)
    ref = nm.bf16_bits_to_f64(_torch_bits(x))
    assert np.array_equal(nm.f64_to_bf16_value(x.astype(np.float64)), ref)


def test_relative_rms_closed_form():
    y_ref = np.array([3.0, 4.0])          # norm 5
    y = np.array([3.0, 4.0]) + np.array([0.3, -0.4])   # error norm 0.5
    assert abs(nm.relative_rms(y, y_ref) - 0.1) < 1e-15
    assert nm.relative_rms(y_ref, y_ref) == 0.0
