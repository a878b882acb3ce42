"""Pins for the oracle's dense patch (.diff / .diff_b / .set_weight): worked examples
from the FastVideo DenseLoRAPatch page, torch's float32 tensor ops as an independent
library, and invariants."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import dense_patch as dp
from oracle.numerics import bf16_bits_to_f32


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "dense_patch_examples.json")) as f:
        return json.load(f)["cases"]


def test_golden_cases(golden_dir):
    for c in _golden(golden_dir):
        if c.get("kind") == "set":
            got = dp.apply_set(np.array(c["payload_bits"], dtype=np.uint16), c["payload_kind"],
                               c["param_kind"], c["strength"])
            assert got.tolist() == c["expect_bits"], c["name"]
            continue
        if c["param_kind"] == "fp32":
            param = np.array(c["param"], dtype=np.float32)
        else:
            param = np.array(c["param_bits"], dtype=np.uint16)
        delta = np.array(c["delta_bits"], dtype=np.uint16)
        got = dp.apply_diff(param, c["param_kind"], delta, c["delta_kind"], c["strength"])
        if "expect_f32" in c:
            assert got.tolist() == c["expect_f32"], c["name"]
        else:
            assert got.tolist() == c["expect_bits"], c["name"]


def _t_bf16(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("strength", [1.0, 0.8, -0.3, 1e-3, 0.7000000000000001])
def test_diff_matches_torch_float32_ops(strength):
    rng = np.random.default_rng(11)
    p = rng.integers(0, 65536, size=50_000, dtype=np.uint32).astype(np.uint16)
    p = p[np.isfinite(bf16_bits_to_f32(p))]
    d = (rng.standard_normal(p.size) * 1e-3).astype(np.float32)
    d_bits = _bits(torch.from_numpy(d).to(torch.bfloat16))
    got = dp.apply_diff(p, "bf16", d_bits, "bf16", strength)
    ref = (_t_bf16(p).to(torch.float32) + _t_bf16(d_bits).to(torch.float32) * strength).to(torch.bfloat16)
    assert np.array_equal(got, _bits(ref))
    # float32 parameter, float32 delta
    p32 = rng.standard_normal(4096).astype(np.float32)
    got32 = dp.apply_diff(p32, "fp32", d[:4096], "fp32", strength)
    ref32 = torch.from_numpy(p32) + torch.from_numpy(d[:4096]) * strength
    assert np.array_equal(got32.view(np.uint32), ref32.numpy().view(np.uint32))


def test_diff_exhaustive_over_one_binade():
    # every bf16 in [1, 2) plus every delta in a small set, all signs of strength
    p = (np.arange(128, dtype=np.uint16) | np.uint16(0x3F80))
    for dval in [2**-8, 2**-9, 3 * 2**-9, -2**-8, 1e-3, -5e-4]:
        d = np.full(p.size, dval, dtype=np.float32)
        d_bits = _bits(torch.from_numpy(d).to(torch.bfloat16))
        for k in [1.0, -1.0, 0.5, 2.0]:
            got = dp.apply_diff(p, "bf16", d_bits, "bf16", k)
            ref = (_t_bf16(p).float() + _t_bf16(d_bits).float() * k).to(torch.bfloat16)
            assert np.array_equal(got, _bits(ref))


def test_set_matches_torch_and_identity_at_unit_strength():
    rng = np.random.default_rng(2)
    v = _bits(torch.from_numpy(rng.standard_normal(10_000).astype(np.float32)).to(torch.bfloat16))
    assert np.array_equal(dp.apply_set(v, "bf16", "bf16", 1.0), v)
    for k in [0.8, -0.3, 1.7]:
        ref = (_t_bf16(v).float() * k).to(torch.bfloat16)
        assert np.array_equal(dp.apply_set(v, "bf16", "bf16", k), _bits(ref))


def test_zero_strength_and_zero_delta_leave_param():
    rng = np.random.default_rng(4)
    p = _bits(torch.from_numpy(rng.standard_normal(1000).astype(np.float32)).to(torch.bfloat16))
    d = _bits(torch.from_numpy(rng.standard_normal(1000).astype(np.float32)).to(torch.bfloat16))
    assert np.array_equal(dp.apply_diff(p, "bf16", d, "bf16", 0.0), p)
    zeros = np.zeros_like(d)
    assert np.array_equal(dp.apply_diff(p, "bf16", zeros, "bf16", 0.9), p)


def test_errors():
    p = np.zeros(4, dtype=np.uint16)
    with pytest.raises(dp.PatchError):
        dp.apply_diff(p, "bf16", np.zeros(5, dtype=np.uint16), "bf16", 1.0)
    with pytest.raises(dp.PatchError):
        dp.apply_diff(p, "bf16", p, "bf16", float("nan"))
    with pytest.raises(dp.PatchError):
        dp.apply_set(p, "bf16", "bf16", float("inf"))
    with pytest.raises(dp.PatchError):
        dp.apply_set(p, "bf16", "bf16", 1.0, param_shape=(5,))
