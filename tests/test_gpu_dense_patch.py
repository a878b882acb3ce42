"""GPU dense patch (.diff / .diff_b / .set_weight) against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import dense_patch as odp
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(gu.DEV)


@pytest.mark.parametrize("scale", ["small", "full"])
def test_c2_diffs(scale):
    _, _, dense = workloads.config2(scale)
    for name, (param, payload, kind) in dense.items():
        p = _bf16_dev(param.data.reshape(-1))
        d = _bf16_dev(payload.data.reshape(-1))
        wpg.lora_dense_patch(p, d, wpg.WP_PATCH_ADD, 1.0)
        torch.cuda.synchronize()
        want = odp.apply_diff(param.data.reshape(-1), "bf16", payload.data.reshape(-1), "bf16", 1.0)
        assert np.array_equal(_bits(p), want), name


@pytest.mark.parametrize("strength", [1.0, 0.8])
def test_c4_set_weight_full(strength):
    _, payload = workloads.config4("full")
    p = torch.empty(payload.rows, payload.cols, dtype=torch.bfloat16, device=gu.DEV)
    d = _bf16_dev(payload.data)
    wpg.lora_dense_patch(p, d, wpg.WP_PATCH_SET, strength)
    torch.cuda.synchronize()
    want = odp.apply_set(payload.data, "bf16", "bf16", strength)
    assert np.array_equal(_bits(p), want)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 4097, 1_000_003])
@pytest.mark.parametrize("strength", [1.0, -0.3, 0.7000000000000001])
def test_ragged_and_unaligned(n, strength):
    rng = np.random.default_rng(n)
    p_bits = workloads.draw(rng, 1, n + 1, 1.0).data.reshape(-1)
    d_bits = workloads.draw(rng, 1, n + 1, 1e-3).data.reshape(-1)
    for off in (0, 1):                           # off = 1 forces the unaligned scalar path
        p = _bf16_dev(p_bits)[off:off + n]
        d = _bf16_dev(d_bits)[off:off + n]
        wpg.lora_dense_patch(p, d, wpg.WP_PATCH_ADD, strength)
        torch.cuda.synchronize()
        want = odp.apply_diff(p_bits[off:off + n], "bf16", d_bits[off:off + n], "bf16", strength)
        assert np.array_equal(_bits(p), want)


def test_fp32_param_and_mixed_payload():
    rng = np.random.default_rng(3)
    p32 = rng.standard_normal(10_001).astype(np.float32)
    d_bits = workloads.draw(rng, 1, 10_001, 1e-3).data.reshape(-1)
    p = torch.from_numpy(p32.copy()).to(gu.DEV)
    wpg.lora_dense_patch(p, _bf16_dev(d_bits), wpg.WP_PATCH_ADD, 0.6)
    torch.cuda.synchronize()
    want = odp.apply_diff(p32, "fp32", d_bits, "bf16", 0.6)
    assert np.array_equal(p.cpu().numpy().view(np.uint32), want.view(np.uint32))
    # .set_weight into an fp32 parameter from an fp32 payload
    v = rng.standard_normal(999).astype(np.float32)
    q = torch.empty(999, dtype=torch.float32, device=gu.DEV)
    wpg.lora_dense_patch(q, torch.from_numpy(v).to(gu.DEV), wpg.WP_PATCH_SET, -0.3)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy().view(np.uint32), odp.apply_set(v, "fp32", "fp32", -0.3).view(np.uint32))


def test_shape_mismatch_raises():
    p = torch.zeros(10, dtype=torch.bfloat16, device=gu.DEV)
    d = torch.zeros(11, dtype=torch.bfloat16, device=gu.DEV)
    with pytest.raises(wpg.WeightPatchesError) as e:
        wpg.lora_dense_patch(p, d, wpg.WP_PATCH_ADD, 1.0)
    assert e.value.status == -2
