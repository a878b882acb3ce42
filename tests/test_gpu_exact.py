"""The exact tier (sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM",
Modifications): the unfused bf16 chain with unit-scale multiplications skipped, run on the
library's own kernels (lora_linear_fwd_exact).

* Skipping the multiplications by exactly 1.0 leaves every bit of the output unchanged
  (the PR's claim for its exact tier), checked bit for bit with and without skipping.
* The chain matches the oracle's simulated chain (oracle.lora.unfused_bf16_chain): the two
  differ only where an fp32-summed GEMM output and its FP64 value round to different bf16
  neighbours, so nearly every element is bit-equal and the rest are close.
* The fused forward is no worse than this chain against the FP64 definition: the PR's
  accuracy gate (Accuracy Tests), with the library's own chain as the reference."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import lora as olora
from oracle.numerics import relative_rms
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _exact(lin, skip=True):
    X = gu.dev(lin.X)
    W = gu.dev(lin.W)
    bias = gu.dev(lin.bias).reshape(-1) if lin.bias is not None else None
    Y = wpg.lora_linear_fwd_exact(X, W, bias, gu.adapters(lin), lin.request_scale, skip_unit_scales=skip,
                                  grouped=lin.groups > 1)
    torch.cuda.synchronize()
    return Y


def _bits(t):
    return t.cpu().view(torch.int16).numpy()


def _layers():
    up, down, _ = workloads.config2("small")       # alpha/r = 1, strength 0.7, scale 0.5
    gate_up, down3 = workloads.config3("small")    # 4-bit base, unit scales
    lin4, _ = workloads.config4("small")           # one FP32 adapter and two bf16 ones
    rng = np.random.default_rng(61)
    T, K, N = 300, 192, 264
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    pats = [workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5), workloads.draw(rng, N, r, 0.02), a, st)
            for r, a, st in ((24, 36.0, 1.3), (8, 8.0, -0.6))]
    pats[0].bias_B = workloads.draw(rng, 1, N, 0.01)
    mixed = workloads.Linear("mixed_scales", X, W, workloads.draw(rng, 1, N, 0.01), pats, request_scale=0.8)
    return {"c1": workloads.config1("small"), "c2_up": up, "c2_down": down, "c3_gate_up": gate_up,
            "c3_down": down3, "c4": lin4, "mixed": mixed}


LAYERS = ["c1", "c2_up", "c2_down", "c3_gate_up", "c3_down", "c4", "mixed"]


@pytest.fixture(scope="module")
def layers():
    return _layers()


@pytest.mark.parametrize("name", LAYERS)
def test_skipping_unit_scales_changes_no_bit(layers, name):
    lin = layers[name]
    y_skip = _exact(lin, skip=True)
    y_all = _exact(lin, skip=False)
    assert wpg.lora_device_status() == 0
    assert np.array_equal(_bits(y_skip), _bits(y_all))


@pytest.mark.parametrize("name", LAYERS)
def test_chain_matches_the_oracle_chain(layers, name):
    lin = layers[name]
    got = gu.to_f64(_exact(lin))
    want = olora.reference_chain(lin)
    same = float(np.mean(got == want))
    assert same >= 0.98, same
    assert relative_rms(got, want) <= 1e-3


@pytest.mark.parametrize("name", LAYERS)
def test_fused_no_worse_than_the_chain(layers, name):
    lin = layers[name]
    ref = olora.reference_output(lin)
    e_chain = relative_rms(gu.to_f64(_exact(lin)), ref)
    e_fused = relative_rms(gu.to_f64(gu.run_fwd(lin)), ref)
    assert e_fused <= e_chain, (e_fused, e_chain)


def test_chain_close_to_torch_eager_chain():
    lin = workloads.config1("small")
    a = gu.to_f64(_exact(lin))
    b = gu.to_f64(gu.torch_unfused_chain(lin))
    assert relative_rms(a, b) <= 1e-3


def test_full_size_wan_qkv_sampled_rows():
    lin = workloads.config1("full")
    Y = _exact(lin)
    assert wpg.lora_device_status() == 0
    rows = workloads.sample_rows(lin.T, 64)
    got = gu.to_f64(Y)[rows]
    want = olora.reference_chain(lin, rows)
    assert float(np.mean(got == want)) >= 0.98
    assert relative_rms(got, want) <= 1e-3
