"""4-bit NormalFloat base weights on the tensor-core path.

Bit-exactness of the dequantisation (codebook lookup, block index, scale, rounding) is
checked through the GEMM itself: with X = I every output element is one exact product
W_eff[o, t] * 1 summed with zeros, so Y = W_eff^T bit for bit.  The 4-bit SwiGLU
workload (grouped gate/up and down, rank-16 bf16 LoRA) is then checked against the FP64
oracle with the bf16 accuracy gate."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import nf4 as onf4
from oracle.numerics import bf16_bits_to_f32
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

BF16_TOL = 4e-3


def _gate(err, chain):
    assert err <= BF16_TOL, err
    assert err <= chain, (err, chain)


@pytest.mark.parametrize("K,N", [(256, 320), (128, 512), (192, 264)])
def test_dequant_bit_exact_through_identity(K, N):
    rng = np.random.default_rng(K + N)
    W = workloads.draw_nf4(rng, N, K)
    X = torch.eye(K, dtype=torch.bfloat16, device=gu.DEV)          # T = K tokens
    Y = wpg.lora_linear_fwd(X, gu.dev(W), None, [])
    torch.cuda.synchronize()
    got = Y.cpu().view(torch.int16).numpy().view(np.uint16)          # [K, N] = W_eff^T
    want = onf4.dequant_bf16_bits(W.data, W.absmax, N, K).T
    # signed zeros may differ through the accumulation (0 * w carries w's sign); every
    # nonzero value must match bit for bit
    gv, wv = bf16_bits_to_f32(got), bf16_bits_to_f32(want)
    assert np.array_equal(gv, wv)
    nz = wv != 0
    assert np.array_equal(got[nz], want[nz])


def test_dequant_grouped_identity():
    rng = np.random.default_rng(9)
    W = workloads.draw_nf4(rng, 2 * 256, 128)
    X = torch.eye(128, dtype=torch.bfloat16, device=gu.DEV)
    zA = torch.zeros(16, 128, dtype=torch.bfloat16, device=gu.DEV)
    zB = torch.zeros(256, 16, dtype=torch.bfloat16, device=gu.DEV)
    ads = [wpg.Adapter(zA, zB, 16.0), wpg.Adapter(zA, zB, 16.0)]      # A = 0: base only
    Y = wpg.lora_linear_fwd_grouped(X, gu.dev(W), None, ads, 1.0)
    torch.cuda.synchronize()
    got = bf16_bits_to_f32(Y.cpu().view(torch.int16).numpy().view(np.uint16))
    want = bf16_bits_to_f32(onf4.dequant_bf16_bits(W.data, W.absmax, 2 * 256, 128).T)
    assert np.array_equal(got, want)


def test_c3_small_gate_up_and_down():
    gate_up, down = workloads.config3("small")
    for lin in (gate_up, down):
        Y = gu.run_fwd(lin)
        _gate(*gu.errors(lin, Y))
    assert wpg.lora_device_status() == 0


def test_c3_full_sampled_rows():
    gate_up, down = workloads.config3("full")
    for lin in (gate_up, down):
        Y = gu.run_fwd(lin)
        rows = workloads.sample_rows(lin.T, 64)
        _gate(*gu.errors(lin, Y, rows))
