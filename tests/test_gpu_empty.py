"""Empty batches (T = 0 tokens) through every entry point that takes a batch: legal, no
error, nothing written -- except the backward, whose dA and dB are sums over no tokens
(zero), which the oracle's closed form gives as well (X^T and dY^T with no rows)."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import lora as ol
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _layer(K=256, N=384, r=16, groups=1, nf4=False, seed=0):
    rng = np.random.default_rng(seed)
    X = workloads.draw(rng, 0, K, 1.0)
    W = workloads.draw_nf4(rng, N, K) if nf4 else workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    og = N // groups
    ps = [workloads.Patch(workloads.draw(rng, r, K, 0.05), workloads.draw(rng, og, r, 0.05), float(r), 1.0)
          for _ in range(groups)]
    return workloads.Linear("empty", X, W, None, ps, groups=groups)


@pytest.mark.parametrize("nf4,groups", [(False, 1), (False, 3), (True, 1)])
def test_forward_empty(nf4, groups):
    lin = _layer(groups=groups, nf4=nf4)
    W = gu.dev(lin.W)
    ads = gu.adapters(lin)
    X = torch.empty(0, lin.X.cols, dtype=torch.bfloat16, device=gu.DEV)
    if groups > 1:
        Y = wpg.lora_linear_fwd_grouped(X, W, None, ads, 1.0)
    else:
        Y = wpg.lora_linear_fwd(X, W, None, ads, 1.0)
    torch.cuda.synchronize()
    assert tuple(Y.shape) == (0, lin.W.rows)
    assert wpg.lora_device_status() == 0


def test_host_and_exact_forward_empty():
    lin = _layer()
    W = gu.dev(lin.W)
    ads = gu.adapters(lin)
    Xh = torch.empty(0, lin.X.cols, dtype=torch.bfloat16).pin_memory()
    Yh = wpg.lora_linear_fwd_host(Xh, W, None, ads, 1.0)
    assert tuple(Yh.shape) == (0, lin.W.rows)
    X = torch.empty(0, lin.X.cols, dtype=torch.bfloat16, device=gu.DEV)
    Y = wpg.lora_linear_fwd_exact(X, W, None, ads, 1.0)
    torch.cuda.synchronize()
    assert tuple(Y.shape) == (0, lin.W.rows)
    assert wpg.lora_device_status() == 0


@pytest.mark.parametrize("nf4,groups", [(False, 1), (False, 2), (True, 2)])
def test_backward_empty_gives_zero_gradients(nf4, groups):
    lin = _layer(groups=groups, nf4=nf4, N=256)
    W = gu.dev(lin.W)
    ads = gu.adapters(lin)
    X = torch.empty(0, lin.X.cols, dtype=torch.bfloat16, device=gu.DEV)
    dY = torch.empty(0, lin.W.rows, dtype=torch.bfloat16, device=gu.DEV)
    dX, dA, dB = wpg.lora_linear_bwd(X, W, dY, ads, 1.0)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    assert tuple(dX.shape) == (0, lin.X.cols)
    # the oracle's closed form on no tokens
    Xf, _, _, patches = ol.decode_linear(lin)
    wdA, wdB = ol.grad_AB(Xf, np.zeros((0, lin.W.rows)), patches, 1.0)
    for g in range(groups):
        assert torch.count_nonzero(dA[g]).item() == 0 and torch.count_nonzero(dB[g]).item() == 0
        assert np.all(wdA[g] == 0) and np.all(wdB[g] == 0)
        assert tuple(dA[g].shape) == wdA[g].shape and tuple(dB[g].shape) == wdB[g].shape


def test_swiglu_and_dense_patch_empty():
    F = 256
    dH = torch.empty(0, F, dtype=torch.bfloat16, device=gu.DEV)
    EG = torch.empty(0, 2 * F, dtype=torch.bfloat16, device=gu.DEV)
    out = wpg.lora_swiglu_bwd(dH, EG)
    torch.cuda.synchronize()
    p = torch.empty(0, dtype=torch.bfloat16, device=gu.DEV)
    wpg.lora_dense_patch(p, torch.empty(0, dtype=torch.bfloat16, device=gu.DEV), wpg.WP_PATCH_ADD, 1.0)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
