"""lora_linear_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace nor allocate one (hosts that own every
device allocation, fixed-budget servers, paths where cudaMalloc's possible device
synchronisation is not acceptable).  This entry point takes its FP32-adapter scratch from
a fixed array inside the library instead.  The test calls it through the C ABI, twice in
a row on different layers (the second call finds the first call's leftovers in the shared
array), and checks each result against lora_linear_fwd with a caller-provided workspace.
It also checks that a call needing more scratch than the array holds is refused before
anything runs.  This file is collected last so that a failure here cannot hide another
test's result in a run that stops at the first failure."""
import ctypes

import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle.numerics import relative_rms
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-5
SCRATCH_BYTES = 4 << 20


def _noalloc(X, W, bias, adapters, request_scale, Y):
    xm, wm, bm, ym = wpg._mat(X), wpg._mat(W), wpg._mat(bias), wpg._out(Y)
    arr = wpg._adapters(adapters)
    st = wpg.lib().lora_linear_fwd_noalloc(
        ctypes.byref(xm), ctypes.byref(wm) if wm is not None else None,
        ctypes.byref(bm) if bm is not None else None, arr, len(adapters), float(request_scale),
        ctypes.byref(ym), torch.cuda.current_stream().cuda_stream)
    return st


def _layer(lin):
    X = gu.dev(lin.X)
    W = gu.dev(lin.W) if lin.W is not None else None
    bias = gu.dev(lin.bias).reshape(-1) if lin.bias is not None else None
    return X, W, bias, gu.adapters(lin)


def _check_against_workspace_entry(X, W, bias, ads, rs):
    want = wpg.lora_linear_fwd(X, W, bias, ads, rs, out_dtype=torch.float32)
    got = torch.full_like(want, float("nan"))
    st = _noalloc(X, W, bias, ads, rs, got)
    assert st == 0, (st, wpg.lib().lora_last_cuda_error())
    torch.cuda.synchronize()
    err = relative_rms(got.double().cpu().numpy(), want.double().cpu().numpy())
    assert err <= FP32_TOL, err


def test_noalloc_matches_workspace_entry_on_two_calls():
    # call 1: the sidecar layer (bf16 base, bf16 patches on the tensor cores, one FP32
    # adapter whose projection goes through the scratch)
    lin4, _ = workloads.config4("small")
    X, W, bias, ads = _layer(lin4)
    assert wpg.lora_workspace_size(wpg.WP_OP_FWD, X, W, ads) > 0
    _check_against_workspace_entry(X, W, bias, ads, lin4.request_scale)
    # call 2: the all-FP32 layer (every adapter's projection goes through the scratch,
    # which still holds call 1's values)
    lin0 = workloads.config0()
    X0, W0, b0, ads0 = _layer(lin0)
    _check_against_workspace_entry(X0, W0, b0, ads0, lin0.request_scale)
    # and the first layer again with another request scale
    _check_against_workspace_entry(X, W, bias, ads, 0.37)
    assert wpg.lora_device_status() == 0


def _few_token_layer(rng, T, K, N, nf4, r=16):
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw_nf4(rng, N, K) if nf4 else workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    bias = workloads.draw(rng, 1, N, 0.01)
    A = workloads.draw(rng, r, K, (1.0 / K) ** 0.5)
    B = workloads.draw(rng, N, r, 0.02)
    return workloads.Linear("few", X, W, bias, [workloads.Patch(A, B, float(r), 0.8)], request_scale=0.5)


def test_noalloc_few_token_routes_after_a_larger_call():
    # a larger call first, so that the shared array holds another layer's leftovers
    lin4, _ = workloads.config4("small")
    X, W, bias, ads = _layer(lin4)
    _check_against_workspace_entry(X, W, bias, ads, lin4.request_scale)
    rng = np.random.default_rng(77)
    # 1 and 4 tokens take the CUDA-core GEMV, 32 tokens (4-bit) the tensor-core small-token
    # kernel; both keep their fp32 partial sums in the array; each call has a bias
    for nf4 in (False, True):
        for T in (1, 4, 32):
            lin = _few_token_layer(rng, T, 512, 1024, nf4)
            _check_against_workspace_entry(*_layer(lin), lin.request_scale)
    assert wpg.lora_device_status() == 0


def test_noalloc_wide_layer_whose_partials_do_not_fit_runs_on_the_general_path():
    # 4-bit 4096 -> 28672 (the stacked gate/up width) at 32 tokens: the small-token route's
    # partial sums would take more than the array holds, so the call runs on the general
    # path (a few KB of scratch) instead of being refused
    rng = np.random.default_rng(78)
    lin = _few_token_layer(rng, 32, 4096, 28672, True)
    X, W, bias, ads = _layer(lin)
    assert wpg.lora_workspace_size(wpg.WP_OP_FWD, X, W, ads) > SCRATCH_BYTES
    _check_against_workspace_entry(X, W, bias, ads, lin.request_scale)
    assert wpg.lora_device_status() == 0


def test_noalloc_refuses_more_scratch_than_the_array_holds():
    T, K, r = 70_000, 64, 16                       # 70000 * 16 * 4 B > 4 MiB
    assert T * r * 4 > SCRATCH_BYTES
    X = torch.zeros(T, K, dtype=torch.float32, device=gu.DEV)
    W = torch.zeros(32, K, dtype=torch.float32, device=gu.DEV)
    A = torch.zeros(r, K, dtype=torch.float32, device=gu.DEV)
    B = torch.zeros(32, r, dtype=torch.float32, device=gu.DEV)
    Y = torch.zeros(T, 32, dtype=torch.float32, device=gu.DEV)
    st = _noalloc(X, W, None, [wpg.Adapter(A, B, float(r))], 1.0, Y)
    assert st == -5                                # WP_ERR_WORKSPACE, nothing launched
    assert float(Y.abs().sum().item()) == 0.0
