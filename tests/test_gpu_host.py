"""lora_linear_fwd_host: the forward with X and Y in host memory, rows in chunks with the
copies overlapped.  Per row it runs the same kernels on the same operands as the device
entry points, so the results must be bit-identical to them."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _layer(T, K, N, ranks, seed, grouped=False, bias=False):
    rng = np.random.default_rng(seed)
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    og = N // len(ranks) if grouped else N
    patches = [workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5), workloads.draw(rng, og, r, 0.02),
                               float(r), 0.7) for r in ranks]
    b = workloads.draw(rng, 1, N, 0.01) if bias else None
    return workloads.Linear("host", X, W, b, patches, groups=len(ranks) if grouped else 1)


@pytest.mark.parametrize("T", [1, 4096, 9000])       # one partial chunk, one full, three (ragged)
def test_host_matches_device_plain(T):
    lin = _layer(T, 256, 512, [16, 8], seed=T, bias=True)
    X = gu.dev(lin.X); W = gu.dev(lin.W); bias = gu.dev(lin.bias).reshape(-1); ads = gu.adapters(lin)
    want = wpg.lora_linear_fwd(X, W, bias, ads, 0.9)
    Xh = X.cpu().pin_memory()
    got = wpg.lora_linear_fwd_host(Xh, W, bias, ads, 0.9)
    torch.cuda.synchronize()
    assert got.device.type == "cpu" and got.is_pinned()
    assert torch.equal(got, want.cpu())


def test_host_matches_device_grouped_fp32_out():
    lin = _layer(9000, 192, 3 * 128, [16, 32, 8], seed=5, grouped=True)
    X = gu.dev(lin.X); W = gu.dev(lin.W); ads = gu.adapters(lin)
    want = wpg.lora_linear_fwd_grouped(X, W, None, ads, 1.1, out_dtype=torch.float32)
    got = wpg.lora_linear_fwd_host(X.cpu().pin_memory(), W, None, ads, 1.1, out_dtype=torch.float32,
                                   grouped=True)
    torch.cuda.synchronize()
    assert torch.equal(got, want.cpu())


def test_host_pageable_and_repeated_calls():
    """Pageable host memory still gives the right result (serialised copies); back-to-back
    calls reuse the library's streams and events."""
    lin = _layer(5000, 128, 256, [16], seed=3)
    X = gu.dev(lin.X); W = gu.dev(lin.W); ads = gu.adapters(lin)
    want = wpg.lora_linear_fwd(X, W, None, ads, 1.0).cpu()
    Xh = X.cpu()
    outs = [wpg.lora_linear_fwd_host(Xh, W, None, ads, 1.0, out=torch.empty_like(want)) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, want)
    assert wpg.lora_device_status() == 0
