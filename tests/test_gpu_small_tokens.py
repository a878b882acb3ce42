"""The small-token path (the weight streamed once over every SM, swapped MMAs, K split,
one reduction pass; 4-bit weights up to 64 tokens, bf16 weights up to 4) against the FP64
oracle with the bf16 accuracy gate.  Token counts just past the bf16 limit check the
hand-over to the general path.

InvokeAI sidecar-patch article, section 五: quantised layers under few tokens go through a
small-batch kernel; here both bf16 and 4-bit weights do, with the LoRA terms fused in.
Covered: one token, ragged token counts, ragged weight rows, 4-bit weights with and
without TMA-fed block scales, one to four tokens on the CUDA-core kernel (4-bit and bf16,
many K splits, and its fallback when the block scales are not 16-byte aligned), stacked column groups, delta-only layers, several adapters,
bias, fp32 output, zero strength, and full-size layers of the workloads (sampled output
columns)."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import lora as olora
from oracle.numerics import relative_rms, to_f64
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

BF16_TOL = 4e-3


def _layer(T, K, N, ranks, kind="bf16", bias=None, groups=1, strengths=None, seed=0, with_w=True):
    rng = np.random.default_rng(seed)
    X = workloads.draw(rng, T, K, 1.0)
    W = None
    if with_w:
        W = workloads.draw_nf4(rng, N, K) if kind == "nf4" else workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    b = None
    if bias is not None:
        b = workloads.draw(rng, 1, N, 0.01, kind=bias)
    og = N // groups
    strengths = strengths or [1.0] * len(ranks)
    patches = [workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5),
                               workloads.draw(rng, og if groups > 1 else N, r, 0.02), float(r), st)
               for r, st in zip(ranks, strengths)]
    return workloads.Linear(f"small_{kind}", X, W, b, patches, groups=groups)


def _check(lin, out_dtype=torch.bfloat16):
    Y = gu.run_fwd(lin, out_dtype=out_dtype)
    assert wpg.lora_device_status() == 0
    err, chain = gu.errors(lin, Y)
    assert err <= BF16_TOL, err
    assert err <= chain, (err, chain)
    return Y


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 16])
@pytest.mark.parametrize("K", [256, 320])
def test_bf16_weight(T, K):
    """K = 256: one to four tokens on the CUDA-core kernel; K = 320 (not a multiple of 256):
    the tensor-core small-token path; five and more tokens: the general path."""
    _check(_layer(T, K, 320, [16], bias="bf16", seed=T + K))


@pytest.mark.parametrize("T,K,N", [(1, 512, 384), (33, 512, 384), (20, 320, 200), (64, 256, 264)])
def test_nf4_weight(T, K, N):
    # K = 512: block scales by TMA; K = 320: block scales loaded by the dequantisation warps
    _check(_layer(T, K, N, [16], kind="nf4", seed=T + K))


@pytest.mark.parametrize("kind", ["nf4", "bf16"])
@pytest.mark.parametrize("T,K,N,ranks", [(1, 1024, 200, [8]), (2, 768, 264, [24, 16]), (3, 2048, 96, [16]),
                                          (4, 512, 384, [40]), (1, 14336, 264, [16]), (4, 14336, 130, [8, 8])])
def test_cuda_core_tokens(T, K, N, ranks, kind):
    """One to four tokens with K a multiple of 256 go to the CUDA-core kernel, 4-bit or bf16
    weight: ragged weight rows (the last 32-row group part-filled), ranks that are not
    multiples of 16, several adapters, a bias, and long rows split into many K ranges (more
    than eight splits for K = 14336)."""
    _check(_layer(T, K, N, ranks, kind=kind, bias="bf16", seed=T * 7 + K + N))


@pytest.mark.parametrize("K,N,ranks,groups", [(2048, 130, [8, 8], 1), (6144, 1000, [16], 1), (4096, 2 * 200, [16, 8], 2)])
def test_plain_load_kernel_one_token(K, N, ranks, groups):
    """One token against a 4-bit weight whose K is a multiple of 2048 takes the plain-load
    kernel (a 2048-element split per slice, a row's slice per warp, X in registers): one, three
    and two splits, ragged rows (130, 1000), several adapters, a bias, stacked groups with fp32
    output and a request scale."""
    lin = _layer(1, K, N, ranks, kind="nf4", bias="bf16" if groups == 1 else None, groups=groups,
                 strengths=[0.5, 1.5][:len(ranks)], seed=K + N)
    if groups > 1:
        lin.request_scale = 0.75
    _check(lin, out_dtype=torch.float32 if groups > 1 else torch.bfloat16)


@pytest.mark.parametrize("kind", ["nf4", "bf16"])
def test_cuda_core_grouped_fp32_out(kind):
    """Stacked gate/up groups with their own adapters, fp32 output, a request scale, one token
    through four."""
    for T in (1, 4):
        lin = _layer(T, 512, 2 * 200, [16, 8], kind=kind, groups=2, strengths=[0.5, 1.5], seed=40 + T)
        lin.request_scale = 0.75
        _check(lin, out_dtype=torch.float32)


@pytest.mark.parametrize("T", [1, 3])
def test_nf4_unaligned_scales_few_tokens(T):
    """Block scales that do not start on a 16-byte boundary cannot be copied by TMA: one to four
    tokens then fall back to the tensor-core small-token path, which reads the scales from
    global memory, within the same gates."""
    lin = _layer(T, 512, 200, [16], kind="nf4", seed=70 + T)
    W = gu.dev(lin.W)
    buf = torch.zeros(W.absmax.numel() + 1, dtype=torch.float32, device=W.absmax.device)
    buf[1:] = W.absmax
    W_off = wpg.NF4Weight(W.packed, buf[1:], W.rows, W.cols)
    assert W_off.absmax.data_ptr() % 16 != 0
    Y = wpg.lora_linear_fwd(gu.dev(lin.X), W_off, None, gu.adapters(lin), lin.request_scale)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    err, chain = gu.errors(lin, Y)
    assert err <= BF16_TOL and err <= chain, (err, chain)


def test_grouped_qkv():
    _check(_layer(3, 320, 3 * 320, [32, 32, 32], groups=3, seed=3))


def test_grouped_nf4():
    _check(_layer(40, 256, 2 * 320, [16, 16], kind="nf4", groups=2, seed=8))


def test_delta_only():
    _check(_layer(2, 256, 264, [8], with_w=False, seed=5))


def test_several_adapters_fp32_out():
    lin = _layer(4, 384, 384, [8, 40, 128], bias="fp32", strengths=[1.0, 0.6, -0.3], seed=6)
    _check(lin, out_dtype=torch.float32)


def test_zero_strength_equals_base():
    lin = _layer(3, 256, 320, [16], strengths=[0.0], seed=7)
    X, W = gu.dev(lin.X), gu.dev(lin.W)
    y0 = wpg.lora_linear_fwd(X, W, None, gu.adapters(lin))
    y1 = wpg.lora_linear_fwd(X, W, None, [])
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("cfg,T", [("c1", 4), ("c3", 1), ("c3", 4), ("c3", 64), ("c3down", 1), ("c3down", 3)])
def test_full_size_layers(cfg, T):
    """Full-size weights of the workloads with few tokens; the oracle checks 256 sampled
    output columns (weight rows decoded one block at a time)."""
    lin = {"c1": lambda: workloads.config1("full"), "c3": lambda: workloads.config3("full")[0],
           "c3down": lambda: workloads.config3("full")[1]}[cfg]()
    X = lin.X.slice_rows(0, T)
    small = workloads.Linear(lin.name, X, lin.W, lin.bias, lin.patches, lin.request_scale, lin.groups)
    Y = gu.run_fwd(small)
    assert wpg.lora_device_status() == 0
    got = gu.to_f64(Y)
    N = lin.W.rows
    og = N // lin.groups
    rng = np.random.default_rng(99)
    cols = np.sort(rng.choice(N, 256, replace=False))
    Xf = to_f64(X)
    bias = to_f64(lin.bias).reshape(-1) if lin.bias is not None else None
    want = np.empty((T, len(cols)))
    Wc = np.empty((len(cols), Xf.shape[1]))
    for k, c in enumerate(cols):
        w = to_f64(lin.W.slice_rows(int(c), int(c) + 1))[0]
        Wc[k] = w
        y = Xf @ w + (bias[c] if bias is not None else 0.0)
        g = c // og if lin.groups > 1 else 0
        p = olora.decode_patch(lin.patches[g])
        s = olora.combined_scale(p.alpha, p.rank, p.strength, lin.request_scale)
        y = y + s * ((Xf @ p.A.T) @ p.B[c - g * og])
        want[:, k] = y
    assert relative_rms(got[:, cols], want) <= BF16_TOL
    # element-wise on the sampled columns: the bound's weight magnitudes from the decoded rows
    Wfull = np.zeros((N, Xf.shape[1]))
    Wfull[cols] = Wc
    pats = [olora.decode_patch(p) for p in lin.patches]
    bound = gu.linear_error_bound(Xf, Wfull, bias, pats, lin.request_scale, lin.groups, False, want, cols=cols)
    gu.assert_elementwise(got[:, cols], want, bound, lin.name)
