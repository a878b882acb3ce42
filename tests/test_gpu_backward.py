"""GPU parity of the closed-form backward (dX, dA, dB) against the FP64 oracle.

dX goes through the bf16 tensor-core kernel (relative RMS <= 4e-3); dA and dB are fp32
reductions over tokens of exact bf16 inputs and fp32 intermediates, held to 1e-4."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import lora as olora
from oracle.numerics import relative_rms, to_f64
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

DX_TOL = 4e-3
DAB_TOL = 1e-4


def _run(lin, need_dX=True, dX_dtype=torch.bfloat16):
    X, W, dY = gu.dev(lin.X), gu.dev(lin.W), gu.dev(lin.dY)
    ads = gu.adapters(lin)
    dX, dA, dB = wpg.lora_linear_bwd(X, W, dY, ads, lin.request_scale, need_dX=need_dX, dX_dtype=dX_dtype)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    return dX, dA, dB


def _check_full(lin, dX, dA, dB, dx_tol=DX_TOL):
    X, W, _, patches = olora.decode_linear(lin)
    dY = to_f64(lin.dY)
    g = olora.linear_bwd(X, W, dY, patches, lin.request_scale)
    bX, bA, bB = gu.bwd_bounds(X, W, dY, patches, lin.request_scale, g.dX, g.dA, g.dB,
                               dX_f32=dX is not None and dX.dtype == torch.float32)
    if dX is not None:
        err = relative_rms(gu.to_f64(dX), g.dX)
        assert err <= dx_tol, err
        gu.assert_elementwise(gu.to_f64(dX), g.dX, bX, "dX")
    for i in range(len(patches)):
        ea = relative_rms(dA[i].double().cpu().numpy(), g.dA[i])
        eb = relative_rms(dB[i].double().cpu().numpy(), g.dB[i])
        assert ea <= DAB_TOL and eb <= DAB_TOL, (i, ea, eb)
        gu.assert_elementwise(dA[i].double().cpu().numpy(), g.dA[i], bA[i], f"dA[{i}]")
        gu.assert_elementwise(dB[i].double().cpu().numpy(), g.dB[i], bB[i], f"dB[{i}]")


def _with_dY(lin, seed):
    rng = np.random.default_rng(seed)
    lin.dY = workloads.draw(rng, lin.T, lin.W.rows, 1.0)
    return lin


def test_bwd_bf16_single_group():
    lin = _with_dY(workloads.config2("small")[0], 21)    # 192 -> 520, rank 64, s = 0.35
    lin.bias = None
    dX, dA, dB = _run(lin)
    _check_full(lin, dX, dA, dB)


def test_bwd_bf16_grouped_and_fp32_dX():
    lin = _with_dY(workloads.config1("small"), 22)        # 3 groups of 320, rank 32
    dX, dA, dB = _run(lin, dX_dtype=torch.float32)
    _check_full(lin, dX, dA, dB, dx_tol=2e-3)


@pytest.mark.parametrize("T", [1, 3])
def test_bwd_few_tokens(T):
    """A handful of tokens: the dX pass also returns s dY B for dA, so it must not take the
    few-token forward routes, which do not store it."""
    rng = np.random.default_rng(90 + T)
    K, N, r = 256, 512, 16
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    p = workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5), workloads.draw(rng, N, r, 0.02), float(r), 1.0)
    lin = _with_dY(workloads.Linear("bwd_few_tokens", X, W, None, [p]), 91 + T)
    dX, dA, dB = _run(lin)
    _check_full(lin, dX, dA, dB)


def test_bwd_without_dX():
    lin = _with_dY(workloads.config1("small"), 23)
    dX, dA, dB = _run(lin, need_dX=False)
    assert dX is None
    _check_full(lin, None, dA, dB)


def test_bwd_nf4_small():
    gate_up, down = workloads.config3("small")
    for lin in (gate_up, down):
        dX, dA, dB = _run(lin)
        _check_full(lin, dX, dA, dB)


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_bwd_nf4_full_sampled(which):
    """The 4-bit C3 layers at full size: the dX pass dequantises the stored weight straight into
    MN-major tiles (no transposed copy); dX on sampled rows, dA and dB everywhere."""
    gate_up, down = workloads.config3("full")
    lin = gate_up if which == "gate_up" else down
    dX, dA, dB = _run(lin)
    X, W, _, patches = olora.decode_linear(lin)
    rows = workloads.sample_rows(lin.T, 48)
    from oracle.numerics import bf16_bits_to_f64
    dY_rows = bf16_bits_to_f64(lin.dY.data[rows])
    want_dX = olora.grad_X(X[rows], W, dY_rows, patches, lin.request_scale)
    assert relative_rms(gu.to_f64(dX)[rows], want_dX) <= DX_TOL
    zero = [np.zeros((p.rank, X.shape[1])) for p in patches]
    zeroB = [np.zeros((p.B.shape[0], p.rank)) for p in patches]
    bX, _, _ = gu.bwd_bounds(X[rows], W, dY_rows, patches, lin.request_scale, want_dX, zero, zeroB)
    gu.assert_elementwise(gu.to_f64(dX)[rows], want_dX, bX, "dX (sampled rows)")
    # dA, dB: sums over all tokens, accumulated over row chunks, with the magnitudes the
    # element-wise bound needs (the bound's T is the whole token count)
    sumA = [0.0] * len(patches)
    sumB = [0.0] * len(patches)
    magA = [0.0] * len(patches)
    magB = [0.0] * len(patches)
    G = len(patches)
    og = W.shape[0] // G
    for r0 in range(0, lin.T, 1024):
        sl = slice(r0, min(lin.T, r0 + 1024))
        dYs = bf16_bits_to_f64(lin.dY.data[sl])
        a, b = olora.grad_AB(X[sl], dYs, patches, lin.request_scale)
        sumA = [x + y for x, y in zip(sumA, a)]
        sumB = [x + y for x, y in zip(sumB, b)]
        for i, p in enumerate(patches):
            s = abs(olora.combined_scale(p.alpha, p.rank, p.strength, lin.request_scale))
            dyg = np.abs(dYs[:, i * og:(i + 1) * og])
            magA[i] = magA[i] + s * ((dyg @ np.abs(p.B)).T @ np.abs(X[sl]))
            magB[i] = magB[i] + s * (dyg.T @ (np.abs(X[sl]) @ np.abs(p.A).T))
    T, K = X.shape
    for i in range(len(patches)):
        gA, gB = dA[i].double().cpu().numpy(), dB[i].double().cpu().numpy()
        assert relative_rms(gA, sumA[i]) <= DAB_TOL
        assert relative_rms(gB, sumB[i]) <= DAB_TOL
        eA = (4.0 * (og + T + 32) * 2.0 ** -24 + 2.0 ** -16) * magA[i]
        eB = (4.0 * (K + T + 32) * 2.0 ** -24 + 2.0 ** -16) * magB[i]
        gu.assert_elementwise(gA, sumA[i], gu.ulp_f32(np.abs(sumA[i]) + eA) + eA, f"dA[{i}]")
        gu.assert_elementwise(gB, sumB[i], gu.ulp_f32(np.abs(sumB[i]) + eB) + eB, f"dB[{i}]")


@pytest.mark.parametrize("ranks", [(128, 128, 128), (100,), (128, 16)])
def test_bwd_large_ranks(ranks):
    """Ranks up to 128 per group: the pieces of every group do not fit one 256-column
    contraction, so dA / dB run one contraction per group; the dX pass takes several rank
    passes."""
    rng = np.random.default_rng(sum(ranks))
    G = len(ranks)
    T, K, og = 300, 192, 136
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw(rng, G * og, K, (1.0 / K) ** 0.5)
    patches = [workloads.Patch(workloads.draw(rng, r, K, (1.0 / K) ** 0.5), workloads.draw(rng, og, r, 0.02),
                               float(r), 0.8) for r in ranks]
    lin = _with_dY(workloads.Linear("bwd_large_r", X, W, None, patches, request_scale=1.1, groups=G), 50 + G)
    dX, dA, dB = _run(lin)
    _check_full(lin, dX, dA, dB)


def test_bwd_rank_above_limit_is_refused():
    X = torch.zeros(64, 64, dtype=torch.bfloat16, device=gu.DEV)
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device=gu.DEV)
    A = torch.zeros(136, 64, dtype=torch.bfloat16, device=gu.DEV)
    B = torch.zeros(64, 136, dtype=torch.bfloat16, device=gu.DEV)
    with pytest.raises(wpg.WeightPatchesError) as e:
        wpg.lora_linear_bwd(X, W, torch.zeros(64, 64, dtype=torch.bfloat16, device=gu.DEV),
                            [wpg.Adapter(A, B, 136.0)], 1.0)
    assert e.value.status == -8


@pytest.mark.parametrize("kind,T,K,N,G", [("bf16", 300, 200, 264, 1), ("bf16", 260, 520, 3 * 136, 3),
                                          ("nf4", 300, 320, 384, 1), ("nf4", 520, 512, 2 * 192, 2),
                                          ("nf4", 129, 192, 128, 1)])
def test_bwd_weight_read_as_stored(kind, T, K, N, G):
    """dX = dY W with W [out, in] read as stored (MN-major tiles): ragged in (the dX columns)
    and out (the reduction), bf16 and 4-bit W, block scales by TMA (in % 256 == 0) and from
    global memory."""
    rng = np.random.default_rng(T + K + N)
    X = workloads.draw(rng, T, K, 1.0)
    W = workloads.draw_nf4(rng, N, K) if kind == "nf4" else workloads.draw(rng, N, K, (1.0 / K) ** 0.5)
    og = N // G
    patches = [workloads.Patch(workloads.draw(rng, 16, K, (1.0 / K) ** 0.5), workloads.draw(rng, og, 16, 0.02),
                               16.0, 0.9) for _ in range(G)]
    lin = _with_dY(workloads.Linear("bwd_stored_w", X, W, None, patches, request_scale=1.2, groups=G), T + 1)
    dX, dA, dB = _run(lin)
    _check_full(lin, dX, dA, dB)
