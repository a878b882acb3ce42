"""SwiGLU around the LoRA MLP on the GPU (Unsloth fast_lora walkthrough, section 4,
LoRA_MLP): the fused front half (gate and up LoRA linears plus the activation in one
pass), the elementwise backward step, and the whole MLP's forward and backward through
the C ABI, each against the FP64 oracle.

Bit-level checks: the saved e | g equal the grouped linear's output (the SwiGLU tile adds
exact zeros for the other half's adapter), and the h the backward recomputes from them
equals the h the forward wrote (one definition of the activation on both sides).

Tolerances: h, de, dg, dH are bf16 outputs of one rounding after bf16 inputs: the bf16
gate (relative RMS <= 4e-3, and no worse than the unfused chain for h).  The whole MLP
chain rounds to bf16 up to six times in sequence (e | g, h, y, dH, de | dg, dX), each
adding about 1.1e-3 relative RMS, so its outputs are held to 1e-2."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import lora as olora
from oracle import swiglu as osw
from oracle.numerics import bf16_bits_to_f64, f64_to_bf16_value, relative_rms, to_f64
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

BF16_TOL = 4e-3
CHAIN_TOL = 1e-2


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _gate_up(kind, T, d, F, r, bias=False, seed=0):
    rng = np.random.default_rng(seed)
    X = workloads.draw(rng, T, d, 1.0)
    W = workloads.draw_nf4(rng, 2 * F, d) if kind == "nf4" else workloads.draw(rng, 2 * F, d, (1.0 / d) ** 0.5)
    b = workloads.draw(rng, 1, 2 * F, 0.01) if bias else None
    patches = [workloads.Patch(workloads.draw(rng, r, d, (1.0 / d) ** 0.5), workloads.draw(rng, F, r, 0.02),
                               float(r), 1.0) for _ in range(2)]
    return workloads.Linear(f"swiglu_{kind}", X, W, b, patches, groups=2)


@pytest.mark.parametrize("kind,T,d,F,r,bias", [
    ("bf16", 300, 256, 320, 16, False),
    ("bf16", 520, 192, 200, 32, True),      # ragged F (200 = 3 x 64 + 8), bias
    ("nf4", 300, 256, 320, 16, False),
    ("nf4", 700, 128, 136, 16, True),       # two 512-row tiles, ragged rows and columns
])
def test_swiglu_fwd(kind, T, d, F, r, bias):
    lin = _gate_up(kind, T, d, F, r, bias, seed=T + F)
    X, W = gu.dev(lin.X), gu.dev(lin.W)
    b = gu.dev(lin.bias).reshape(-1) if lin.bias is not None else None
    ads = gu.adapters(lin)
    h, eg = wpg.lora_swiglu_fwd(X, W, b, ads, lin.request_scale, save_eg=True)
    y = wpg.lora_linear_fwd_grouped(X, W, b, ads, lin.request_scale)
    _, h2 = wpg.lora_swiglu_bwd(torch.zeros_like(h), eg, want_h=True)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    assert np.array_equal(_bits(eg), _bits(y))
    assert np.array_equal(_bits(h), _bits(h2))
    ref = olora.reference_output(lin)                     # exact e | g
    h_ref = osw.swiglu(ref[:, :F], ref[:, F:])
    # element-wise: e | g within the linear's bound, h within the bound carried through silu
    b_eg = gu.fwd_bound(lin, y_ref=ref)
    gu.assert_elementwise(gu.to_f64(eg), ref, b_eg, "e|g")
    gu.assert_elementwise(gu.to_f64(h), h_ref, gu.swiglu_bound(ref[:, :F], ref[:, F:], b_eg[:, :F], b_eg[:, F:]), "h")
    chain = olora.reference_chain(lin)                    # unfused bf16 chain's e | g
    h_chain = f64_to_bf16_value(osw.swiglu(chain[:, :F], chain[:, F:]))
    err, err_chain = relative_rms(gu.to_f64(h), h_ref), relative_rms(h_chain, h_ref)
    assert err <= BF16_TOL, err
    assert err <= err_chain, (err, err_chain)


def test_swiglu_fwd_zero_strength_is_base_only():
    lin = _gate_up("bf16", 260, 128, 136, 16, seed=4)
    X, W = gu.dev(lin.X), gu.dev(lin.W)
    ads = [wpg.Adapter(a.A, a.B, a.alpha, 0.0) for a in gu.adapters(lin)]
    h, eg = wpg.lora_swiglu_fwd(X, W, None, ads, 1.0, save_eg=True)
    y0 = wpg.lora_linear_fwd(X, W, None, [])             # the plain base output
    _, h0 = wpg.lora_swiglu_bwd(torch.zeros_like(h), y0, want_h=True)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(eg), _bits(y0))
    assert np.array_equal(_bits(h), _bits(h0))


def test_swiglu_bwd_step():
    rng = np.random.default_rng(5)
    T, F = 257, 136
    dH = workloads.draw(rng, T, F, 1.0)
    EG = workloads.draw(rng, T, 2 * F, 3.0)
    # special values of e: zero, saturated sigmoid, exp overflow in float32
    bits = EG.data.copy()
    special = np.array([0.0, 30.0, -30.0, 100.0, -100.0, -90.0], dtype=np.float32)
    sb = (special.view(np.uint32) >> 16).astype(np.uint16)
    bits[:len(sb), 0] = sb
    EG = workloads.Mat("bf16", bits, T, 2 * F)
    deg, h = wpg.lora_swiglu_bwd(gu.dev(dH), gu.dev(EG), want_h=True)
    torch.cuda.synchronize()
    dh64, eg64 = bf16_bits_to_f64(dH.data), bf16_bits_to_f64(EG.data)
    h_ref, dg_ref, de_ref = osw.swiglu_bwd(dh64, eg64[:, :F], eg64[:, F:])
    got = gu.to_f64(deg)
    for g_, w_ in ((got[:, :F], de_ref), (got[:, F:], dg_ref), (gu.to_f64(h), h_ref)):
        assert relative_rms(g_, w_) <= BF16_TOL
        # elementwise: one bf16 rounding (half an ulp, 2^-9 relative) plus float32 noise
        big = np.abs(w_) > 1e-30
        assert np.all(np.abs(g_[big] - w_[big]) <= 2.0 ** -8 * np.abs(w_[big]))
        assert np.all(np.abs(g_[~big]) <= 1e-30)


@pytest.mark.parametrize("kind", ["bf16", "nf4"])
def test_swiglu_mlp_chain(kind):
    """The whole LoRA MLP, forward and backward, through the C ABI."""
    T, d, F, r = 300, 256, 320, 16
    gate_up = _gate_up(kind, T, d, F, r, seed=11)
    rng = np.random.default_rng(12)
    Wd = workloads.draw_nf4(rng, d, F) if kind == "nf4" else workloads.draw(rng, d, F, (1.0 / F) ** 0.5)
    pd = workloads.Patch(workloads.draw(rng, r, F, (1.0 / F) ** 0.5), workloads.draw(rng, d, r, 0.02), float(r), 0.7)
    dY = workloads.draw(rng, T, d, 1.0)
    X, Wgu, Wdd = gu.dev(gate_up.X), gu.dev(gate_up.W), gu.dev(Wd)
    ads = gu.adapters(gate_up)
    ad_d = [wpg.Adapter(gu.dev(pd.A), gu.dev(pd.B), pd.alpha, pd.strength)]
    rs = 0.9
    h, eg = wpg.lora_swiglu_fwd(X, Wgu, None, ads, rs, save_eg=True)
    y = wpg.lora_linear_fwd(h, Wdd, None, ad_d, rs)
    dH, dA_d, dB_d = wpg.lora_linear_bwd(h, Wdd, gu.dev(dY), ad_d, rs)
    deg, h2 = wpg.lora_swiglu_bwd(dH, eg, want_h=True)
    dX, dA_gu, dB_gu = wpg.lora_linear_bwd(X, Wgu, deg, ads, rs)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    assert np.array_equal(_bits(h), _bits(h2))

    Xf, Wguf, _, pgu = olora.decode_linear(gate_up)
    Wdf = to_f64(Wd)
    pdf = olora.decode_patch(pd)
    _, _, _, y_ref = osw.lora_mlp_fwd(Xf, Wguf, None, pgu, Wdf, None, [pdf], rs)
    gr = osw.lora_mlp_bwd(Xf, Wguf, None, pgu, Wdf, None, [pdf], rs, bf16_bits_to_f64(dY.data))
    checks = [("y", gu.to_f64(y), y_ref), ("dH", gu.to_f64(dH), gr["dH"]), ("dX", gu.to_f64(dX), gr["dX"]),
              ("dA_down", dA_d[0].cpu().double().numpy(), gr["down"][0][0]),
              ("dB_down", dB_d[0].cpu().double().numpy(), gr["down"][0][1])]
    for k in range(2):
        checks.append((f"dA_{k}", dA_gu[k].cpu().double().numpy(), gr["gate_up"][k][0]))
        checks.append((f"dB_{k}", dB_gu[k].cpu().double().numpy(), gr["gate_up"][k][1]))
    for name, got, want in checks:
        err = relative_rms(got, want)
        assert err <= CHAIN_TOL, (name, err)


def test_swiglu_c3_full_sampled_rows():
    """The 4-bit SwiGLU workload at full size (T = 8192, 4096 -> 2 x 14336): e | g equal the
    grouped linear bit for bit everywhere, h matches the oracle on sampled rows."""
    gate_up, _ = workloads.config3("full")
    X, W = gu.dev(gate_up.X), gu.dev(gate_up.W)
    ads = gu.adapters(gate_up)
    h, eg = wpg.lora_swiglu_fwd(X, W, None, ads, 1.0, save_eg=True)
    y = wpg.lora_linear_fwd_grouped(X, W, None, ads, 1.0)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    assert torch.equal(eg.view(torch.int16), y.view(torch.int16))
    del y
    F = gate_up.W.rows // 2
    rows = workloads.sample_rows(gate_up.T, 6)
    ref = olora.reference_output(gate_up, rows)
    h_ref = osw.swiglu(ref[:, :F], ref[:, F:])
    got = gu.to_f64(h[torch.as_tensor(rows, device=h.device)])
    assert relative_rms(got, h_ref) <= BF16_TOL
    b_eg = gu.fwd_bound(gate_up, rows, y_ref=ref)
    gu.assert_elementwise(gu.to_f64(eg[torch.as_tensor(rows, device=eg.device)]), ref, b_eg, "e|g")
    gu.assert_elementwise(got, h_ref, gu.swiglu_bound(ref[:, :F], ref[:, F:], b_eg[:, :F], b_eg[:, F:]), "h")
