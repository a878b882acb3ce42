"""The legacy adapter bias vector (older adapters' lora_B.bias; piper-offload docs, "LoRA
merge") on the GPU against the FP64 oracle: every forward path adds s * bias_B to the
adapter's output columns (the vector folded with the layer's bias into one fp32 vector
before the epilogue), and the merge adds the vectors to the module's bias, bit for bit
against the oracle's fp32 add, refusing before any write when the module has no bias."""
import numpy as np
import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from oracle import merge as om
from oracle.lora import decode_patch
from oracle.numerics import bf16_bits_to_f64, relative_rms, to_f64
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _layer(seed, T, d_in, d_out, ranks, G=1, w_kind="bf16", bias="bf16", vecs=("bf16",), rs=0.7,
           kind="bf16", strengths=None):
    """A LoRA linear whose patches carry legacy vectors of the given kinds (None: no vector)."""
    rng = np.random.default_rng(seed)
    X = workloads.draw(rng, T, d_in, 1.0, kind)
    N = G * d_out
    if w_kind == "nf4":
        W = workloads.draw_nf4(rng, N, d_in)
    elif w_kind is None:
        W = None
    else:
        W = workloads.draw(rng, N, d_in, (1.0 / d_in) ** 0.5, w_kind)
    b = workloads.draw(rng, 1, N, 0.01, bias) if bias else None
    strengths = strengths or [0.8] * len(ranks)
    patches = []
    for i, (r, st) in enumerate(zip(ranks, strengths)):
        A = workloads.draw(rng, r, d_in, (1.0 / d_in) ** 0.5, kind)
        B = workloads.draw(rng, d_out, r, 0.05, kind)
        vk = vecs[i % len(vecs)]
        v = workloads.draw(rng, 1, d_out, 0.1, vk) if vk else None
        patches.append(workloads.Patch(A, B, float(r), st, bias_B=v))
    return workloads.Linear(f"legacy{seed}", X, W, b, patches, request_scale=rs, groups=G)


CASES = {
    # tensor-core path, two adapters (bf16 and fp32 vectors), bf16 layer bias
    "tc_two_adapters": dict(seed=1, T=300, d_in=256, d_out=384, ranks=(16, 8), vecs=("bf16", "fp32")),
    # stacked groups: vectors on groups 0 and 2 only, no layer bias of its own
    "grouped3_no_bias": dict(seed=2, T=520, d_in=320, d_out=320, ranks=(32, 32, 32), G=3,
                             bias=None, vecs=("bf16", None, "fp32")),
    # 4-bit base, general path and the small-token path
    "nf4_grouped": dict(seed=3, T=200, d_in=256, d_out=320, ranks=(16, 16), G=2, w_kind="nf4", bias=None),
    "nf4_small_t1": dict(seed=4, T=1, d_in=256, d_out=320, ranks=(16, 16), G=2, w_kind="nf4", bias="fp32"),
    "nf4_small_t5": dict(seed=5, T=5, d_in=512, d_out=256, ranks=(16,), w_kind="nf4"),
    # bf16 weight, small-token path
    "bf16_small_t2": dict(seed=6, T=2, d_in=256, d_out=384, ranks=(8,), vecs=("fp32",)),
    # delta only
    "delta_only": dict(seed=7, T=64, d_in=128, d_out=256, ranks=(8,), w_kind=None, bias=None),
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_adds_the_vectors(name):
    lin = _layer(**CASES[name])
    Y = gu.run_fwd(lin)
    err, chain = gu.errors(lin, Y)
    assert err <= 4e-3 and err <= chain, (err, chain)
    # the vectors matter here (the same call without them is far off)
    plain = workloads.Linear(lin.name, lin.X, lin.W, lin.bias,
                             [workloads.Patch(p.A, p.B, p.alpha, p.strength) for p in lin.patches],
                             lin.request_scale, lin.groups)
    Y0 = gu.run_fwd(plain)
    assert relative_rms(gu.to_f64(Y0), gu.to_f64(Y)) > 2 * err


def test_fp32_path_adds_the_vectors():
    """All-fp32 layer on the exact FP32 path: within 1e-5 of the definition."""
    lin = _layer(seed=8, T=64, d_in=128, d_out=256, ranks=(8,), w_kind="fp32", bias="fp32", vecs=("fp32",),
                 kind="fp32")
    Y = gu.run_fwd(lin, out_dtype=torch.float32)
    err, _ = gu.errors(lin, Y)
    assert err <= 1e-5, err


def test_zero_scale_vector_adds_nothing():
    lin = _layer(seed=9, T=300, d_in=256, d_out=384, ranks=(16, 8), strengths=[0.0, 0.8], vecs=("bf16", None))
    Y = gu.run_fwd(lin)
    plain = workloads.Linear(lin.name, lin.X, lin.W, lin.bias,
                             [workloads.Patch(p.A, p.B, p.alpha, p.strength) for p in lin.patches],
                             lin.request_scale, lin.groups)
    assert torch.equal(Y, gu.run_fwd(plain))


def test_workspace_holds_the_folded_bias():
    lin = _layer(seed=10, T=300, d_in=256, d_out=384, ranks=(16,))
    X, W = gu.dev(lin.X), gu.dev(lin.W)
    ads = gu.adapters(lin)
    with_vec = wpg.lora_workspace_size(wpg.WP_OP_FWD, X, W, ads)
    ads[0].bias_B = None
    without = wpg.lora_workspace_size(wpg.WP_OP_FWD, X, W, ads)
    assert with_vec >= without + 4 * 384


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("w_kind,bias_kind", [("bf16", "bf16"), ("bf16", "fp32"), ("nf4", "bf16")])
def test_merge_updates_the_bias(w_kind, bias_kind):
    lin = _layer(seed=11, T=1, d_in=256, d_out=320, ranks=(8, 16), w_kind=w_kind, bias=bias_kind,
                 vecs=("bf16", "fp32"))
    W = gu.dev(lin.W)
    bias = gu.dev(lin.bias).reshape(-1)
    ads = gu.adapters(lin)
    scale = 0.6
    wpg.lora_merge(W, ads, scale, bias=bias)
    torch.cuda.synchronize()
    want = om.merge_bias_values(to_f64(lin.bias).reshape(-1), [decode_patch(p) for p in lin.patches], scale,
                                bias_kind == "bf16")
    got = bf16_bits_to_f64(_bits(bias)) if bias_kind == "bf16" else bias.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, want)


def test_merge_refuses_a_vector_without_a_bias():
    lin = _layer(seed=12, T=1, d_in=256, d_out=320, ranks=(8,), bias=None)
    W = gu.dev(lin.W)
    before = W.clone()
    with pytest.raises(wpg.WeightPatchesError) as ex:
        wpg.lora_merge(W, gu.adapters(lin), 1.0)
    assert ex.value.status == -1                     # WP_ERR_INVALID
    torch.cuda.synchronize()
    assert torch.equal(W, before)                    # nothing was written
