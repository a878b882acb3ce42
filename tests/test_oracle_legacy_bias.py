"""Pins of the legacy adapter bias vector in the oracle (piper-offload docs, "LoRA merge":
older PEFT/Wan adapters carry a vector beside A and B, their lora_B.bias; routed mode adds
it to the output, merge mode to the module's bias, with the adapter's own strength).

What pins it, without the oracle's own formula:
  * PEFT builds the second factor as a torch Linear with that bias, so the patch's term is
    scaling * lora_B(lora_A(x)): computed here with torch's own Linear layers in float64;
  * a vector is the same thing as one more rank-1 patch on a column of ones appended to X
    (whose low-rank term the brute-force pins of the forward already fix);
  * the merge of one adapter's vector is the dense bias patch's add with k = fl32(s)
    (FastVideo DenseLoRAPatch.apply_to, pinned bit for bit in its own tests);
  * the merged weight and bias reproduce the unmerged forward (the forward is linear).
"""
import numpy as np
import pytest
import torch

from oracle import dense_patch as odp
from oracle import merge as om
from oracle.lora import DecodedPatch, combined_scale, linear_fwd, linear_fwd_grouped, unfused_bf16_chain
from oracle.numerics import f32_to_bf16_bits, f64_to_bf16_value


def _patch(rng, r, d_in, d_out, alpha=8.0, strength=0.7, vec=True):
    A = f64_to_bf16_value(rng.normal(0, (1.0 / d_in) ** 0.5, (r, d_in)))
    B = f64_to_bf16_value(rng.normal(0, 0.05, (d_out, r)))
    v = f64_to_bf16_value(rng.normal(0, 0.02, d_out)) if vec else None
    return DecodedPatch(A, B, alpha, strength, bias_B=v)


def test_matches_peft_linear_with_bias():
    """scaling * lora_B(lora_A(x)) with lora_B = Linear(r, out, bias=True), in float64."""
    rng = np.random.default_rng(1)
    T, d_in, d_out, r = 7, 24, 20, 4
    X = rng.normal(0, 1, (T, d_in))
    W = rng.normal(0, 0.2, (d_out, d_in))
    bias = rng.normal(0, 0.1, d_out)
    p = _patch(rng, r, d_in, d_out, alpha=6.0, strength=-0.4)
    rs = 0.8
    lora_A = torch.nn.Linear(d_in, r, bias=False).double()
    lora_B = torch.nn.Linear(r, d_out, bias=True).double()
    base = torch.nn.Linear(d_in, d_out, bias=True).double()
    with torch.no_grad():
        lora_A.weight.copy_(torch.from_numpy(p.A))
        lora_B.weight.copy_(torch.from_numpy(p.B))
        lora_B.bias.copy_(torch.from_numpy(p.bias_B))
        base.weight.copy_(torch.from_numpy(W))
        base.bias.copy_(torch.from_numpy(bias))
        x = torch.from_numpy(X)
        want = (base(x) + lora_B(lora_A(x)) * (p.alpha / r * p.strength * rs)).numpy()
    got = linear_fwd(X, W, bias, [p], rs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def _ones_column_form(X, W, patches, rs):
    """The same layer with a column of ones appended to X and each legacy vector moved into
    an extra rank-1 patch that reads only that column."""
    T, d_in = X.shape
    X1 = np.hstack([X, np.ones((T, 1))])
    W1 = None if W is None else np.hstack([W, np.zeros((W.shape[0], 1))])
    out = []
    for p in patches:
        out.append(DecodedPatch(np.hstack([p.A, np.zeros((p.rank, 1))]), p.B, p.alpha, p.strength))
        if p.bias_B is not None:
            e = np.zeros((1, d_in + 1))
            e[0, -1] = 1.0
            # s' = alpha' / 1 * strength' * rs must equal the patch's own s
            out.append(DecodedPatch(e, np.asarray(p.bias_B).reshape(-1, 1), p.alpha / p.rank, p.strength))
    return X1, W1, out


def test_equals_a_rank_one_patch_on_a_ones_column():
    rng = np.random.default_rng(2)
    T, d_in, d_out = 9, 16, 12
    X = rng.normal(0, 1, (T, d_in))
    W = rng.normal(0, 0.3, (d_out, d_in))
    patches = [_patch(rng, 3, d_in, d_out, 3.0, 1.0), _patch(rng, 2, d_in, d_out, 8.0, 0.25, vec=False),
               _patch(rng, 5, d_in, d_out, 10.0, -0.6)]
    for rs in (1.0, 0.35):
        X1, W1, p1 = _ones_column_form(X, W, patches, rs)
        np.testing.assert_allclose(linear_fwd(X, W, None, patches, rs), linear_fwd(X1, W1, None, p1, rs),
                                   rtol=1e-12, atol=1e-12)
        # delta only (no W)
        np.testing.assert_allclose(linear_fwd(X, None, None, patches, rs, out_features=d_out),
                                   linear_fwd(X1, None, None, p1, rs, out_features=d_out), rtol=1e-12, atol=1e-12)


def test_grouped_vector_stays_in_its_group():
    rng = np.random.default_rng(3)
    T, d_in, og, G = 5, 16, 8, 3
    X = rng.normal(0, 1, (T, d_in))
    W = rng.normal(0, 0.3, (G * og, d_in))
    gp = [_patch(rng, 2, d_in, og, 2.0, 1.0, vec=(g != 1)) for g in range(G)]
    Y = linear_fwd_grouped(X, W, None, gp, 1.0)
    plain = [DecodedPatch(p.A, p.B, p.alpha, p.strength) for p in gp]
    Y0 = linear_fwd_grouped(X, W, None, plain, 1.0)
    for g, p in enumerate(gp):
        sl = slice(g * og, (g + 1) * og)
        want = 0.0 if p.bias_B is None else combined_scale(p.alpha, p.rank, p.strength, 1.0) * p.bias_B
        np.testing.assert_allclose(Y[:, sl] - Y0[:, sl], np.broadcast_to(want, (T, og)), rtol=1e-12, atol=1e-13)


def test_zero_strength_and_linearity():
    rng = np.random.default_rng(4)
    X = rng.normal(0, 1, (6, 16))
    W = rng.normal(0, 0.3, (10, 16))
    p = _patch(rng, 4, 16, 10)
    base = X @ W.T
    z = DecodedPatch(p.A, p.B, p.alpha, 0.0, bias_B=p.bias_B)
    np.testing.assert_array_equal(linear_fwd(X, W, None, [z], 1.0), base)
    d1 = linear_fwd(X, W, None, [p], 0.5) - base
    d2 = linear_fwd(X, W, None, [p], 1.0) - base
    np.testing.assert_allclose(d2, 2.0 * d1, rtol=1e-12, atol=1e-13)


def test_chain_keeps_the_vector_with_the_second_factor():
    """The unfused chain's d = bf16(t B^T + vec): on an all-FP32 layer (no rounding) it equals
    the definition, and on a bf16 layer it stays within the bf16 chain's usual error."""
    rng = np.random.default_rng(5)
    X = f64_to_bf16_value(rng.normal(0, 1, (32, 64)))
    W = f64_to_bf16_value(rng.normal(0, 0.125, (48, 64)))
    p = _patch(rng, 8, 64, 48, 8.0, 0.75)        # scales exact in fp32, as the chain keeps them
    exact = linear_fwd(X, W, None, [p], 1.0)
    np.testing.assert_allclose(unfused_bf16_chain(X, W, None, [p], 1.0, bf16_tensors=False), exact,
                               rtol=1e-12, atol=1e-12)
    chain = unfused_bf16_chain(X, W, None, [p], 1.0)
    assert np.sqrt(np.sum((chain - exact) ** 2) / np.sum(exact ** 2)) < 8e-3


@pytest.mark.parametrize("bf16", [True, False])
def test_merge_of_one_vector_is_the_dense_bias_add(bf16):
    rng = np.random.default_rng(6)
    d_out = 300
    b = rng.normal(0, 0.1, d_out)
    bias = f64_to_bf16_value(b) if bf16 else b.astype(np.float32).astype(np.float64)
    p = _patch(rng, 4, 16, d_out, alpha=5.0, strength=0.3)
    scale = 0.9
    got = om.merge_bias_values(bias, [p], scale, bf16)
    k = float(np.float32(combined_scale(p.alpha, p.rank, p.strength, scale)))
    if bf16:
        want_bits = odp.apply_diff(f32_to_bf16_bits(bias.astype(np.float32)), "bf16",
                                   f32_to_bf16_bits(p.bias_B.astype(np.float32)), "bf16", k)
        np.testing.assert_array_equal(f32_to_bf16_bits(got.astype(np.float32)), want_bits)
    else:
        want = odp.apply_diff(bias.astype(np.float32), "fp32", p.bias_B.astype(np.float32), "fp32", k)
        np.testing.assert_array_equal(got.astype(np.float32), want)


def test_merged_weight_and_bias_reproduce_the_forward():
    rng = np.random.default_rng(7)
    T, d_in, d_out = 16, 64, 40
    X = f64_to_bf16_value(rng.normal(0, 1, (T, d_in)))
    W = f64_to_bf16_value(rng.normal(0, 0.125, (d_out, d_in)))
    bias = f64_to_bf16_value(rng.normal(0, 0.1, d_out))
    patches = [_patch(rng, 4, d_in, d_out, 4.0, 0.8), _patch(rng, 8, d_in, d_out, 16.0, -0.3)]
    Wm = om.merge_bf16_values(W, patches, 1.0)
    bm = om.merge_bias_values(bias, patches, 1.0, True)
    got = X @ Wm.T + bm.reshape(1, -1)
    want = linear_fwd(X, W, bias, patches, 1.0)
    assert np.sqrt(np.sum((got - want) ** 2) / np.sum(want ** 2)) < 4e-3
    # zero strength leaves the bias bit for bit
    z = [DecodedPatch(p.A, p.B, p.alpha, 0.0, bias_B=p.bias_B) for p in patches]
    np.testing.assert_array_equal(om.merge_bias_values(bias, z, 1.0, True), bias)
