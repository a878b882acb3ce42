"""Pins for the oracle's LoRA linear: hand-worked examples, brute-force loops, the
merged-weight identity, invariants from the method's definition, and finite
differences for the closed-form backward."""
import itertools
import json
import os

import numpy as np
import pytest

import workloads
from oracle import lora
from oracle.numerics import relative_rms, f64_to_bf16_value


def _patch(A, B, alpha, strength, fp32=False):
    return lora.DecodedPatch(np.asarray(A, float), np.asarray(B, float), alpha, strength, fp32)


def _examples(golden_dir):
    with open(os.path.join(golden_dir, "lora_hand_examples.json")) as f:
        return json.load(f)


def test_hand_examples_forward(golden_dir):
    for ex in _examples(golden_dir)["examples"]:
        p = _patch(ex["A"], ex["B"], ex["alpha"], ex["strength"])
        assert lora.combined_scale(p.alpha, p.rank, p.strength, ex["request_scale"]) == ex["s"]
        bias = None if ex["bias"] is None else np.array(ex["bias"], float)
        Y = lora.linear_fwd(np.array(ex["X"], float), np.array(ex["W"], float), bias, [p],
                            ex["request_scale"])
        assert Y.tolist() == ex["Y"], ex["name"]


def test_hand_example_backward(golden_dir):
    ex = _examples(golden_dir)["examples"][1]
    p = _patch(ex["A"], ex["B"], ex["alpha"], ex["strength"])
    g = lora.linear_bwd(np.array(ex["X"], float), np.array(ex["W"], float),
                        np.array(ex["dY"], float), [p], ex["request_scale"])
    assert g.dX.tolist() == ex["dX"]
    assert g.dA[0].tolist() == ex["dA"]
    assert g.dB[0].tolist() == ex["dB"]


def test_combined_scales_of_the_workloads(golden_dir):
    cs = _examples(golden_dir)["combined_scales"]
    lin0 = workloads.config0("small")
    p = lin0.patches[0]
    assert abs(lora.combined_scale(p.alpha, p.rank, p.strength, lin0.request_scale) - cs["tiny_fp32"]) < 1e-15
    up, _, _ = workloads.config2("small")
    p = up.patches[0]
    assert abs(lora.combined_scale(p.alpha, p.rank, p.strength, up.request_scale) - cs["ffn_pair"]) < 1e-15
    lin4, _ = workloads.config4("small")
    got = [lora.combined_scale(p.alpha, p.rank, p.strength, lin4.request_scale) for p in lin4.patches]
    assert np.allclose(got, cs["sidecar"], rtol=0, atol=1e-15)


def _brute_force(X, W, bias, patches, rs):
    T, n_in = len(X), len(X[0])
    n_out = len(W)
    Y = [[0.0] * n_out for _ in range(T)]
    for t, o in itertools.product(range(T), range(n_out)):
        acc = sum(X[t][i] * W[o][i] for i in range(n_in))
        if bias is not None:
            acc += bias[o]
        for (A, B, alpha, strength) in patches:
            r = len(A)
            s = alpha / r * strength * rs
            for j in range(r):
                h = sum(X[t][i] * A[j][i] for i in range(n_in))
                acc += s * h * B[o][j]
        Y[t][o] = acc
    return Y


@pytest.mark.parametrize("seed", range(6))
def test_forward_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    T, n_in, n_out = rng.integers(1, 6), rng.integers(1, 9), rng.integers(1, 7)
    X = rng.standard_normal((T, n_in)); W = rng.standard_normal((n_out, n_in))
    bias = rng.standard_normal(n_out) if seed % 2 else None
    raw = []
    for r in rng.integers(1, 4, size=rng.integers(1, 4)):
        raw.append((rng.standard_normal((r, n_in)), rng.standard_normal((n_out, r)),
                    float(rng.uniform(1, 64)), float(rng.uniform(-1, 1))))
    rs = float(rng.uniform(0.1, 2))
    want = _brute_force(X.tolist(), W.tolist(), None if bias is None else bias.tolist(),
                        [(A.tolist(), B.tolist(), a, s) for A, B, a, s in raw], rs)
    got = lora.linear_fwd(X, W, bias, [_patch(A, B, a, s) for A, B, a, s in raw], rs)
    assert np.allclose(got, np.array(want), rtol=1e-12, atol=1e-12)


def _rand_problem(rng, T=7, n_in=12, n_out=10, ranks=(3, 5)):
    X = rng.standard_normal((T, n_in)); W = rng.standard_normal((n_out, n_in))
    bias = rng.standard_normal(n_out)
    patches = [_patch(rng.standard_normal((r, n_in)), rng.standard_normal((n_out, r)),
                      float(2 * r), float(rng.uniform(-1, 1))) for r in ranks]
    return X, W, bias, patches


def test_merged_weight_identity():
    # the forward is linear: X (W + s B A)^T == X W^T + s (X A^T) B^T
    rng = np.random.default_rng(1)
    X, W, bias, patches = _rand_problem(rng)
    Wm = W.copy()
    for p in patches:
        Wm += lora.combined_scale(p.alpha, p.rank, p.strength, 0.7) * (p.B @ p.A)
    assert np.allclose(lora.linear_fwd(X, W, bias, patches, 0.7), X @ Wm.T + bias, rtol=1e-12, atol=1e-12)


def test_zero_scale_or_zero_A_is_the_base_linear():
    rng = np.random.default_rng(2)
    X, W, bias, patches = _rand_problem(rng)
    base = X @ W.T + bias
    assert np.array_equal(lora.linear_fwd(X, W, bias, patches, 0.0), base)
    zeroA = [_patch(np.zeros_like(p.A), p.B, p.alpha, p.strength) for p in patches]
    assert np.array_equal(lora.linear_fwd(X, W, bias, zeroA, 1.3), base)
    assert np.array_equal(lora.linear_fwd(X, W, bias, [], 1.3), base)   # adapter disabled


def test_delta_is_linear_in_s():
    rng = np.random.default_rng(3)
    X, W, bias, patches = _rand_problem(rng)
    base = X @ W.T + bias
    d1 = lora.linear_fwd(X, W, bias, patches, 0.4) - base
    d2 = lora.linear_fwd(X, W, bias, patches, 0.8) - base
    assert np.allclose(d2, 2 * d1, rtol=1e-12, atol=1e-12)


def test_multi_patch_is_sum_of_single_patches():
    rng = np.random.default_rng(4)
    X, W, bias, patches = _rand_problem(rng, ranks=(2, 4, 6))
    base = X @ W.T + bias
    total = lora.linear_fwd(X, W, bias, patches, 0.9) - base
    singles = sum(lora.linear_fwd(X, W, bias, [p], 0.9) - base for p in patches)
    assert np.allclose(total, singles, rtol=1e-12, atol=1e-12)


def test_grouped_equals_separate_linears():
    rng = np.random.default_rng(5)
    G, og = 3, 4
    X = rng.standard_normal((6, 8)); W = rng.standard_normal((G * og, 8))
    bias = rng.standard_normal(G * og)
    gp = [_patch(rng.standard_normal((2, 8)), rng.standard_normal((og, 2)), 4.0, 0.5 + g) for g in range(G)]
    Y = lora.linear_fwd_grouped(X, W, bias, gp, 1.5)
    for g in range(G):
        sl = slice(g * og, (g + 1) * og)
        assert np.allclose(Y[:, sl], lora.linear_fwd(X, W[sl], bias[sl], [gp[g]], 1.5), rtol=1e-12, atol=1e-12)


def test_backward_finite_differences():
    rng = np.random.default_rng(6)
    T, n_in, n_out, r = 4, 5, 6, 2
    X = rng.standard_normal((T, n_in)); W = rng.standard_normal((n_out, n_in))
    A = rng.standard_normal((r, n_in)); B = rng.standard_normal((n_out, r))
    dY = rng.standard_normal((T, n_out))
    alpha, strength, rs = 3.0, 0.7, 1.1

    def loss(X_, A_, B_):
        return float(np.sum(dY * lora.linear_fwd(X_, W, None, [_patch(A_, B_, alpha, strength)], rs)))

    g = lora.linear_bwd(X, W, dY, [_patch(A, B, alpha, strength)], rs)
    h = 1e-6
    for name, arr, grad in (("X", X, g.dX), ("A", A, g.dA[0]), ("B", B, g.dB[0])):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h; minus[idx] -= h
            args = {"X": X, "A": A, "B": B}
            args[name] = plus; lp = loss(args["X"], args["A"], args["B"])
            args[name] = minus; lm = loss(args["X"], args["A"], args["B"])
            num[idx] = (lp - lm) / (2 * h)
        assert np.allclose(grad, num, rtol=1e-6, atol=1e-7), name


def test_backward_dX_merged_identity_grouped():
    rng = np.random.default_rng(8)
    G, og, n_in, T = 2, 5, 6, 3
    X = rng.standard_normal((T, n_in)); W = rng.standard_normal((G * og, n_in))
    dY = rng.standard_normal((T, G * og))
    gp = [_patch(rng.standard_normal((3, n_in)), rng.standard_normal((og, 3)), 3.0, 1.0 - g) for g in range(G)]
    g = lora.linear_bwd(X, W, dY, gp, 0.5)
    Wm = W.copy()
    for i, p in enumerate(gp):
        Wm[i * og:(i + 1) * og] += lora.combined_scale(p.alpha, p.rank, p.strength, 0.5) * (p.B @ p.A)
    assert np.allclose(g.dX, dY @ Wm, rtol=1e-12, atol=1e-12)


def test_unfused_chain_exact_on_small_integers_and_bf16_valued():
    # with small integers every intermediate is exact in bf16, so the chain equals
    # the definition
    rng = np.random.default_rng(9)
    X = rng.integers(-3, 4, (5, 6)).astype(float); W = rng.integers(-3, 4, (4, 6)).astype(float)
    A = rng.integers(-2, 3, (2, 6)).astype(float); B = rng.integers(-2, 3, (4, 2)).astype(float)
    p = _patch(A, B, 4.0, 0.5)     # s = 1: alpha/r = 2, strength 0.5
    y = lora.linear_fwd(X, W, None, [p], 1.0)
    c = lora.unfused_bf16_chain(X, W, None, [p], 1.0)
    assert np.array_equal(c, y)
    rng = np.random.default_rng(10)
    X, W, bias, patches = _rand_problem(rng)
    c = lora.unfused_bf16_chain(X, W, bias, patches, 0.3)
    assert np.array_equal(f64_to_bf16_value(c), c)
    assert relative_rms(c, lora.linear_fwd(X, W, bias, patches, 0.3)) < 2e-2


def test_workload_generators_are_deterministic_and_shaped():
    a = workloads.config1("small"); b = workloads.config1("small")
    assert np.array_equal(a.X.data, b.X.data) and np.array_equal(a.patches[2].B.data, b.patches[2].B.data)
    assert a.W.shape == (3 * 320, 320) and a.groups == 3 and a.patches[0].rank == 32
    gu, down = workloads.config3("small")
    assert gu.W.kind == "nf4" and gu.W.absmax.shape == (2 * 320 * 256 // 64,)
    lin4, payload = workloads.config4("small")
    assert [p.A.kind for p in lin4.patches] == ["fp32", "bf16", "bf16"]
    assert payload.shape == (384, 384)


# ----------------------------------------------------------------- the unfused chain's roundings
def _chain_examples(golden_dir):
    with open(os.path.join(golden_dir, "unfused_chain_examples.json")) as f:
        return json.load(f)["examples"]


def _chain_inputs(ex):
    X = np.array(ex["X"], float)
    W = np.array(ex["W"], float)
    bias = None if ex["bias"] is None else np.array(ex["bias"], float)
    pats = []
    for q in ex["patches"]:
        p = _patch(q["A"], q["B"], q["alpha"], q["strength"], q["fp32"])
        if q.get("bias_B") is not None:
            p.bias_B = np.array(q["bias_B"], float)
        pats.append(p)
    return X, W, bias, pats, ex["request_scale"]


def test_unfused_chain_hand_examples(golden_dir):
    """Each hand-worked example pins one or two of the chain's bf16 roundings (the values
    in the file were worked by hand, step by step)."""
    for ex in _chain_examples(golden_dir):
        X, W, bias, pats, rs = _chain_inputs(ex)
        assert lora.unfused_bf16_chain(X, W, bias, pats, rs).tolist() == ex["Y_chain"], ex["name"]
        assert lora.linear_fwd(X, W, bias, pats, rs).tolist() == ex["Y_def"], ex["name"]


MUTATIONS = ["no_base_round", "bias_after_round", "no_t_round", "no_d_round", "bias_B_after_round",
             "no_alpha_round", "no_strength_round", "no_scale_round", "one_round_for_scales",
             "no_add_round", "sum_deltas_then_round", "fp32_adapter_rounded", None]


def _mutant_chain(X, W, bias, patches, rs, mut):
    """A test-side variant of the chain with one rounding taken out or one added; mut=None
    is the chain as the sglang PR's Motivation describes it."""
    rnd = f64_to_bf16_value
    keep = lambda v, m: v if mut == m else rnd(v)
    xw = X @ W.T
    if mut == "bias_after_round":
        base = rnd(rnd(xw) + (0.0 if bias is None else bias))
    else:
        base = keep(xw + (0.0 if bias is None else bias), "no_base_round")
    Y = base
    deltas = []
    for p in patches:
        vb = 0.0 if p.bias_B is None else p.bias_B.reshape(1, -1)
        cs = [np.float64(np.float32(p.alpha / p.rank)), np.float64(np.float32(p.strength)),
              np.float64(np.float32(rs))]
        if p.fp32_adapter and mut != "fp32_adapter_rounded":
            d = (X @ p.A.T) @ p.B.T + vb
            for c in cs:
                d = d * c
        else:
            t = keep(X @ p.A.T, "no_t_round")
            if mut == "bias_B_after_round":
                d = rnd(rnd(t @ p.B.T) + vb)
            else:
                d = keep(t @ p.B.T + vb, "no_d_round")
            if mut == "one_round_for_scales":
                d = rnd(d * cs[0] * cs[1] * cs[2])
            else:
                for c, m in zip(cs, ("no_alpha_round", "no_strength_round", "no_scale_round")):
                    if c != 1.0:
                        d = keep(d * c, m)
        deltas.append(d)
    if mut == "sum_deltas_then_round":
        return rnd(Y + sum(deltas))
    for d in deltas:
        Y = keep(Y + d, "no_add_round")
    return Y


@pytest.mark.parametrize("mut", MUTATIONS)
def test_chain_examples_catch_each_rounding_mutation(golden_dir, mut):
    """A chain with one rounding dropped or one extra rounding fails at least one stored
    example; the unmutated variant reproduces all of them (so the variant is faithful)."""
    exs = _chain_examples(golden_dir)
    diffs = []
    for ex in exs:
        X, W, bias, pats, rs = _chain_inputs(ex)
        diffs.append(_mutant_chain(X, W, bias, pats, rs, mut).tolist() != ex["Y_chain"])
    if mut is None:
        assert not any(diffs)
    else:
        assert any(diffs), mut
