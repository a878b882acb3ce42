"""Pins of the SwiGLU oracle against closed forms, identities and finite differences
(Unsloth fast_lora walkthrough, section 4, LoRA_MLP)."""
import math

import numpy as np

from oracle import swiglu as osw
from oracle.lora import DecodedPatch


def test_sigmoid_closed_forms():
    # exp(-ln 3) = 1/3, so sigmoid(ln 3) = 1 / (1 + 1/3) = 3/4 and sigmoid(-ln 3) = 1/4
    x = np.array([0.0, math.log(3.0), -math.log(3.0)])
    np.testing.assert_allclose(osw.sigmoid(x), [0.5, 0.75, 0.25], rtol=0, atol=1e-15)
    np.testing.assert_allclose(osw.silu(x), [0.0, 0.75 * math.log(3.0), -0.25 * math.log(3.0)],
                               rtol=0, atol=1e-15)


def test_sigmoid_symmetry_and_range():
    # sigmoid(x) + sigmoid(-x) = 1 and silu(x) - silu(-x) = x, far past exp's overflow
    x = np.concatenate([np.linspace(-800, 800, 1601), np.array([1e-300, -1e-300, 37.5, -37.5])])
    s = osw.sigmoid(x)
    assert np.all(np.isfinite(s)) and np.all(s >= 0) and np.all(s <= 1)
    np.testing.assert_allclose(s + osw.sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(osw.silu(x) - osw.silu(-x), x, rtol=1e-14, atol=1e-300)
    # limits: silu(x) -> x for large x, -> 0 for very negative x
    assert osw.silu(np.array([800.0]))[0] == 800.0
    assert abs(osw.silu(np.array([-800.0]))[0]) < 1e-300


def _fd(fun, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp = x.copy(); xp[i] += h
        xm = x.copy(); xm[i] -= h
        g[i] = (fun(xp) - fun(xm)) / (2 * h)
    return g


def test_swiglu_bwd_matches_finite_differences():
    rng = np.random.default_rng(0)
    e = rng.normal(0, 2.0, (4, 6))
    g = rng.normal(0, 1.0, (4, 6))
    dh = rng.normal(0, 1.0, (4, 6))
    h, dg, de = osw.swiglu_bwd(dh, e, g)
    np.testing.assert_allclose(h, osw.swiglu(e, g), rtol=1e-15, atol=0)
    loss_e = lambda ee: float(np.sum(dh * osw.swiglu(ee, g)))
    loss_g = lambda gg: float(np.sum(dh * osw.swiglu(e, gg)))
    np.testing.assert_allclose(de, _fd(loss_e, e), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dg, _fd(loss_g, g), rtol=1e-6, atol=1e-8)


def _patch(rng, r, d_in, d_out, alpha, strength):
    return DecodedPatch(rng.normal(0, 0.5, (r, d_in)), rng.normal(0, 0.5, (d_out, r)), alpha, strength)


def test_mlp_gradients_match_finite_differences():
    rng = np.random.default_rng(1)
    T, d, F, r = 3, 5, 4, 2
    X = rng.normal(0, 1, (T, d))
    Wgu = rng.normal(0, 0.5, (2 * F, d))
    bgu = rng.normal(0, 0.1, 2 * F)
    Wd = rng.normal(0, 0.5, (d, F))
    bd = rng.normal(0, 0.1, d)
    pg, pu = _patch(rng, r, d, F, 4.0, 0.7), _patch(rng, r, d, F, 2.0, -1.3)
    pdn = [_patch(rng, r, F, d, 2.0, 0.9), _patch(rng, 3, F, d, 1.5, 0.4)]   # two patches on down
    rs = 0.8
    dY = rng.normal(0, 1, (T, d))

    def loss(X_=X, pg_=pg, pu_=pu, pd_=pdn):
        return float(np.sum(dY * osw.lora_mlp_fwd(X_, Wgu, bgu, [pg_, pu_], Wd, bd, pd_, rs)[3]))

    gr = osw.lora_mlp_bwd(X, Wgu, bgu, [pg, pu], Wd, bd, pdn, rs, dY)
    np.testing.assert_allclose(gr["dX"], _fd(lambda x: loss(X_=x), X), rtol=1e-6, atol=1e-8)

    def with_patch(p, A=None, B=None):
        return DecodedPatch(p.A if A is None else A, p.B if B is None else B, p.alpha, p.strength)

    for k, p in enumerate([pg, pu]):
        dA, dB = gr["gate_up"][k]
        sel = (lambda q: dict(pg_=q)) if k == 0 else (lambda q: dict(pu_=q))
        np.testing.assert_allclose(dA, _fd(lambda a: loss(**sel(with_patch(p, A=a))), p.A), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(dB, _fd(lambda b: loss(**sel(with_patch(p, B=b))), p.B), rtol=1e-6, atol=1e-8)
    for k, p in enumerate(pdn):
        dA, dB = gr["down"][k]

        def repl(q):
            lst = list(pdn)
            lst[k] = q
            return dict(pd_=lst)
        np.testing.assert_allclose(dA, _fd(lambda a: loss(**repl(with_patch(p, A=a))), p.A), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(dB, _fd(lambda b: loss(**repl(with_patch(p, B=b))), p.B), rtol=1e-6, atol=1e-8)


def test_mlp_forward_composes_the_linears():
    # with all strengths zero the MLP is the plain SwiGLU MLP of the base weights
    rng = np.random.default_rng(2)
    T, d, F, r = 4, 6, 5, 2
    X = rng.normal(0, 1, (T, d))
    Wgu = rng.normal(0, 0.5, (2 * F, d))
    Wd = rng.normal(0, 0.5, (d, F))
    pg, pu, pdn = (_patch(rng, r, d, F, 2.0, 0.0), _patch(rng, r, d, F, 2.0, 0.0),
                   _patch(rng, r, F, d, 2.0, 0.0))
    e, g, h, y = osw.lora_mlp_fwd(X, Wgu, None, [pg, pu], Wd, None, [pdn], 1.0)
    e0, g0 = X @ Wgu[:F].T, X @ Wgu[F:].T
    np.testing.assert_allclose(e, e0, rtol=1e-14)
    np.testing.assert_allclose(g, g0, rtol=1e-14)
    np.testing.assert_allclose(y, (e0 / (1 + np.exp(-e0)) * g0) @ Wd.T, rtol=1e-13)
