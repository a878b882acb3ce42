"""Pins for the stochastic re-encoding of a 4-bit merge and its generator (oracle side).

piper-offload docs, "LoRA merge": a quantised merge re-encodes stochastically by default, so
that updates smaller than one quantisation step are not rounded away systematically; only
the terminal code is sampled, between the two neighbouring values of the finalised grid;
exact endpoints keep their code; samples are keyed by logical element index.  The pages name
no generator, so the generator is pinned by the properties any good counter-based one has
(and a weakened one loses), and the rule by what the pages fix: the two neighbours only,
exact levels kept, and no bias on average.
"""
import numpy as np
import pytest

from oracle import merge as om
from oracle import nf4 as onf4
from oracle import rng as orng


def _words(n, seed=99, rounds=orng.ROUNDS, base=0):
    q = np.arange(base, base + n, dtype=np.uint64)
    k0, k1 = orng.seed_words(seed)
    z = np.zeros(n, dtype=np.uint32)
    c0 = (q & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    c1 = (q >> np.uint64(32)).astype(np.uint32)
    return np.stack(orng.philox4x32(c0, c1, z, z, k0, k1, rounds=rounds))


def _chi2(counts):
    exp = counts.sum() / counts.size
    return float(((counts - exp) ** 2 / exp).sum())


def test_bytes_and_draws_uniform():
    w = _words(1 << 16)
    by = w.astype(np.uint32).view(np.uint8).ravel()
    c = np.bincount(by, minlength=256)
    # chi-square with 255 degrees of freedom: mean 255, sd 22.6
    assert 120 < _chi2(c) < 390
    U = orng.element_uniform23(np.arange(1 << 18), 5)
    assert U.max() < (1 << 23)
    c = np.bincount(U >> 15, minlength=256)
    assert 120 < _chi2(c) < 390


def _avalanche(rounds, trials=64):
    rng = np.random.default_rng(3)
    base = rng.integers(0, 2 ** 32, size=(trials, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2 ** 32, size=(trials, 2), dtype=np.uint64).astype(np.uint32)
    out0 = np.stack(orng.philox4x32(*base.T, *key.T, rounds=rounds), axis=1)
    worst = 0.0
    for bit in range(128 + 64):
        c, k = base.copy(), key.copy()
        if bit < 128:
            c[:, bit // 32] ^= np.uint32(1 << (bit % 32))
        else:
            k[:, (bit - 128) // 32] ^= np.uint32(1 << ((bit - 128) % 32))
        out1 = np.stack(orng.philox4x32(*c.T, *k.T, rounds=rounds), axis=1)
        flips = np.unpackbits((out0 ^ out1).view(np.uint8), axis=1).sum(axis=1)
        worst = max(worst, abs(flips.mean() - 64.0))
    return worst


def test_full_avalanche_after_ten_rounds():
    # every input bit flips each output bit with probability 1/2: 64 of 128 on average (the
    # mean of 64 trials has sd 0.7)
    assert _avalanche(orng.ROUNDS) < 4.0
    # teeth: one round is far from it
    assert _avalanche(1) > 20.0


def test_no_collisions_and_no_neighbour_correlation():
    w = _words(1 << 20, seed=1)
    flat = w.T.copy().view(np.dtype((np.void, 16))).ravel()
    assert np.unique(flat).size == flat.size
    U = orng.element_uniform23(np.arange(1 << 18), 11).astype(np.float64)
    r = np.corrcoef(U[:-1], U[1:])[0, 1]
    assert abs(r) < 5 / np.sqrt(U.size)


def test_seed_words_both_matter():
    e = np.arange(4096)
    a = orng.element_uniform23(e, 1)
    assert not np.array_equal(a, orng.element_uniform23(e, 2))
    assert not np.array_equal(a, orng.element_uniform23(e, 1 + (1 << 32)))
    assert np.array_equal(a, orng.element_uniform23(e, 1))


def _blocks(rows=64, cols=128, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)


def test_codes_are_neighbours_and_exact_levels_kept():
    u = _blocks()
    lv = onf4.codebook_f32()
    # a block of exact levels times a power of two (so x = level exactly)
    u[0, :64] = np.resize(lv, 64) * np.float32(0.25)
    codes, m, x, slack = om.quantize_blocks_stochastic(u, 17)
    det, m2, x2 = om.quantize_blocks(u)
    assert np.array_equal(m, m2) and np.array_equal(x, x2)
    below = np.sum(x[..., None] > lv, axis=-1)
    exact = lv[np.minimum(below, 15)] == x
    lo_i = np.where(exact, np.minimum(below, 15), below - 1)
    hi_i = np.where(exact, lo_i, below)
    assert np.all((codes == lo_i) | (codes == hi_i))
    assert np.array_equal(codes[exact], lo_i[exact])
    assert np.array_equal(codes[0, :64], np.resize(np.arange(16), 64).astype(np.uint8))
    assert np.all(np.abs(codes.astype(int) - det.astype(int)) <= 1)
    z = np.zeros((2, 64), dtype=np.float32)
    assert np.all(om.quantize_blocks_stochastic(z, 3)[0] == 7)


def test_unbiased_on_average():
    u = _blocks(8, 128, seed=4)
    lv = onf4.codebook_f64()
    n = 600
    acc = np.zeros(u.shape)
    for s in range(n):
        codes, m, x, _ = om.quantize_blocks_stochastic(u, 1000 + s)
        acc += lv[codes]
    mean = acc / n
    x = x.astype(np.float64)
    below = np.sum(x[..., None] > lv, axis=-1)
    hi = lv[np.clip(below, 1, 15)]
    lo = lv[np.clip(below, 1, 15) - 1]
    p = np.clip((x - lo) / (hi - lo), 0, 1)
    sd = np.sqrt(p * (1 - p) / n) * (hi - lo) + 1e-12
    z = (mean - x) / sd
    assert np.all(np.abs(z) < 6)
    # the deterministic code is biased by up to half a step; the stochastic mean is not
    det = lv[om.quantize_blocks(u)[0]]
    assert np.abs(mean - x).mean() < 0.25 * np.abs(det - x).mean()


def test_a_broken_generator_is_caught(monkeypatch):
    u = _blocks(8, 128, seed=5)
    monkeypatch.setattr(orng, "element_uniform23", lambda e, seed: np.full(np.shape(e), 1 << 22, np.uint32))
    lv = onf4.codebook_f64()
    acc = np.zeros(u.shape)
    for s in range(50):
        acc += lv[om.quantize_blocks_stochastic(u, s)[0]]
    x = om.quantize_blocks(u)[2].astype(np.float64)
    # a constant draw rounds at the halfway point between levels: as biased as round to nearest
    assert np.abs(acc / 50 - x).mean() > 0.5 * np.abs(lv[om.quantize_blocks(u)[0]] - x).mean()


@pytest.mark.parametrize("seed", [0, 2 ** 63 + 5])
def test_merge_nf4_with_seed(seed):
    rng = np.random.default_rng(8)
    import workloads
    from oracle.lora import decode_patch
    W0 = workloads.draw_nf4(rng, 64, 128)
    A = workloads.draw(rng, 4, 128, 0.1)
    B = workloads.draw(rng, 64, 4, 0.1)
    p = decode_patch(workloads.Patch(A, B, 4.0, 1.0))
    c1, m1, x1, _ = om.merge_nf4(W0.data, W0.absmax, 64, 128, [p], 1.0, rounding_seed=seed)
    c2, m2, x2 = om.merge_nf4(W0.data, W0.absmax, 64, 128, [p], 1.0)
    assert np.array_equal(m1, m2) and np.array_equal(x1, x2)
    assert np.all(np.abs(c1.astype(int) - c2.astype(int)) <= 1)
    again = om.merge_nf4(W0.data, W0.absmax, 64, 128, [p], 1.0, rounding_seed=seed)[0]
    assert np.array_equal(c1, again)
