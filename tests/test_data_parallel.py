"""The N > 1 path on CPU: two gloo ranks, each holding a contiguous block of token rows.

The per-shard backward is the FP64 oracle here (no GPU in these tests); what is under test
is the sharding, the single all-reduce of dA/dB and the max-over-ranks timing, against the
single-process oracle on the whole batch (dA and dB are sums over token rows, so the shards'
results must add up to the full result; dX is per row)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import lora as olora
from weight_patches_gb300 import data_parallel as wdp


def test_shard_rows_cover_exactly():
    for T in (0, 1, 7, 300, 32760):
        for world in (1, 2, 3, 8):
            spans = [wdp.shard_rows(T, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        wdp.shard_rows(10, 2, 2)


def _problem(seed=0):
    rng = np.random.default_rng(seed)
    T, K, G, og, r = 37, 24, 2, 16, 4
    X = rng.normal(0, 1, (T, K))
    W = rng.normal(0, 0.2, (G * og, K))
    dY = rng.normal(0, 1, (T, G * og))
    patches = [olora.DecodedPatch(rng.normal(0, 0.3, (r, K)), rng.normal(0, 0.3, (og, r)), 8.0, 0.7)
               for _ in range(G)]
    return X, W, dY, patches


def _oracle_bwd(X, W, dY, patches, request_scale):
    """A per-shard backward with the library's call shape, computed by the oracle."""
    g = olora.linear_bwd(X.double().numpy(), W, dY.double().numpy(), patches, request_scale)
    return (torch.from_numpy(g.dX), [torch.from_numpy(a).float() for a in g.dA],
            [torch.from_numpy(b).float() for b in g.dB])


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, W, dY, patches = _problem()
        a, b = wdp.shard_rows(X.shape[0], rank, world)
        dX, dA, dB = wdp.lora_linear_bwd_dp(torch.from_numpy(X[a:b]), W, torch.from_numpy(dY[a:b]), patches,
                                            0.9, local_bwd=_oracle_bwd)
        t = wdp.max_over_ranks(1.0 + rank)
        results[rank] = (a, b, dX.numpy(), [x.numpy() for x in dA], [x.numpy() for x in dB], t)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_match_the_whole_batch():
    world = 2
    # every process here starts by spawn (no fork after a CUDA context may exist)
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    X, W, dY, patches = _problem()
    full = olora.linear_bwd(X, W, dY, patches, 0.9)
    for rank in range(world):
        a, b, dX, dA, dB, t = res[rank]
        np.testing.assert_allclose(dX, full.dX[a:b], rtol=1e-12, atol=1e-12)
        for got, want in zip(dA + dB, full.dA + full.dB):
            np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6)
        assert t == float(world)                       # the slowest rank's value
    # both ranks hold the same reduced dA/dB
    for x, y in zip(res[0][3] + res[0][4], res[1][3] + res[1][4]):
        assert np.array_equal(x, y)


def test_single_process_is_a_no_op():
    X, W, dY, patches = _problem(1)
    dX, dA, dB = wdp.lora_linear_bwd_dp(torch.from_numpy(X), W, torch.from_numpy(dY), patches, 1.0,
                                        local_bwd=_oracle_bwd)
    full = olora.linear_bwd(X, W, dY, patches, 1.0)
    np.testing.assert_allclose(dA[0].numpy(), full.dA[0], rtol=1e-5)
    assert wdp.max_over_ranks(3.5) == 3.5


@pytest.mark.gpu
def test_default_backend_is_the_library():
    """Single process: the data-parallel call is the library's backward, bit for bit."""
    import weight_patches_gb300 as wpg
    import workloads
    from tests import gpu_util as gu
    _, down = workloads.config3("small")
    X, W, dY = gu.dev(down.X), gu.dev(down.W), gu.dev(down.dY)
    ads = gu.adapters(down)
    dX0, dA0, dB0 = wpg.lora_linear_bwd(X, W, dY, ads, 1.0)
    dX1, dA1, dB1 = wdp.lora_linear_bwd_dp(X, W, dY, ads, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(dX0, dX1) and all(torch.equal(a, b) for a, b in zip(dA0 + dB0, dA1 + dB1))
