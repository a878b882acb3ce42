"""The element-wise bound the GPU parity tests apply (tests/gpu_util.py), checked on the CPU:
a float32 simulation of the single-rounding design (fp32 sums, s X A^T rounded once to bf16,
one output rounding) stays inside it on every element, and one corrupted element of that
output -- zeroed, negated, taken from the neighbouring column, or 10 % off --
falls outside it."""
import numpy as np
import pytest
import torch

import workloads
from oracle import lora as olora
from oracle.numerics import to_f64
from tests import gpu_util as gu


def _simulated_fused(lin):
    """Y = bf16(fl32(X W^T) + sum_p fl32(bf16(s_p fl32(X A_p^T)) B_p^T)) in torch float32."""
    X = lin.X.torch_cpu().float()
    W = torch.from_numpy(to_f64(lin.W)).float()       # a 4-bit weight as its bf16 W_eff
    Y = X @ W.T
    G = lin.groups
    og = W.shape[0] // G
    for i, p in enumerate(lin.patches):
        s = np.float32(olora.combined_scale(p.alpha, p.rank, p.strength, lin.request_scale))
        H = (X @ p.A.torch_cpu().float().T) * float(s)
        Ht = H.to(torch.bfloat16).float()
        sl = slice(i * og, (i + 1) * og) if G > 1 else slice(None)
        Y[:, sl] += Ht @ p.B.torch_cpu().float().T
    if lin.bias is not None:
        Y += lin.bias.torch_cpu().float().reshape(1, -1)
    return Y.to(torch.bfloat16).float().double().numpy()


@pytest.mark.parametrize("cfg", ["c1", "c2up", "c3down"])
def test_bound_accepts_the_single_rounding_design(cfg):
    lin = {"c1": lambda: workloads.config1("small"), "c2up": lambda: workloads.config2("small")[0],
           "c3down": lambda: workloads.config3("small")[1]}[cfg]()
    got = _simulated_fused(lin)
    want = olora.reference_output(lin)
    gu.assert_elementwise(got, want, gu.fwd_bound(lin, y_ref=want), cfg)


@pytest.mark.parametrize("how", ["zero", "negate", "neighbour", "ten_percent"])
def test_bound_rejects_one_corrupted_element(how):
    lin = workloads.config1("small")
    got = _simulated_fused(lin)
    want = olora.reference_output(lin)
    bound = gu.fwd_bound(lin, y_ref=want)
    # a typical element (not one that cancels to nearly zero)
    t, o = np.unravel_index(np.argsort(np.abs(want), axis=None)[want.size // 2], want.shape)
    bad = got.copy()
    bad[t, o] = {"zero": 0.0, "negate": -got[t, o], "neighbour": got[t, (o + 1) % got.shape[1]],
                 "ten_percent": got[t, o] * 1.1}[how]
    with pytest.raises(AssertionError):
        gu.assert_elementwise(bad, want, bound, how)
