"""The bounded-wait abort path of the fused forward, made to run out on purpose in the
sanctioned form: a row-block flag that nothing sets.

lora_debug_hold_flags(1) makes every tile wait for one more rank-item release than any rank
item gives; with the wait limit at 50 ms each CTA pair's bounded flag wait expires, records
WP_ERR_TIMEOUT in the device status word, raises its CTAs' abort flags (the MMA issuer and
the epilogue warps leave their own bounded waits), waits for its copies in flight, frees its
tensor memory and returns.  The host reads the status after the stream has finished; then,
with the hook off and the default limit back, a normal call on the same device must be
correct -- the context survived.  No wait is unbounded, nothing faults or traps."""
import time

import pytest
import torch

import weight_patches_gb300 as wpg
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_flag_wait_runs_out_and_the_device_stays_usable():
    lin = workloads.config1("small")
    lib = wpg.lib()
    assert wpg.lora_device_status(reset=True) in (0, -7)       # start clean
    wpg.lora_set_wait_limit(50_000_000)
    lib.lora_debug_hold_flags(1)
    try:
        t0 = time.time()
        gu.run_fwd(lin)                                          # launches; returns WP_OK
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        assert wpg.lora_device_status(reset=True) == -7          # WP_ERR_TIMEOUT, then cleared
    finally:
        lib.lora_debug_hold_flags(0)
        wpg.lora_set_wait_limit(2_000_000_000)
    assert elapsed < 30.0, elapsed
    # the same device, a normal call: correct, and no timeout recorded
    Y = gu.run_fwd(lin)
    err, chain = gu.errors(lin, Y)
    assert err <= 4e-3 and err <= chain
    assert wpg.lora_device_status() == 0


@pytest.mark.parametrize("cols", [512, 320])      # the 256-column and the 64-column one-pass merge
def test_merge_wait_runs_out_and_the_device_stays_usable(cols):
    """The one-pass 4-bit merge under the same hook: its CTAs' last MMAs are never issued, so
    the compute warps' bounded waits for them expire; every warp (and the producer) leaves,
    the copies and MMAs in flight are waited for, tensor memory is freed.  Then a normal merge
    on the same device matches the oracle."""
    import numpy as np
    from oracle import merge as om
    from oracle import nf4 as onf4
    from oracle.lora import decode_patch
    rng = np.random.default_rng(cols)
    rows = 256
    W0 = workloads.draw_nf4(rng, rows, cols)
    p = workloads.Patch(workloads.draw(rng, 16, cols, 0.05), workloads.draw(rng, rows, 16, 0.05), 16.0, 1.0)
    ads = [wpg.Adapter(gu.dev(p.A), gu.dev(p.B), p.alpha, p.strength)]
    lib = wpg.lib()
    assert wpg.lora_device_status(reset=True) in (0, -7)
    wpg.lora_set_wait_limit(50_000_000)
    lib.lora_debug_hold_flags(1)
    try:
        t0 = time.time()
        wpg.lora_merge(gu.dev(W0), ads, 1.0)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        assert wpg.lora_device_status(reset=True) == -7
    finally:
        lib.lora_debug_hold_flags(0)
        wpg.lora_set_wait_limit(2_000_000_000)
    assert elapsed < 30.0, elapsed
    W = gu.dev(W0)
    wpg.lora_merge(W, ads, 1.0)
    torch.cuda.synchronize()
    assert wpg.lora_device_status() == 0
    want_codes, want_am, x = om.merge_nf4(W0.data, W0.absmax, rows, cols, [decode_patch(p)], 1.0)
    got = onf4.unpack_codes(W.packed.cpu().numpy(), rows, cols)
    np.testing.assert_allclose(W.absmax.cpu().numpy(), want_am, rtol=1e-5, atol=0)
    lv = onf4.codebook_f64()
    near = np.min(np.abs(x[..., None].astype(np.float64) - (lv[:-1] + lv[1:]) / 2), axis=-1) <= 1e-5
    assert np.array_equal(got[~near], want_codes[~near])


def test_wait_limit_range_is_checked():
    with pytest.raises(wpg.WeightPatchesError):
        wpg.lora_set_wait_limit(10)                              # below 1 ms
    wpg.lora_set_wait_limit(2_000_000_000)
