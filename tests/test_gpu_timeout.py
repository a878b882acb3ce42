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


def test_wait_limit_range_is_checked():
    with pytest.raises(wpg.WeightPatchesError):
        wpg.lora_set_wait_limit(10)                              # below 1 ms
    wpg.lora_set_wait_limit(2_000_000_000)
