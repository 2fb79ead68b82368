"""Failure detection on the GPU without a GPU fault.

Every pipeline wait inside the kernels has a time limit.  The library's
self-test kernel waits on a barrier that nothing ever signals; with a 20 ms
limit the wait runs out, records FA_ERR_DEVICE_TIMEOUT in the device status
record and returns.  The test checks that the status is reported once,
cleared, and that the GPU context still runs attention afterwards.
"""
import pytest
import torch

from tiled_attention_bwd_gb300 import (fa_check_device_status,
                                       fa_debug_expire_wait, fa_fwd,
                                       fa_set_wait_timeout_ns)
from tiled_attention_bwd_gb300.workloads import make_inputs

FA_ERR_DEVICE_TIMEOUT = 4


@pytest.mark.gpu
def test_expired_wait_is_reported_and_context_survives():
    dev = torch.device("cuda:0")
    assert fa_check_device_status(dev) == 0
    fa_set_wait_timeout_ns(20_000_000)
    try:
        fa_debug_expire_wait(dev)
        assert fa_check_device_status(dev) == FA_ERR_DEVICE_TIMEOUT
        assert fa_check_device_status(dev) == 0  # reported once, then cleared
    finally:
        fa_set_wait_timeout_ns(0)
    inp = make_inputs(1, 1, 256, 128, seed=1)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o, lse = fa_fwd(q, k, v, True, 0.125)
    assert fa_check_device_status(dev) == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
