"""Failure detection on the GPU without a GPU fault.

Every pipeline wait inside the kernels has a time limit.
  * The library's self-test kernel waits on a barrier that nothing ever
    signals; with a 20 ms limit the wait runs out, records
    FA_ERR_DEVICE_TIMEOUT in the device status record and returns.
  * In the production kernels, the test hook fa_debug_expire_at makes the
    real waits at one site (those whose barrier is not complete at the first
    test) behave as if their limit had passed.  Each site below is a real
    wait at its first reach in the problem used here, and stops its grid
    with work in flight of the kind named beside it (TMA loads, tensor-core
    products), so the drains that run before tensor memory is released are
    exercised: the status must name the site, the next check must be clean,
    and a following call must match the CPU oracle.  The warps that wait as
    a whole (softmax, P/dS, dQ read-out) stop at their next wait through the
    block's abort flag in every case; their own first waits are not used as
    sites because a warp's first test of a barrier can suspend until the
    phase completes, so it may never take the slow path the hook is on.
No trap, fault or hang is ever provoked.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_bwd_gb300 import (fa_bwd, fa_check_device_status,
                                       fa_debug_expire_at,
                                       fa_debug_expire_wait, fa_fwd,
                                       fa_last_failure_site,
                                       fa_set_wait_timeout_ns)
from tiled_attention_bwd_gb300.workloads import default_scale, make_inputs

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


def _rel_fro(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def _check_against_oracle(inp, o, lse, grads, causal, scale):
    o_ref, lse_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], causal, scale)
    o = o.double().cpu().numpy()
    assert np.max(np.abs(o - o_ref)) <= 2e-2 and _rel_fro(o, o_ref) <= 1e-2
    assert np.max(np.abs(lse.double().cpu().numpy() - lse_ref)) <= 1e-3
    refs = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], causal, scale)
    for g, r in zip(grads, refs):
        assert _rel_fro(g.double().cpu().numpy(), r) <= 5e-2


# site, which pass, what is in flight when it stops (1 x 2 x 384 x 128
# causal: three key tiles, so the K/V ring of the forward fills and the
# first key tile of the backward visits three query tiles)
SITES = [
    (0x101, "fwd", "producer: K/V ring full, loads in flight"),
    (0x201, "fwd", "MMA thread: first Q wait, Q loads in flight"),
    (0x203, "fwd", "MMA thread: P wait, Q K^T products in flight"),
    (0x111, "bwd", "producer: third Q stage wait, loads and products in flight"),
    (0x112, "bwd", "producer: second dO wait"),
    (0x211, "bwd", "MMA thread: K wait, V, Q, dO, K loads in flight"),
    (0x214, "bwd", "MMA thread: P wait, S and dP products in flight"),
    (0x215, "bwd", "MMA thread: dS wait, dV and S products in flight"),
    (0x213, "bwd", "MMA thread: dQ read-out wait, dK and dQ in flight"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("site,which,what", SITES)
def test_production_kernel_timeout_path(site, which, what):
    dev = torch.device("cuda:0")
    B, H, N, d, causal = 1, 2, 384, 128, True
    inp = make_inputs(B, H, N, d, seed=4242)
    scale = default_scale(d)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    assert fa_check_device_status(dev) == 0
    if which == "bwd":
        o, lse = fa_fwd(q, k, v, causal, scale)
        assert fa_check_device_status(dev) == 0
    try:
        fa_debug_expire_at(site)
        if which == "fwd":
            fa_fwd(q, k, v, causal, scale)
        else:
            fa_bwd(q, k, v, o, lse, do, causal, scale)
        assert fa_check_device_status(dev) == FA_ERR_DEVICE_TIMEOUT, what
        assert fa_last_failure_site() == site, what
    finally:
        fa_debug_expire_at(0)
    assert fa_check_device_status(dev) == 0   # reported once, then cleared
    assert fa_last_failure_site() == 0
    # The context and the library work normally afterwards.
    o, lse = fa_fwd(q, k, v, causal, scale)
    grads = fa_bwd(q, k, v, o, lse, do, causal, scale)
    assert fa_check_device_status(dev) == 0
    _check_against_oracle(inp, o, lse, grads, causal, scale)
