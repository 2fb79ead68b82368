"""The allocation-free backward entry point (fa_bwd_noalloc).

Callers that cannot allocate device memory use fa_bwd_noalloc, which runs the
same kernels as fa_bwd with the library's fixed device scratch array in place
of a caller workspace.  This checks, through the C ABI, that two calls in a
row give the same gradients as fa_bwd (within the backward tolerance), that
its gradients match the CPU fp64 oracle on their own, also after a call of
another shape has left its own values in the shared scratch, and that shapes
whose scratch would exceed the fixed maximum are refused.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_bwd_gb300 import fa
from tiled_attention_bwd_gb300.workloads import default_scale, make_inputs

GRAD_REL_FRO = 5e-2
FA_ERR_WORKSPACE = 5


def _rel_fro(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 333, 128, True),
                                            (2, 2, 512, 64, False)])
def test_noalloc_backward_matches_workspace_backward(B, H, N, d, causal):
    dev = torch.device("cuda:0")
    inp = make_inputs(B, H, N, d, seed=77 + N)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o, lse = fa.fa_fwd(q, k, v, causal, scale)
    ref = fa.fa_bwd(q, k, v, o, lse, do, causal, scale)
    assert fa.fa_check_device_status(dev) == 0
    for _ in range(2):
        got = tuple(torch.full_like(q, float("nan")) for _ in range(3))
        fa.fa_bwd_noalloc(q, k, v, o, lse, do, causal, scale, *got)
        assert fa.fa_check_device_status(dev) == 0
        for g, r in zip(got, ref):
            assert torch.isfinite(g.float()).all()
            assert _rel_fro(g, r) <= GRAD_REL_FRO


@pytest.mark.gpu
def test_noalloc_backward_matches_oracle_across_shapes():
    # Shape A, then shape B (a different layout of the shared scratch), then
    # shape A again: each call's gradients are checked against the oracle,
    # so nothing a previous call left in the scratch may leak into them.
    dev = torch.device("cuda:0")
    shapes = [(2, 3, 333, 128, True), (1, 2, 700, 64, False),
              (2, 3, 333, 128, True)]
    for x, (B, H, N, d, causal) in enumerate(shapes):
        inp = make_inputs(B, H, N, d, seed=500 + N)
        q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
        scale = default_scale(d)
        o, lse = fa.fa_fwd(q, k, v, causal, scale)
        got = tuple(torch.full_like(q, float("nan")) for _ in range(3))
        fa.fa_bwd_noalloc(q, k, v, o, lse, do, causal, scale, *got)
        assert fa.fa_check_device_status(dev) == 0
        refs = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                          scale)
        for name, g, r in zip(("dq", "dk", "dv"), got, refs):
            g = g.double().cpu().numpy()
            assert np.isfinite(g).all(), (x, name)
            rf = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
            assert rf <= GRAD_REL_FRO, (x, name, rf)


@pytest.mark.gpu
def test_noalloc_backward_refuses_shapes_beyond_its_scratch():
    lib = fa.load_library()
    limit = lib.fa_bwd_noalloc_max_workspace()
    B, H, N, d = 1, 64, 4096, 128
    assert lib.fa_bwd_workspace_size(B, H, N, d) > limit
    p = ctypes.c_void_p(16)
    status = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 1,
                                0.125, None)
    assert status == FA_ERR_WORKSPACE
