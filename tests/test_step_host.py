"""fa_step_host: the training step on host tensors, pipelined by head chunks.

Every chunk runs the same kernels on its heads as fa_fwd + fa_bwd do on all
of them, so O, LSE, dK and dV must be bit-identical to the device-resident
calls (heads are independent and each element has one writer); dQ sums its
key tiles through fp32 reductions in any order and is compared within a
tight relative bound.  A small case is also checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_bwd_gb300 import (fa_bwd, fa_check_device_status, fa_fwd,
                                       fa_step_host)
from tiled_attention_bwd_gb300.workloads import default_scale, make_inputs

pytestmark = pytest.mark.gpu


def run_host(inp, causal, scale, chunk_heads):
    B, H, N, d = inp["q"].shape
    host = {n: inp[n].pin_memory() for n in ("q", "k", "v", "do")}
    outs = {n: torch.empty_like(host["q"]).pin_memory()
            for n in ("o", "dq", "dk", "dv")}
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    dev = torch.device("cuda:0")
    fa_step_host(host["q"], host["k"], host["v"], host["do"], causal, scale,
                 outs["o"], lse, outs["dq"], outs["dk"], outs["dv"],
                 chunk_heads=chunk_heads, device=dev)
    torch.cuda.synchronize(dev)
    assert fa_check_device_status(dev) == 0
    return outs["o"], lse, outs["dq"], outs["dk"], outs["dv"]


def run_device(inp, causal, scale):
    dev = torch.device("cuda:0")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa_fwd(q, k, v, causal, scale)
    dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal, scale)
    assert fa_check_device_status(dev) == 0
    return tuple(t.cpu() for t in (o, lse, dq, dk, dv))


@pytest.mark.parametrize("B,H,N,d,causal,chunk", [
    (2, 8, 512, 128, True, 0),       # default: about eight chunks
    (2, 8, 512, 128, False, 5),      # ragged last chunk
    (1, 3, 333, 64, True, 1),        # one head per chunk, ragged N
    (1, 4, 256, 128, True, 100),     # one chunk
])
def test_host_step_equals_device_calls(B, H, N, d, causal, chunk):
    inp = make_inputs(B, H, N, d, seed=404 + N + chunk)
    scale = default_scale(d)
    got = run_host(inp, causal, scale, chunk)
    ref = run_device(inp, causal, scale)
    for name, g, r in zip(("o", "lse", "dk", "dv"), (got[0], got[1], got[3], got[4]),
                          (ref[0], ref[1], ref[3], ref[4])):
        assert torch.equal(g, r), name
    dq_g, dq_r = got[2].double().numpy(), ref[2].double().numpy()
    assert np.linalg.norm(dq_g - dq_r) <= 1e-2 * np.linalg.norm(dq_r)


def test_host_step_against_the_oracle():
    B, H, N, d, causal = 1, 2, 384, 128, True
    inp = make_inputs(B, H, N, d, seed=99)
    scale = default_scale(d)
    o, lse, dq, dk, dv = run_host(inp, causal, scale, 1)
    o_ref, lse_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], causal, scale)
    g_ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], causal, scale)
    assert np.max(np.abs(o.double().numpy() - o_ref)) <= 2e-2
    assert np.max(np.abs(lse.double().numpy() - lse_ref)) <= 1e-3
    for g, r in zip((dq, dk, dv), g_ref):
        g = g.double().numpy()
        assert np.linalg.norm(g - r) <= 5e-2 * np.linalg.norm(r)
