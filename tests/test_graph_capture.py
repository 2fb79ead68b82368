"""The forward and backward calls captured into one CUDA graph.

A training or serving loop that replays a captured step (as the benchmark
does) gets the same results as eager calls: the graph is captured once on
static buffers, then replayed on two different seeded inputs copied into
them, and each replay is compared with the CPU fp64 oracle at the parity
tolerances.  The main-kernel events of fa_bwd_set_phase_events, recorded
inside the graph, time the kernel on every replay.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_bwd_gb300 import (fa_bwd, fa_bwd_set_phase_events,
                                       fa_bwd_workspace_size,
                                       fa_check_device_status, fa_fwd)
from tiled_attention_bwd_gb300.workloads import default_scale, make_inputs

pytestmark = pytest.mark.gpu

O_MAX_ABS, LSE_MAX_ABS, GRAD_REL_FRO = 2e-2, 1e-3, 5e-2


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def f64(t):
    return t.detach().to("cpu").double().numpy()


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 333, 128, True),
                                            (2, 4, 512, 64, False)])
def test_captured_step_matches_oracle_on_every_replay(B, H, N, d, causal):
    dev = torch.device("cuda:0")
    scale = default_scale(d)
    first = make_inputs(B, H, N, d, seed=101 + N)
    q, k, v, do = (first[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8,
                     device=dev)
    # The library records these itself, as external events of the graph.
    ev = (torch.cuda.Event(enable_timing=True),
          torch.cuda.Event(enable_timing=True))
    for e in ev:                      # torch creates events on first record
        e.record()

    def step():
        fa_fwd(q, k, v, causal, scale, out=o, lse=lse)
        fa_bwd(q, k, v, o, lse, do, causal, scale, dq=dq, dk=dk, dv=dv,
               workspace=ws)

    step()                            # eager warm-up outside the capture
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    fa_bwd_set_phase_events(*ev)
    try:
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            step()
    finally:
        fa_bwd_set_phase_events(None, None)

    for seed in (101 + N, 202 + N):
        inp = make_inputs(B, H, N, d, seed=seed)
        for name, t in (("q", q), ("k", k), ("v", v), ("do", do)):
            t.copy_(inp[name].to(dev))
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan"))     # a replay that skips a write shows
        g.replay()
        torch.cuda.synchronize(dev)
        assert fa_check_device_status(dev) == 0
        assert ev[0].elapsed_time(ev[1]) > 0.0
        o_ref, lse_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], causal,
                                    scale)
        refs = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                          scale)
        assert np.max(np.abs(f64(o) - o_ref)) <= O_MAX_ABS, seed
        assert np.max(np.abs(f64(lse) - lse_ref)) <= LSE_MAX_ABS, seed
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            got = f64(got)
            assert np.isfinite(got).all(), (seed, name)
            assert rel_fro(got, ref) <= GRAD_REL_FRO, (seed, name)
