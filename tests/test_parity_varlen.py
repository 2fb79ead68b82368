"""GPU parity of the per-sequence-length entry points.

fa_fwd_varlen / fa_bwd_varlen (batch entry b attends over its first L_b rows
of a padded [B,H,N,d] batch) against the CPU fp64 oracle's fwd_varlen /
bwd_varlen on the same seeded bf16 inputs, with the tolerances of the base
operation (O max-abs 2e-2 and rel-Frobenius 1e-2, LSE max-abs 1e-3, each
gradient rel-Frobenius 5e-2).  Lengths cover the tile edges (0, 1, 127, 128,
129, N) and compose with grouped heads, split head groups and the window.
Padding rows must hold finite values of any size: the inputs are random
there.  Also checked: the forward leaves padding rows of O and LSE as they
were, the backward zeroes every padding row of dQ, dK, dV, each sequence's
rows equal a standalone call on that sequence alone (bit for bit where each
element has one writer), and a captured CUDA graph honours lengths changed
in place between replays.  Thousands of short sequences cover both
forward schedules (the balanced item table and, where it does not fit in
shared memory, the plain order).
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_bwd_gb300 import (fa_bwd_ext, fa_bwd_varlen,
                                       fa_check_device_status, fa_fwd_ext,
                                       fa_fwd_varlen)
from tiled_attention_bwd_gb300.workloads import (default_scale,
                                                 make_grouped_inputs,
                                                 make_seq_lens, sample_heads)

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_FRO, LSE_MAX_ABS, GRAD_REL_FRO = 2e-2, 1e-2, 1e-3, 5e-2
SENTINEL = 7.0


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def f64(t):
    return t.detach().to("cpu").double().numpy()


def run_varlen(inp, lens, causal, scale, window, backward=True):
    dev = torch.device("cuda:0")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    sl = lens.to(dev)
    B, H, N, d = q.shape
    o = torch.full_like(q, SENTINEL)
    lse = torch.full((B, H, N), SENTINEL, dtype=torch.float32, device=dev)
    fa_fwd_varlen(q, k, v, sl, causal, scale, window, out=o, lse=lse)
    out = {"o": o, "lse": lse}
    if backward:
        # gradient buffers start non-zero: padding rows must be written
        dq = torch.full_like(q, SENTINEL)
        dk = torch.full_like(k, SENTINEL)
        dv = torch.full_like(v, SENTINEL)
        fa_bwd_varlen(q, k, v, o, lse, do, sl, causal, scale, window,
                      dq=dq, dk=dk, dv=dv)
        out.update(dq=dq, dk=dk, dv=dv)
    assert fa_check_device_status(dev) == 0
    return {k_: v_.cpu() for k_, v_ in out.items()}


def check_rows(got, lens, inp, causal, scale, window, tag):
    """Forward on real rows against the oracle, padding rows untouched."""
    o_ref, lse_ref = oracle.fwd_varlen(inp["q"], inp["k"], inp["v"], lens,
                                       causal, scale, window)
    o, lse = f64(got["o"]), f64(got["lse"])
    N = o.shape[2]
    real = np.arange(N)[None, :] < np.asarray(lens)[:, None]      # [B, N]
    sel = np.broadcast_to(real[:, None, :], lse.shape)            # [B, H, N]
    assert np.all(o[~sel] == SENTINEL) and np.all(lse[~sel] == SENTINEL), tag
    if sel.any():
        ov, orf = o[sel], o_ref[sel]
        assert np.isfinite(ov).all(), tag
        err = np.max(np.abs(ov - orf))
        assert err <= O_MAX_ABS, "%s O max-abs %.3g" % (tag, err)
        assert rel_fro(ov, orf) <= O_REL_FRO, tag
        le = np.max(np.abs(lse[sel] - lse_ref[sel]))
        assert le <= LSE_MAX_ABS, "%s LSE max-abs %.3g" % (tag, le)
    return real


def check_grads(got, lens, inp, causal, scale, window, tag):
    g_ref = oracle.bwd_varlen(inp["q"], inp["k"], inp["v"], inp["do"], lens,
                              causal, scale, window)
    N = got["dq"].shape[2]
    pad = np.arange(N)[None, :] >= np.asarray(lens)[:, None]
    for name, r in zip(("dq", "dk", "dv"), g_ref):
        g = f64(got[name])
        assert np.isfinite(g).all(), "%s %s" % (tag, name)
        assert not g[np.broadcast_to(pad[:, None, :], g.shape[:3])].any(), \
            "%s %s: padding rows not zero" % (tag, name)
        rf = rel_fro(g, r)
        assert rf <= GRAD_REL_FRO, "%s %s rel-Frobenius %.3g" % (tag, name, rf)


CASES = [
    # B, H, Hkv, N, d, causal, window, fixed lengths
    (6, 4, 2, 333, 128, True, -1, [0, 1, 127, 128, 129, 333]),
    (4, 2, 2, 512, 64, False, -1, [512, 300, 17, 256]),
    (3, 4, 1, 700, 128, False, 150, [700, 450, 129]),
    (3, 2, 1, 600, 64, True, 100, [600, 1, 257]),
    (2, 16, 1, 300, 128, True, -1, [300, 200]),      # split head groups
    (5, 2, 2, 1000, 128, True, -1, []),              # random lengths
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,window,fixed", CASES)
def test_varlen_every_element(B, H, Hkv, N, d, causal, window, fixed):
    inp = make_grouped_inputs(B, H, Hkv, N, d, seed=900 + N + H)
    lens = make_seq_lens(B, N, seed=N, fixed=fixed)
    scale = default_scale(d)
    tag = "%dx%d/%dx%dx%d causal=%d window=%d lens=%s" % (
        B, H, Hkv, N, d, causal, window, lens.tolist())
    got = run_varlen(inp, lens, causal, scale, window)
    check_rows(got, lens, inp, causal, scale, window, tag)
    check_grads(got, lens, inp, causal, scale, window, tag)


@pytest.mark.parametrize("lens,causal", [([0, 0, 0], True),
                                         ([260, -3, 7], False),
                                         ([999, 0, 300], True)])
def test_empty_and_out_of_range_lengths(lens, causal):
    # Every sequence empty: nothing is written but zero gradients.  Lengths
    # outside [0, N] are clamped (N = 300 here).
    B, H, Hkv, N, d = 3, 2, 1, 300, 64
    inp = make_grouped_inputs(B, H, Hkv, N, d, seed=55)
    lens = torch.tensor(lens, dtype=torch.int32)
    scale = default_scale(d)
    tag = "lens=%s causal=%d" % (lens.tolist(), causal)
    got = run_varlen(inp, lens, causal, scale, -1)
    clamped = lens.clamp(0, N)
    check_rows(got, clamped, inp, causal, scale, -1, tag)
    check_grads(got, clamped, inp, causal, scale, -1, tag)


@pytest.mark.parametrize("B,causal", [(2000, False), (2000, True),
                                      (4400, True), (4400, False)])
def test_many_short_sequences(B, causal):
    # The forward balances its items through a table in shared memory; with
    # 2000 sequences at d = 128 it fits, with 4400 it does not and the plain
    # item order (empty items skipped) runs instead.  Both must give the
    # same operation.
    H, N, d = 1, 130, 128
    inp = make_grouped_inputs(B, H, H, N, d, seed=B + causal)
    lens = make_seq_lens(B, N, seed=B, fixed=[0, 1, 128, 129, 130])
    lens[5::7] = 0
    scale = default_scale(d)
    tag = "B=%d causal=%d" % (B, causal)
    got = run_varlen(inp, lens, causal, scale, -1)
    check_rows(got, lens, inp, causal, scale, -1, tag)
    check_grads(got, lens, inp, causal, scale, -1, tag)


@pytest.mark.parametrize("H,Hkv,N,d,causal,window", [
    (4, 2, 640, 128, True, -1),
    (2, 1, 513, 64, False, 200),
])
def test_each_sequence_equals_a_standalone_call(H, Hkv, N, d, causal, window):
    B = 4
    inp = make_grouped_inputs(B, H, Hkv, N, d, seed=31 + N)
    lens = make_seq_lens(B, N, seed=77, fixed=[N, 129, 1, 300])
    scale = default_scale(d)
    got = run_varlen(inp, lens, causal, scale, window)
    dev = torch.device("cuda:0")
    for b, L in enumerate(lens.tolist()):
        sl = {n: inp[n][b:b + 1, :, :L].contiguous().to(dev)
              for n in ("q", "k", "v", "do")}
        o, lse = fa_fwd_ext(sl["q"], sl["k"], sl["v"], causal, scale, window)
        dq, dk, dv = fa_bwd_ext(sl["q"], sl["k"], sl["v"], o, lse, sl["do"],
                                causal, scale, window)
        assert fa_check_device_status(dev) == 0
        assert torch.equal(got["o"][b, :, :L], o[0].cpu()), b
        assert torch.equal(got["lse"][b, :, :L], lse[0].cpu()), b
        # one writer per element (H / Hkv <= 8): bit for bit
        assert torch.equal(got["dk"][b, :, :L], dk[0].cpu()), b
        assert torch.equal(got["dv"][b, :, :L], dv[0].cpu()), b
        # dQ sums key tiles through fp32 reductions in any order
        g, r = f64(got["dq"][b, :, :L]), f64(dq[0])
        assert np.linalg.norm(g - r) <= 1e-2 * max(np.linalg.norm(r), 1e-30)


def test_full_lengths_equal_the_grouped_call():
    B, H, Hkv, N, d = 2, 4, 2, 384, 128
    inp = make_grouped_inputs(B, H, Hkv, N, d, seed=8)
    lens = torch.full((B,), N, dtype=torch.int32)
    scale = default_scale(d)
    got = run_varlen(inp, lens, True, scale, -1)
    dev = torch.device("cuda:0")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa_fwd_ext(q, k, v, True, scale)
    dq, dk, dv = fa_bwd_ext(q, k, v, o, lse, do, True, scale)
    for name, r in (("o", o), ("lse", lse), ("dk", dk), ("dv", dv)):
        assert torch.equal(got[name], r.cpu()), name


def test_lengths_change_between_graph_replays():
    B, H, Hkv, N, d = 3, 4, 2, 400, 128
    dev = torch.device("cuda:0")
    inp = make_grouped_inputs(B, H, Hkv, N, d, seed=12)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    sl = torch.tensor([400, 200, 5], dtype=torch.int32, device=dev)
    o = torch.zeros_like(q)
    lse = torch.zeros((B, H, N), dtype=torch.float32, device=dev)
    grads = [torch.zeros_like(t) for t in (q, k, v)]
    ws = torch.empty(1 << 26, dtype=torch.uint8, device=dev)

    def step():
        fa_fwd_varlen(q, k, v, sl, True, scale, out=o, lse=lse)
        fa_bwd_varlen(q, k, v, o, lse, do, sl, True, scale, dq=grads[0],
                      dk=grads[1], dv=grads[2], workspace=ws)

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        step()                      # first use outside the capture
    torch.cuda.current_stream(dev).wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for new in ([130, 400, 0], [1, 2, 399]):
        sl.copy_(torch.tensor(new, dtype=torch.int32))
        o.fill_(SENTINEL)
        lse.fill_(SENTINEL)
        graph.replay()
        torch.cuda.synchronize(dev)
        assert fa_check_device_status(dev) == 0
        got = {"o": o.cpu(), "lse": lse.cpu(), "dq": grads[0].cpu(),
               "dk": grads[1].cpu(), "dv": grads[2].cpu()}
        lens = torch.tensor(new, dtype=torch.int32)
        check_rows(got, lens, inp, True, scale, -1, "replay %s" % new)
        check_grads(got, lens, inp, True, scale, -1, "replay %s" % new)


def test_full_size_whole_sequences():
    # 4 x 64 x 4096 x 128 causal, lengths from the first tile to the full N
    B, H, N, d = 4, 64, 4096, 128
    inp = make_grouped_inputs(B, H, H, N, d, seed=1004)
    lens = make_seq_lens(B, N, seed=5, fixed=[N, 2049, 1, 3000])
    scale = default_scale(d)
    got = run_varlen(inp, lens, True, scale, -1)
    pad = (torch.arange(N)[None, :] >= lens[:, None].long())
    for name in ("dq", "dk", "dv"):
        assert not got[name][pad[:, None, :].expand(B, H, N)].any(), name
    assert (got["o"][pad[:, None, :].expand(B, H, N)] == SENTINEL).all()
    for bh in sample_heads(B * H, 8, seed=3):
        b, h = divmod(bh, H)
        L = int(lens[b])
        one = {n: inp[n][b:b + 1, h:h + 1, :L] for n in ("q", "k", "v", "do")}
        o_ref, lse_ref = oracle.fwd_ext(one["q"], one["k"], one["v"], True,
                                        scale)
        o = f64(got["o"][b, h, :L])
        assert np.max(np.abs(o - o_ref[0, 0])) <= O_MAX_ABS, bh
        assert rel_fro(o, o_ref[0, 0]) <= O_REL_FRO, bh
        assert np.max(np.abs(f64(got["lse"][b, h, :L]) - lse_ref[0, 0])) \
            <= LSE_MAX_ABS, bh
        g_ref = oracle.bwd_ext(one["q"], one["k"], one["v"], one["do"], True,
                               scale)
        for name, r in zip(("dq", "dk", "dv"), g_ref):
            g = f64(got[name][b, h, :L])
            assert rel_fro(g, r[0, 0]) <= GRAD_REL_FRO, (bh, name)
