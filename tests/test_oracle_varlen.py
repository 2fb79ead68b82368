"""Pins of the oracle's per-sequence-length forward and backward (CPU only).

fwd_varlen / bwd_varlen restrict each batch entry to its first L_b rows by
slicing.  They are checked against a formulation that shares none of that
code: torch float64 autograd of a dense masked softmax over the whole padded
length, with the mask written from the definition (key j visible to query i
when both are below L_b, j <= i if causal, |i - j| <= window).  Padding
content must not matter, full lengths must give fwd_ext / bwd_ext exactly,
and an empty sequence must give no rows at all.
"""
import numpy as np
import pytest
import torch

import oracle


def dense_masked(q, k, v, dout, lens, causal, scale, window):
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    kr = kt.repeat_interleave(g, dim=1)
    vr = vt.repeat_interleave(g, dim=1)
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    o_all, lse_all, loss = [], [], 0.0
    for b in range(B):
        L = int(lens[b])
        vis = (i < L) & (j < L)
        if causal:
            vis &= j <= i
        if window >= 0:
            vis &= (i - j).abs() <= window
        s = scale * qt[b] @ kr[b].transpose(-1, -2)
        s = s.masked_fill(~vis, float("-inf"))
        rows = vis.any(dim=1)                     # real query rows
        lse = torch.logsumexp(s[:, rows], dim=-1)
        p = torch.exp(s[:, rows] - lse[..., None])
        o = p @ vr[b]
        loss = loss + (o * torch.tensor(dout[b][:, rows.numpy()])).sum()
        o_all.append((o, rows))
        lse_all.append(lse)
    loss.backward()
    return o_all, lse_all, qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


CASES = [
    # B, H, Hkv, N, d, causal, window, lengths
    (3, 2, 1, 9, 4, True, -1, [9, 4, 1]),
    (3, 4, 2, 11, 3, False, -1, [0, 11, 6]),
    (2, 2, 2, 13, 5, False, 3, [13, 7]),
    (2, 3, 1, 10, 4, True, 2, [5, 10]),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,window,lens", CASES)
def test_varlen_matches_dense_masked_autograd(B, H, Hkv, N, d, causal, window,
                                              lens):
    rng = np.random.default_rng(B * 100 + N)
    q = rng.normal(size=(B, H, N, d))
    k = rng.normal(size=(B, Hkv, N, d))
    v = rng.normal(size=(B, Hkv, N, d))
    dout = rng.normal(size=(B, H, N, d))
    scale = 0.7
    o, lse = oracle.fwd_varlen(q, k, v, lens, causal, scale, window)
    dq, dk, dv = oracle.bwd_varlen(q, k, v, dout, lens, causal, scale, window)
    o_ref, lse_ref, dq_ref, dk_ref, dv_ref = dense_masked(
        q, k, v, dout, lens, causal, scale, window)
    for b in range(B):
        ob, rows = o_ref[b]
        rows = rows.numpy()
        assert np.allclose(o[b][:, rows], ob.detach().numpy(), atol=1e-12)
        assert np.allclose(lse[b][:, rows], lse_ref[b].detach().numpy(),
                           atol=1e-12)
        assert np.isnan(o[b][:, ~rows]).all() and np.isnan(lse[b][:, ~rows]).all()
    for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert np.allclose(got, ref, atol=1e-11)


def test_padding_content_does_not_matter():
    rng = np.random.default_rng(21)
    B, H, Hkv, N, d, lens = 3, 4, 2, 12, 4, [12, 5, 0]
    q, dout = rng.normal(size=(2, B, H, N, d))
    k, v = rng.normal(size=(2, B, Hkv, N, d))
    a = oracle.fwd_varlen(q, k, v, lens, True, 0.5)
    ga = oracle.bwd_varlen(q, k, v, dout, lens, True, 0.5)
    q2, k2, v2, d2 = q.copy(), k.copy(), v.copy(), dout.copy()
    for b, L in enumerate(lens):
        for t in (q2, k2, v2, d2):
            t[b, :, L:] = rng.normal(size=t[b, :, L:].shape) * 100
    b_ = oracle.fwd_varlen(q2, k2, v2, lens, True, 0.5)
    gb = oracle.bwd_varlen(q2, k2, v2, d2, lens, True, 0.5)
    assert np.array_equal(a[0], b_[0], equal_nan=True)
    assert np.array_equal(a[1], b_[1], equal_nan=True)
    for x, y in zip(ga, gb):
        assert np.array_equal(x, y)
    # gradients of padding rows are zero; an empty sequence has no outputs
    assert not ga[0][1, :, 5:].any() and not ga[1][2].any()
    assert np.isnan(a[0][2]).all()


def test_full_lengths_are_the_grouped_operation():
    rng = np.random.default_rng(5)
    q, dout = rng.normal(size=(2, 2, 4, 20, 8))
    k, v = rng.normal(size=(2, 2, 2, 20, 8))
    lens = [20, 20]
    for causal, window in ((True, -1), (False, 6)):
        o, lse = oracle.fwd_varlen(q, k, v, lens, causal, 0.3, window)
        o2, lse2 = oracle.fwd_ext(q, k, v, causal, 0.3, window)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
        g = oracle.bwd_varlen(q, k, v, dout, lens, causal, 0.3, window)
        g2 = oracle.bwd_ext(q, k, v, dout, causal, 0.3, window)
        for x, y in zip(g, g2):
            assert np.array_equal(x, y)


def test_lengths_are_clamped_and_checked():
    rng = np.random.default_rng(9)
    q = rng.normal(size=(2, 1, 6, 4))
    o1, _ = oracle.fwd_varlen(q, q, q, [-3, 99], False, 1.0)
    o2, _ = oracle.fwd_varlen(q, q, q, [0, 6], False, 1.0)
    assert np.array_equal(o1, o2, equal_nan=True)
    with pytest.raises(ValueError):
        oracle.fwd_varlen(q, q, q, [1], False, 1.0)
