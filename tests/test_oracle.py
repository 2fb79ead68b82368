"""Pins for the CPU fp64 oracle (CPU only).

The oracle is checked against things other than itself:
  * torch fp64 softmax + autograd (an independent library routine),
  * central finite differences of L = sum(O * dO) (derivative consistency),
  * a hand-derived worked example (tests/golden/closed_form_three_keys.txt),
  * closed forms and invariants of softmax attention.
Each is chosen so that a plausible slip in the oracle (a dropped scale, a
dropped D term, a transposed operand, a causal mask pointing the wrong way,
a wrong LSE base) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, mult=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape) * mult


def _torch_reference(q, k, v, do, causal, scale):
    """softmax(scale QK^T + mask) V and its autograd gradients, in fp64."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True)
                  for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        n = s.shape[-1]
        above = torch.ones(n, n, dtype=torch.bool).triu(1)
        s = s.masked_fill(above, float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = p @ tv
    lse = torch.logsumexp(s, dim=-1)
    o.backward(torch.tensor(do, dtype=torch.float64))
    return (o.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(),
            tk.grad.numpy(), tv.grad.numpy())


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 8), (2, 2, 37, 8),
                                     (1, 2, 128, 64), (2, 1, 256, 8),
                                     (1, 1, 200, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_autograd(B, H, N, d, causal):
    shape = (B, H, N, d)
    q, k, v, do = (_rand(shape, s) for s in (1, 2, 3, 4))
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref, dq_ref, dk_ref, dv_ref = _torch_reference(
        q, k, v, do, causal, scale)
    o, lse = oracle.fwd(q, k, v, causal, scale)
    dq, dk, dv = oracle.bwd(q, k, v, do, causal, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(dq, dq_ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(dk, dk_ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(dv, dv_ref, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("d", [2, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(N, d, causal):
    shape = (1, 1, N, d)
    q, k, v, do = (_rand(shape, 10 + s) for s in range(4))
    scale = 0.7

    def loss(qq, kk, vv):
        o, _ = oracle.fwd(qq, kk, vv, causal, scale)
        return float(np.sum(o * do))

    grads = oracle.bwd(q, k, v, do, causal, scale)
    h = 1e-6
    for which, g in zip(range(3), grads):
        fd = np.zeros(shape)
        for idx in np.ndindex(*shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.linalg.norm(g - fd) / max(np.linalg.norm(fd), 1e-12)
        assert err < 1e-6 or np.max(np.abs(g - fd)) < 1e-8, (which, err)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, expr = line.split(":", 1)
            env = {"__builtins__": {}, "ln": math.log}
            vals[key.strip()] = np.array(
                [eval(e, env) for e in expr.split(",")], dtype=np.float64)
    return vals


@pytest.mark.parametrize("causal", [False, True])
def test_hand_derived_worked_example(causal):
    g = _read_golden("closed_form_three_keys.txt")
    shape = (1, 1, 3, 1)
    q, k, v, do = (g[n].reshape(shape) for n in ("q", "k", "v", "do"))
    scale = float(g["scale"][0])
    tag = "causal" if causal else "noncausal"
    o, lse = oracle.fwd(q, k, v, causal, scale)
    dq, dk, dv = oracle.bwd(q, k, v, do, causal, scale)
    np.testing.assert_allclose(o.ravel(), g[tag + ".o"], atol=1e-14)
    np.testing.assert_allclose(lse.ravel(), g[tag + ".lse"], atol=1e-14)
    np.testing.assert_allclose(dq.ravel(), g[tag + ".dq"], atol=1e-14)
    np.testing.assert_allclose(dk.ravel(), g[tag + ".dk"], atol=1e-14)
    np.testing.assert_allclose(dv.ravel(), g[tag + ".dv"], atol=1e-14)


@pytest.mark.parametrize("tile", [1, 3, 7, 64, 300])
@pytest.mark.parametrize("tau", [0.0, 8.0 * math.log(2.0)])
@pytest.mark.parametrize("causal", [False, True])
def test_online_update_equals_two_pass(tile, tau, causal):
    shape = (1, 2, 300, 16)
    # Sharp scores (x4) so the running max moves and rescales happen.
    q, k = _rand(shape, 21, 4.0), _rand(shape, 22, 4.0)
    v = _rand(shape, 23)
    o2, lse2 = oracle.fwd(q, k, v, causal, 0.25)
    o1, lse1 = oracle.fwd_online(q, k, v, causal, 0.25, tile=tile, tau=tau)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse1, lse2, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    # With V = identity (d = N), O is the probability matrix P itself.
    N = 24
    q, k = _rand((1, 1, N, N), 31), _rand((1, 1, N, N), 32)
    v = np.eye(N).reshape(1, 1, N, N)
    p, _ = oracle.fwd(q, k, v, causal, 0.3)
    p = p[0, 0]
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    if causal:
        assert np.all(np.triu(p, 1) == 0.0)
        assert np.all(np.diag(p) > 0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_value_rows_give_that_row(causal):
    shape = (2, 1, 50, 8)
    q, k = _rand(shape, 41), _rand(shape, 42)
    c = _rand((8,), 43)
    v = np.broadcast_to(c, shape).copy()
    o, _ = oracle.fwd(q, k, v, causal, 0.4)
    np.testing.assert_allclose(o, np.broadcast_to(c, shape), atol=1e-13)


def test_first_causal_row():
    shape = (1, 3, 40, 8)
    q, k, v = _rand(shape, 51), _rand(shape, 52), _rand(shape, 53)
    scale = 0.37
    o, lse = oracle.fwd(q, k, v, True, scale)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-15)
    np.testing.assert_allclose(
        lse[:, :, 0], scale * np.sum(q[:, :, 0] * k[:, :, 0], -1), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_lse_is_logsumexp_of_scores(causal):
    shape = (1, 2, 64, 16)
    q, k, v = _rand(shape, 61, 2.0), _rand(shape, 62, 2.0), _rand(shape, 63)
    scale = 0.25
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if causal:
        s = np.where(np.triu(np.ones((64, 64), bool), 1), -np.inf, s)
    _, lse = oracle.fwd(q, k, v, causal, scale)
    np.testing.assert_allclose(lse, logsumexp(s, axis=-1), rtol=1e-13,
                               atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_uniform_weights(causal):
    N, d = 30, 4
    q = np.zeros((1, 1, N, d))
    k, v = _rand((1, 1, N, d), 71), _rand((1, 1, N, d), 72)
    o, lse = oracle.fwd(q, k, v, causal, 0.5)
    if causal:
        counts = np.arange(1, N + 1)
        expect_o = np.cumsum(v[0, 0], axis=0) / counts[:, None]
        expect_lse = np.log(counts)
    else:
        expect_o = np.broadcast_to(v[0, 0].mean(axis=0), (N, d))
        expect_lse = np.full(N, math.log(N))
    np.testing.assert_allclose(o[0, 0], expect_o, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], expect_lse, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_adding_a_vector_to_every_key_leaves_output_unchanged(causal):
    shape = (1, 2, 45, 8)
    q, k, v = _rand(shape, 81), _rand(shape, 82), _rand(shape, 83)
    shift = _rand((8,), 84, 3.0)
    o1, _ = oracle.fwd(q, k, v, causal, 0.4)
    o2, _ = oracle.fwd(q, k + shift, v, causal, 0.4)
    np.testing.assert_allclose(o1, o2, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    shape = (2, 2, 70, 8)
    q, k, v, do = (_rand(shape, 90 + s) for s in range(4))
    dq, dk, dv = oracle.bwd(q, k, v, do, causal, 0.35)
    # Rows of P sum to one  =>  sum_j dV_j = sum_i dO_i.
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)
    # sum_j dS_ij = 0 for every row  =>  sum_j dK_j = 0.
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # Identical key rows  =>  dQ = 0.
    k_same = np.broadcast_to(k[:, :, :1], shape).copy()
    dq2, _, _ = oracle.bwd(q, k_same, v, do, causal, 0.35)
    np.testing.assert_allclose(dq2, 0.0, atol=1e-13)


def test_thread_count_is_reported():
    assert oracle.num_threads() >= 1


@pytest.mark.parametrize("causal", [False, True])
def test_row_ranges_agree_with_full_computation(causal):
    shape = (1, 2, 90, 8)
    q, k, v, do = (_rand(shape, 110 + s) for s in range(4))
    o, lse = oracle.fwd(q, k, v, causal, 0.3)
    dq, dk, dv = oracle.bwd(q, k, v, do, causal, 0.3)
    parts = [(0, 17), (17, 60), (60, 90)]
    sum_dk = np.zeros(shape)
    sum_dv = np.zeros(shape)
    for r0, r1 in parts:
        o_r, lse_r = oracle.fwd_rows(q, k, v, causal, 0.3, r0, r1)
        np.testing.assert_allclose(o_r[:, :, r0:r1], o[:, :, r0:r1], atol=1e-15)
        np.testing.assert_allclose(lse_r[:, :, r0:r1], lse[:, :, r0:r1], atol=1e-15)
        assert np.isnan(o_r[:, :, :r0]).all() and np.isnan(o_r[:, :, r1:]).all()
        dq_r, dk_r, dv_r = oracle.bwd_rows(q, k, v, do, causal, 0.3, r0, r1)
        np.testing.assert_allclose(dq_r[:, :, r0:r1], dq[:, :, r0:r1], atol=1e-14)
        assert np.all(dq_r[:, :, :r0] == 0) and np.all(dq_r[:, :, r1:] == 0)
        sum_dk += dk_r
        sum_dv += dv_r
    # Contributions of disjoint row ranges add up to the full gradients.
    np.testing.assert_allclose(sum_dk, dk, atol=1e-13)
    np.testing.assert_allclose(sum_dv, dv, atol=1e-13)
    if causal:
        # Keys j >= r0 are seen only by rows i >= r0.
        _, dk_t, dv_t = oracle.bwd_rows(q, k, v, do, True, 0.3, 60, 90)
        np.testing.assert_allclose(dk_t[:, :, 60:], dk[:, :, 60:], atol=1e-14)
        np.testing.assert_allclose(dv_t[:, :, 60:], dv[:, :, 60:], atol=1e-14)


# ---------------------------------------------- grouped heads, sliding window
def _torch_reference_ext(q, k, v, do, causal, scale, window):
    """Grouped / windowed attention with torch fp64 autograd: K/V heads are
    repeated to the query heads (so autograd sums dK/dV over each group) and
    the band is an explicit mask."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True)
                  for x in (q, k, v))
    group = q.shape[1] // k.shape[1]
    kk = tk.repeat_interleave(group, dim=1)
    vv = tv.repeat_interleave(group, dim=1)
    s = scale * tq @ kk.transpose(-1, -2)
    n = s.shape[-1]
    i = torch.arange(n)[:, None]
    j = torch.arange(n)[None, :]
    hidden = torch.zeros(n, n, dtype=torch.bool)
    if causal:
        hidden |= j > i
    if window >= 0:
        hidden |= (i - j) > window
        if not causal:
            hidden |= (j - i) > window
    s = s.masked_fill(hidden, float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = p @ vv
    lse = torch.logsumexp(s, dim=-1)
    o.backward(torch.tensor(do, dtype=torch.float64))
    return (o.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(),
            tk.grad.numpy(), tv.grad.numpy())


@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (6, 1)])
@pytest.mark.parametrize("window", [-1, 0, 3, 40])
@pytest.mark.parametrize("causal", [False, True])
def test_ext_matches_torch_autograd(H, Hkv, window, causal):
    B, N, d = 2, 37, 8
    q, do = _rand((B, H, N, d), 201), _rand((B, H, N, d), 202)
    k, v = _rand((B, Hkv, N, d), 203), _rand((B, Hkv, N, d), 204)
    ref = _torch_reference_ext(q, k, v, do, causal, 0.4, window)
    o, lse = oracle.fwd_ext(q, k, v, causal, 0.4, window=window)
    grads = oracle.bwd_ext(q, k, v, do, causal, 0.4, window=window)
    for got, want in zip((o, lse) + grads, ref):
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("window", [0, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_ext_gradients_match_finite_differences(window, causal):
    B, H, Hkv, N, d = 1, 2, 1, 6, 3
    q, do = _rand((B, H, N, d), 211), _rand((B, H, N, d), 212)
    k, v = _rand((B, Hkv, N, d), 213), _rand((B, Hkv, N, d), 214)

    def loss(qq, kk, vv):
        o, _ = oracle.fwd_ext(qq, kk, vv, causal, 0.6, window=window)
        return float(np.sum(o * do))

    grads = oracle.bwd_ext(q, k, v, do, causal, 0.6, window=window)
    h = 1e-6
    for which, g in zip(range(3), grads):
        args = [q, k, v]
        fd = np.zeros(args[which].shape)
        for idx in np.ndindex(*fd.shape):
            ap = [a.copy() for a in args]
            am = [a.copy() for a in args]
            ap[which][idx] += h
            am[which][idx] -= h
            fd[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        err = np.linalg.norm(g - fd) / max(np.linalg.norm(fd), 1e-12)
        assert err < 1e-6 or np.max(np.abs(g - fd)) < 1e-8, (which, err)


@pytest.mark.parametrize("causal", [False, True])
def test_ext_without_groups_or_window_is_the_base_operation(causal):
    shape = (2, 3, 50, 8)
    q, k, v, do = (_rand(shape, 220 + s) for s in range(4))
    o1, l1 = oracle.fwd(q, k, v, causal, 0.3)
    o2, l2 = oracle.fwd_ext(q, k, v, causal, 0.3, window=-1)
    o3, l3 = oracle.fwd_ext(q, k, v, causal, 0.3, window=50)  # window >= N
    np.testing.assert_allclose(o2, o1, atol=1e-15)
    np.testing.assert_allclose(l2, l1, atol=1e-15)
    np.testing.assert_allclose(o3, o1, atol=1e-15)
    g1 = oracle.bwd(q, k, v, do, causal, 0.3)
    g2 = oracle.bwd_ext(q, k, v, do, causal, 0.3, window=-1)
    for a, b in zip(g2, g1):
        np.testing.assert_allclose(a, b, atol=1e-14)


def test_causal_window_zero_sees_only_the_diagonal():
    shape = (1, 2, 20, 8)
    q, k, v = _rand(shape, 231), _rand(shape, 232), _rand(shape, 233)
    o, lse = oracle.fwd_ext(q, k, v, True, 0.5, window=0)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.5 * np.sum(q * k, -1), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_window_band_of_the_probability_matrix(causal):
    # V = identity makes O the probability matrix: zero outside the band,
    # rows summing to one.
    N, w = 24, 5
    q, k = _rand((1, 1, N, N), 241), _rand((1, 1, N, N), 242)
    v = np.eye(N).reshape(1, 1, N, N)
    p, _ = oracle.fwd_ext(q, k, v, causal, 0.3, window=w)
    p = p[0, 0]
    i, j = np.indices((N, N))
    outside = (i - j > w) | ((j - i > w) if not causal else (j > i))
    assert np.all(p[outside] == 0.0)
    assert np.all(p[~outside] > 0.0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads_equal_repeated_heads(causal):
    # Hkv < H equals the plain operation on K/V repeated per query head,
    # with dK/dV summed over each group (no torch involved).
    B, H, Hkv, N, d = 2, 6, 2, 30, 8
    q, do = _rand((B, H, N, d), 251), _rand((B, H, N, d), 252)
    k, v = _rand((B, Hkv, N, d), 253), _rand((B, Hkv, N, d), 254)
    kr, vr = np.repeat(k, H // Hkv, axis=1), np.repeat(v, H // Hkv, axis=1)
    o1, l1 = oracle.fwd_ext(q, k, v, causal, 0.3, window=7)
    o2, l2 = oracle.fwd_ext(q, kr, vr, causal, 0.3, window=7)
    np.testing.assert_allclose(o1, o2, atol=1e-15)
    np.testing.assert_allclose(l1, l2, atol=1e-15)
    dq1, dk1, dv1 = oracle.bwd_ext(q, k, v, do, causal, 0.3, window=7)
    dq2, dk2, dv2 = oracle.bwd_ext(q, kr, vr, do, causal, 0.3, window=7)
    np.testing.assert_allclose(dq1, dq2, atol=1e-14)
    g = H // Hkv
    np.testing.assert_allclose(dk1, dk2.reshape(B, Hkv, g, N, d).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv1, dv2.reshape(B, Hkv, g, N, d).sum(2), atol=1e-13)


def test_ext_row_ranges():
    B, H, Hkv, N, d = 1, 4, 2, 40, 8
    q, do = _rand((B, H, N, d), 261), _rand((B, H, N, d), 262)
    k, v = _rand((B, Hkv, N, d), 263), _rand((B, Hkv, N, d), 264)
    o, lse = oracle.fwd_ext(q, k, v, True, 0.3, window=9)
    o_r, lse_r = oracle.fwd_ext(q, k, v, True, 0.3, window=9, r0=10, r1=25)
    np.testing.assert_allclose(o_r[:, :, 10:25], o[:, :, 10:25], atol=1e-15)
    assert np.isnan(o_r[:, :, :10]).all() and np.isnan(lse_r[:, :, 25:]).all()
    dq, dk, dv = oracle.bwd_ext(q, k, v, do, True, 0.3, window=9)
    a = oracle.bwd_ext(q, k, v, do, True, 0.3, window=9, r0=0, r1=20)
    b = oracle.bwd_ext(q, k, v, do, True, 0.3, window=9, r0=20, r1=40)
    np.testing.assert_allclose(a[0] + b[0], dq, atol=1e-14)
    np.testing.assert_allclose(a[1] + b[1], dk, atol=1e-13)
    np.testing.assert_allclose(a[2] + b[2], dv, atol=1e-13)
