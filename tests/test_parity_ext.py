"""GPU parity of the grouped-head and sliding-window entry points.

fa_fwd_ext / fa_bwd_ext (query heads sharing Hkv key/value heads; keys
limited to |i - j| <= window) against the CPU fp64 oracle's fwd_ext /
bwd_ext on the same seeded bf16 inputs, with the tolerances of the base
operation (O max-abs 2e-2 and rel-Frobenius 1e-2, LSE max-abs 1e-3, each
gradient rel-Frobenius 5e-2).  Small shapes are compared element by element;
full-size shapes on whole key/value groups, every row.  Identities: Hkv = H
with no window is the base operation bit for bit; a window of N - 1 or more
is no window; grouped heads equal repeated heads.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_bwd_gb300 import (fa_bwd, fa_bwd_ext,
                                       fa_check_device_status, fa_fwd,
                                       fa_fwd_ext)
from tiled_attention_bwd_gb300.workloads import (default_scale,
                                                 make_grouped_inputs)

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_FRO, LSE_MAX_ABS, GRAD_REL_FRO = 2e-2, 1e-2, 1e-3, 5e-2


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def f64(t):
    return t.detach().to("cpu").double().numpy()


def run_ext(inp, causal, scale, window, backward=True):
    dev = torch.device("cuda:0")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa_fwd_ext(q, k, v, causal, scale, window)
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv = fa_bwd_ext(q, k, v, o, lse, do, causal, scale, window)
        out.update(dq=dq, dk=dk, dv=dv)
    assert fa_check_device_status(dev) == 0
    return {k_: v_.cpu() for k_, v_ in out.items()}


def check_forward(o, lse, o_ref, lse_ref, tag):
    o, lse = f64(o), f64(lse)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), tag
    err = np.max(np.abs(o - o_ref))
    assert err <= O_MAX_ABS, "%s O max-abs %.3g" % (tag, err)
    rf = rel_fro(o, o_ref)
    assert rf <= O_REL_FRO, "%s O rel-Frobenius %.3g" % (tag, rf)
    le = np.max(np.abs(lse - lse_ref))
    assert le <= LSE_MAX_ABS, "%s LSE max-abs %.3g" % (tag, le)


def check_grad(name, g, r, tag):
    g = f64(g) if isinstance(g, torch.Tensor) else g
    assert np.isfinite(g).all(), "%s %s not finite" % (tag, name)
    rf = rel_fro(g, r)
    assert rf <= GRAD_REL_FRO, "%s %s rel-Frobenius %.3g" % (tag, name, rf)


SMALL = [
    # B, H, Hkv, N, d, causal, window
    (1, 4, 1, 256, 128, False, -1),      # multi-query
    (1, 4, 1, 256, 128, True, -1),
    (2, 8, 2, 384, 64, True, -1),        # grouped, odd tile count
    (1, 6, 3, 333, 128, False, -1),      # grouped, ragged
    (1, 2, 2, 512, 128, True, 0),        # diagonal only
    (1, 2, 2, 512, 128, False, 0),
    (1, 2, 1, 640, 128, True, 100),      # window not a tile multiple
    (1, 2, 2, 640, 64, False, 100),
    (1, 2, 2, 600, 128, False, 128),     # window = one tile, ragged N
    (1, 2, 2, 600, 128, True, 128),
    (2, 4, 2, 1000, 128, True, 300),     # grouped + window + ragged
    (1, 4, 4, 1000, 128, False, 257),
    (1, 2, 1, 777, 64, True, 1),
    (1, 3, 1, 17, 64, False, 3),         # one partial tile
    (1, 2, 1, 1, 128, True, 0),          # N = 1
    (1, 4, 2, 1280, 128, False, 700),    # band wider than several tiles
    # more than 8 query heads per K/V head: split over blocks, dK/dV summed
    # in fp32 workspace
    (1, 16, 1, 384, 128, True, -1),
    (1, 12, 1, 333, 64, False, 100),
    (2, 32, 2, 256, 128, False, -1),
    (1, 24, 2, 517, 128, True, 200),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,window", SMALL)
def test_small_every_element(B, H, Hkv, N, d, causal, window):
    inp = make_grouped_inputs(B, H, Hkv, N, d, seed=31 + N + d + H + Hkv)
    scale = default_scale(d)
    got = run_ext(inp, causal, scale, window)
    o_ref, lse_ref = oracle.fwd_ext(inp["q"], inp["k"], inp["v"], causal,
                                    scale, window)
    dq, dk, dv = oracle.bwd_ext(inp["q"], inp["k"], inp["v"], inp["do"],
                                causal, scale, window)
    tag = "%dx%d/%dx%dx%d causal=%d w=%d" % (B, H, Hkv, N, d, causal, window)
    check_forward(got["o"], got["lse"], o_ref, lse_ref, tag)
    for name, g, r in (("dq", got["dq"], dq), ("dk", got["dk"], dk),
                       ("dv", got["dv"], dv)):
        check_grad(name, g, r, tag)


def test_sharp_scores_with_window():
    # Large scores: the running max jumps across tiles inside the band and
    # rows start with fully masked tiles.
    inp = make_grouped_inputs(1, 4, 2, 768, 128, seed=77, qk_mult=4.0)
    scale = default_scale(128)
    for causal, window in ((True, 200), (False, 150)):
        got = run_ext(inp, causal, scale, window)
        o_ref, lse_ref = oracle.fwd_ext(inp["q"], inp["k"], inp["v"], causal,
                                        scale, window)
        refs = oracle.bwd_ext(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                              scale, window)
        check_forward(got["o"], got["lse"], o_ref, lse_ref, "sharp")
        for name, r in zip(("dq", "dk", "dv"), refs):
            check_grad(name, got[name], r, "sharp")


def test_defaults_are_the_base_operation_bit_for_bit():
    dev = torch.device("cuda:0")
    inp = make_grouped_inputs(2, 3, 3, 500, 128, seed=5)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    for causal in (False, True):
        o1, l1 = fa_fwd(q, k, v, causal, 0.09)
        o2, l2 = fa_fwd_ext(q, k, v, causal, 0.09, -1)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        # A window that hides nothing is no window.
        for w in (499, 500, 10 ** 6):
            o3, l3 = fa_fwd_ext(q, k, v, causal, 0.09, w)
            assert torch.equal(o1, o3) and torch.equal(l1, l3)
        g1 = fa_bwd(q, k, v, o1, l1, do, causal, 0.09)
        g2 = fa_bwd_ext(q, k, v, o1, l1, do, causal, 0.09, -1)
        # dK, dV have one writer per element: identical; dQ sums key tiles
        # in any order through fp32 reduce-adds.
        assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
        assert rel_fro(f64(g1[0]), f64(g2[0])) <= 1e-2
    assert fa_check_device_status(dev) == 0


@pytest.mark.parametrize("causal,window", [(True, -1), (False, 200)])
def test_grouped_equals_repeated_heads(causal, window):
    dev = torch.device("cuda:0")
    B, H, Hkv, N, d = 2, 8, 2, 640, 128
    inp = make_grouped_inputs(B, H, Hkv, N, d, seed=17)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    g = H // Hkv
    kr = k.repeat_interleave(g, dim=1).contiguous()
    vr = v.repeat_interleave(g, dim=1).contiguous()
    scale = default_scale(d)
    o1, l1 = fa_fwd_ext(q, k, v, causal, scale, window)
    o2, l2 = fa_fwd_ext(q, kr, vr, causal, scale, window)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    dq1, dk1, dv1 = fa_bwd_ext(q, k, v, o1, l1, do, causal, scale, window)
    dq2, dk2, dv2 = fa_bwd_ext(q, kr, vr, o2, l2, do, causal, scale, window)
    assert rel_fro(f64(dq1), f64(dq2)) <= 1e-2
    dk_sum = f64(dk2).reshape(B, Hkv, g, N, d).sum(axis=2)
    dv_sum = f64(dv2).reshape(B, Hkv, g, N, d).sum(axis=2)
    assert rel_fro(f64(dk1), dk_sum) <= 1e-2
    assert rel_fro(f64(dv1), dv_sum) <= 1e-2
    assert fa_check_device_status(dev) == 0


# ------------------------------------------------ full-size shapes
FULL = [
    # name, B, H, Hkv, N, d, causal, window
    ("xl_gqa8", 4, 64, 8, 4096, 128, True, -1),
    ("xl_mqa", 4, 64, 1, 4096, 128, True, -1),
    ("xl_window1024", 4, 64, 64, 4096, 128, True, 1024),
    ("long_window4096", 1, 16, 16, 16384, 128, True, 4096),
    ("medium_gqa4_window300_noncausal", 4, 32, 8, 1024, 128, False, 300),
]


@pytest.mark.parametrize("name,B,H,Hkv,N,d,causal,window", FULL)
def test_full_size_whole_groups(name, B, H, Hkv, N, d, causal, window):
    inp = make_grouped_inputs(B, H, Hkv, N, d, seed=2001 + H + Hkv + N)
    scale = default_scale(d)
    got = run_ext(inp, causal, scale, window)
    g = H // Hkv
    # Whole key/value groups (a K/V head with every query head that reads
    # it), all rows: the first group of the first batch entry and the last
    # group of the last one (only the last when a group holds more than 16
    # query heads: multi-query groups are whole batch entries).  O, LSE and
    # dQ are per query head; dK and dV are the group's sums, so only a whole
    # group gives them exactly.
    groups = {(B - 1, Hkv - 1)} if g > 16 else {(0, 0), (B - 1, Hkv - 1)}
    for b, kvh in sorted(groups):
        hs = slice(kvh * g, (kvh + 1) * g)
        sub = {"q": inp["q"][b:b + 1, hs], "do": inp["do"][b:b + 1, hs],
               "k": inp["k"][b:b + 1, kvh:kvh + 1],
               "v": inp["v"][b:b + 1, kvh:kvh + 1]}
        tag = "%s b=%d kvh=%d" % (name, b, kvh)
        o_ref, lse_ref = oracle.fwd_ext(sub["q"], sub["k"], sub["v"], causal,
                                        scale, window)
        check_forward(got["o"][b:b + 1, hs], got["lse"][b:b + 1, hs], o_ref,
                      lse_ref, tag)
        del o_ref, lse_ref
        dq, dk, dv = oracle.bwd_ext(sub["q"], sub["k"], sub["v"], sub["do"],
                                    causal, scale, window)
        check_grad("dq", got["dq"][b:b + 1, hs], dq, tag)
        check_grad("dk", got["dk"][b:b + 1, kvh:kvh + 1], dk, tag)
        check_grad("dv", got["dv"][b:b + 1, kvh:kvh + 1], dv, tag)
