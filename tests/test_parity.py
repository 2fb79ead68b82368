"""GPU parity: libfa.so (through its C ABI) against the CPU fp64 oracle.

Both sides consume the same seeded bf16 inputs.  Tolerances (the bar the
kernels are held to, bf16 outputs against an exact fp64 result):
  O      : max-abs <= 2e-2 and relative Frobenius <= 1e-2
  LSE    : max-abs <= 1e-3 (natural log)
  dQ/dK/dV: relative Frobenius <= 5e-2 each
Small shapes are compared element by element on every head; the five
benchmark workloads run at full size in the launch configuration the
benchmark times, and are compared on whole heads (every head of the two
smaller ones; the first, the last and a seeded sample of the others).
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_bwd_gb300 import (fa_bwd, fa_check_device_status, fa_fwd)
from tiled_attention_bwd_gb300.workloads import (WORKLOADS, default_scale,
                                                 make_inputs, sample_heads,
                                                 workload_inputs)

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_FRO, LSE_MAX_ABS, GRAD_REL_FRO = 2e-2, 1e-2, 1e-3, 5e-2


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def f64(t):
    return t.detach().to("cpu").double().numpy()


def run_gpu(inp, causal, scale, backward=True):
    dev = torch.device("cuda:0")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa_fwd(q, k, v, causal, scale)
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal, scale)
        out.update(dq=dq, dk=dk, dv=dv)
    assert fa_check_device_status(dev) == 0
    return {k_: v_.cpu() for k_, v_ in out.items()}


def heads_of(t, heads):
    B, H = t.shape[0], t.shape[1]
    flat = t.reshape(B * H, *t.shape[2:])
    return flat[heads]


def check_forward(o_gpu, lse_gpu, o_ref, lse_ref, tag=""):
    o_gpu, lse_gpu = f64(o_gpu), f64(lse_gpu)
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), tag
    err = np.max(np.abs(o_gpu - o_ref))
    assert err <= O_MAX_ABS, "%s O max-abs %.3g" % (tag, err)
    rf = rel_fro(o_gpu, o_ref)
    assert rf <= O_REL_FRO, "%s O rel-Frobenius %.3g" % (tag, rf)
    le = np.max(np.abs(lse_gpu - lse_ref))
    assert le <= LSE_MAX_ABS, "%s LSE max-abs %.3g" % (tag, le)


def check_grads(got, ref, tag=""):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = f64(g)
        assert np.isfinite(g).all(), "%s %s not finite" % (tag, name)
        rf = rel_fro(g, r)
        assert rf <= GRAD_REL_FRO, "%s %s rel-Frobenius %.3g" % (tag, name, rf)


SMALL = [
    # B, H, N, d, causal
    (1, 1, 128, 128, False), (1, 1, 128, 128, True),
    (1, 1, 128, 64, False), (1, 1, 128, 64, True),
    (1, 2, 256, 128, False), (1, 2, 256, 128, True),
    (2, 1, 384, 64, False), (2, 1, 384, 64, True),      # odd tile count
    (3, 5, 640, 128, True), (2, 3, 512, 128, False),
    # ragged lengths: tiles past N are masked / zero-filled
    (1, 1, 1, 128, False), (1, 1, 1, 64, True),
    (1, 2, 17, 128, True), (1, 2, 17, 64, False),
    (2, 1, 100, 128, False), (1, 1, 200, 64, True),
    (1, 3, 333, 128, True), (2, 2, 333, 128, False),
    (1, 1, 1000, 64, True),
    # With fewer pairs of Q tiles than SMs (every case above) the forward's
    # work items are single Q tiles; these have more, so they run the pair
    # items, with a ragged last tile.
    (2, 80, 333, 128, True), (2, 80, 200, 64, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_small_shapes_every_element(B, H, N, d, causal):
    inp = make_inputs(B, H, N, d, seed=7 + N + d + B * 10 + H)
    scale = default_scale(d)
    got = run_gpu(inp, causal, scale)
    o_ref, lse_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], causal, scale)
    refs = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], causal, scale)
    tag = "%dx%dx%dx%d causal=%d" % (B, H, N, d, causal)
    check_forward(got["o"], got["lse"], o_ref, lse_ref, tag)
    check_grads((got["dq"], got["dk"], got["dv"]), refs, tag)


def test_sharp_scores_exercise_lazy_rescaling():
    # Large scores make the running max jump by far more than 2^8 across
    # tiles, so the O rescale path runs.
    inp = make_inputs(1, 2, 512, 128, seed=99, qk_mult=4.0)
    scale = default_scale(128)
    for causal in (False, True):
        got = run_gpu(inp, causal, scale)
        o_ref, lse_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], causal, scale)
        refs = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                          scale)
        check_forward(got["o"], got["lse"], o_ref, lse_ref, "sharp")
        check_grads((got["dq"], got["dk"], got["dv"]), refs, "sharp")


def test_forward_is_deterministic():
    inp = make_inputs(2, 2, 384, 128, seed=5)
    a = run_gpu(inp, True, 0.1, backward=False)
    b = run_gpu(inp, True, 0.1, backward=False)
    assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"])


@pytest.mark.parametrize("d", [128, 64])
def test_output_only_16_byte_aligned(d):
    # O rows leave in 32-byte stores when O is 32-byte aligned, else in
    # 16-byte ones (the boundary asks for 16): both give the same bits.
    dev = torch.device("cuda:0")
    B, H, N, causal = 1, 3, 333, True
    scale = default_scale(d)
    inp = make_inputs(B, H, N, d, seed=37)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    n = q.numel()
    buf = torch.empty(n + 8, dtype=torch.bfloat16, device=dev)
    o16 = buf[8:].view(q.shape)                   # 16 bytes past a 256-byte base
    assert o16.data_ptr() % 16 == 0 and o16.data_ptr() % 32 != 0
    o16.fill_(float("nan"))
    o16, lse16 = fa_fwd(q, k, v, causal, scale, out=o16)
    o32, lse32 = fa_fwd(q, k, v, causal, scale)
    assert o32.data_ptr() % 32 == 0
    assert fa_check_device_status(dev) == 0
    assert torch.equal(o16, o32) and torch.equal(lse16, lse32)
    o_ref, lse_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], causal, scale)
    check_forward(o16, lse16, o_ref, lse_ref, "16-byte aligned O")


@pytest.mark.parametrize("H,N,d", [(120, 1700, 128), (100, 4000, 64)])
def test_dynamic_schedule_ragged(H, N, d):
    # K and V of all heads above 96 MB (4 N d bytes per head) select the
    # head-grouped dynamic schedule, whose kernels store O through shared
    # memory by TMA; a ragged N makes the stores of the last tile clip.
    assert H * 4 * N * d > 96 << 20 and N % 128 != 0
    causal, scale = True, default_scale(d)
    inp = make_inputs(1, H, N, d, seed=53 + d)
    got = run_gpu(inp, causal, scale, backward=False)
    heads = sample_heads(H, 6, seed=N)
    assert heads[0] == 0 and heads[-1] == H - 1
    sub = {n: heads_of(inp[n], heads) for n in ("q", "k", "v")}
    o_ref, lse_ref = oracle.fwd(sub["q"], sub["k"], sub["v"], causal, scale)
    check_forward(heads_of(got["o"], heads), heads_of(got["lse"], heads),
                  o_ref, lse_ref, "dynamic schedule H=%d N=%d d=%d" % (H, N, d))


# ----------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_gpu_invariants(causal):
    B, H, N, d = 1, 2, 384, 128
    inp = make_inputs(B, H, N, d, seed=11)
    scale = default_scale(d)
    # Constant value rows give that row.
    c = torch.randn(d, generator=torch.Generator().manual_seed(3))
    inp_c = dict(inp)
    inp_c["v"] = c.to(torch.bfloat16).expand(B, H, N, d).contiguous()
    got = run_gpu(inp_c, causal, scale)
    cexp = inp_c["v"].double().numpy()
    assert np.max(np.abs(f64(got["o"]) - cexp)) <= O_MAX_ABS
    # Gradient sums: sum_j dV_j = sum_i dO_i ; sum_j dK_j = 0.
    got = run_gpu(inp, causal, scale)
    dv_sum = f64(got["dv"]).sum(axis=2)
    do_sum = inp["do"].double().numpy().sum(axis=2)
    assert rel_fro(dv_sum, do_sum) <= GRAD_REL_FRO
    dk = f64(got["dk"])
    assert np.linalg.norm(dk.sum(axis=2)) <= GRAD_REL_FRO * np.linalg.norm(dk)
    if causal:
        # First causal row: O_0 = V_0 and LSE_0 = scale q_0 . k_0.
        v0 = inp["v"][:, :, 0].double().numpy()
        assert np.max(np.abs(f64(got["o"])[:, :, 0] - v0)) <= 1e-6
        s00 = scale * (inp["q"][:, :, 0].double() * inp["k"][:, :, 0].double()).sum(-1)
        assert np.max(np.abs(f64(got["lse"])[:, :, 0] - s00.numpy())) <= LSE_MAX_ABS
    # Identical key rows give dQ = 0.
    inp_k = dict(inp)
    inp_k["k"] = inp["k"][:, :, :1].expand(B, H, N, d).contiguous()
    got = run_gpu(inp_k, causal, scale)
    dq = f64(got["dq"])
    ref_scale = np.linalg.norm(f64(run_gpu(inp, causal, scale)["dq"]))
    assert np.linalg.norm(dq) <= GRAD_REL_FRO * ref_scale


def test_empty_problem_is_a_no_op():
    dev = torch.device("cuda:0")
    q = torch.zeros((1, 1, 0, 128), dtype=torch.bfloat16, device=dev)
    o, lse = fa_fwd(q, q, q, True, 0.1)
    assert o.numel() == 0 and lse.numel() == 0
    dq, dk, dv = fa_bwd(q, q, q, o, lse, q, True, 0.1)
    assert dq.numel() == 0
    assert fa_check_device_status(dev) == 0


# ------------------------------------------------ full-size workloads
# Whole heads of the five workloads, compared element by element with the
# oracle (every query row of O, LSE and dQ, every key row of dK and dV).
# The first and the last head are always among them; the rest are a seeded
# sample.  Each runs in the launch configuration the benchmark times.
HEAD_SAMPLES = {
    "small_2x8x512x64": None,                # every head
    "medium_4x32x1024x128_causal": None,     # every head
    "large_8x64x2048x128_causal_sharp": 16,
    "xl_4x64x4096x128_causal": 12,
    "long_1x16x16384x128_causal": 2,
}


@pytest.mark.parametrize("name", list(HEAD_SAMPLES))
def test_workload_whole_heads(name):
    w = WORKLOADS[name]
    inp = workload_inputs(w)
    got = run_gpu(inp, w.causal, w.scale)
    count = HEAD_SAMPLES[name]
    heads = (list(range(w.heads)) if count is None
             else sample_heads(w.heads, count, seed=w.seed))
    assert heads[0] == 0 and heads[-1] == w.heads - 1
    sub = {n: heads_of(inp[n], heads) for n in ("q", "k", "v", "do")}
    del inp
    o_ref, lse_ref = oracle.fwd(sub["q"], sub["k"], sub["v"], w.causal, w.scale)
    check_forward(heads_of(got["o"], heads), heads_of(got["lse"], heads),
                  o_ref, lse_ref, name)
    del o_ref, lse_ref
    refs = oracle.bwd(sub["q"], sub["k"], sub["v"], sub["do"], w.causal, w.scale)
    check_grads([heads_of(got[n], heads) for n in ("dq", "dk", "dv")], refs,
                name)
    # Each head on its own too, so that one bad head cannot hide in the
    # norm of the others.
    for x, h in enumerate(heads):
        for n, r in zip(("dq", "dk", "dv"), refs):
            rf = rel_fro(f64(heads_of(got[n], [h])), r[x:x + 1])
            assert rf <= GRAD_REL_FRO, "%s head %d %s %.3g" % (name, h, n, rf)
