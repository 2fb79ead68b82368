"""GPU parity of the FP8 forward path against the CPU oracle.

* fa_quantize_e4m3 (the quantisation step of fa_fwd_fp8) produces exactly
  the oracle's E4M3 codes and float32 scales: both decide the codes in
  float32 with IEEE division and round-to-nearest-even, so the comparison is
  byte for byte.
* fa_fwd_fp8 matches oracle.fp8.fwd_fp8 (the plain forward on dequantised
  Q and K, in float64) within the tolerances of the bf16 forward (O max-abs
  2e-2 and rel-Frobenius 1e-2, LSE max-abs 1e-3): the kernel's fp8 products
  are exact, so only fp32 accumulation and the bf16 P and O roundings remain.
"""
import numpy as np
import pytest
import torch

import oracle.fp8 as ofp8
from tiled_attention_bwd_gb300 import (fa_check_device_status, fa_fwd_fp8,
                                       fa_quantize_e4m3)
from tiled_attention_bwd_gb300.workloads import (WORKLOADS, default_scale,
                                                 make_inputs, sample_heads,
                                                 workload_inputs)

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_FRO, LSE_MAX_ABS = 2e-2, 1e-2, 1e-3


def rel_fro(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("B,H,N,d,mult", [(1, 1, 128, 128, 1.0),
                                          (2, 3, 333, 128, 1.0),
                                          (1, 2, 17, 64, 4.0),
                                          (1, 4, 1000, 128, 30.0),
                                          (1, 1, 1, 128, 1.0)])
def test_quantisation_is_bit_exact(B, H, N, d, mult):
    dev = torch.device("cuda:0")
    x = (make_inputs(B, H, N, d, seed=N + d)["q"].float() * mult)
    x[..., :min(N, 16), :] = 0.0        # an all-zero block
    if N > 40:
        x[..., 33, 5] = 60000.0          # one block dominated by an outlier
    x = x.to(torch.bfloat16)
    codes, scales = fa_quantize_e4m3(x.to(dev))
    assert fa_check_device_status(dev) == 0
    ref_codes, ref_scales = ofp8.quantize_rowblocks(x)
    nb = ref_scales.shape[-1]
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    got_scales = scales.cpu().numpy()
    assert np.array_equal(got_scales[..., :nb], ref_scales)
    assert np.all(got_scales[..., nb:] == 1.0)     # padding blocks past N


def check_forward(o, lse, o_ref, lse_ref, tag):
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all(), tag
    err = np.max(np.abs(o - o_ref))
    assert err <= O_MAX_ABS, "%s O max-abs %.3g" % (tag, err)
    rf = rel_fro(o, o_ref)
    assert rf <= O_REL_FRO, "%s O rel-Frobenius %.3g" % (tag, rf)
    le = np.max(np.abs(lse - lse_ref))
    assert le <= LSE_MAX_ABS, "%s LSE max-abs %.3g" % (tag, le)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,H,N,causal,mult", [(1, 1, 128, False, 1.0),
                                               (1, 2, 256, True, 1.0),
                                               (2, 2, 384, True, 2.0),
                                               (1, 3, 333, False, 1.0),
                                               (1, 2, 1000, True, 1.0),
                                               (1, 1, 17, True, 1.0),
                                               (2, 8, 512, False, 1.0)])
def test_fp8_forward_every_element(B, H, N, causal, mult, d):
    dev = torch.device("cuda:0")
    inp = make_inputs(B, H, N, d, seed=77 + N + d, qk_mult=mult)
    scale = default_scale(d)
    o, lse = fa_fwd_fp8(*(inp[n].to(dev) for n in ("q", "k", "v")), causal,
                        scale)
    assert fa_check_device_status(dev) == 0
    o_ref, lse_ref = ofp8.fwd_fp8(inp["q"], inp["k"], inp["v"], causal, scale)
    check_forward(o, lse, o_ref, lse_ref,
                  "%dx%dx%dx%d causal=%d" % (B, H, N, d, causal))


def test_fp8_forward_full_size_sampled_heads():
    w = WORKLOADS["xl_4x64x4096x128_causal"]
    dev = torch.device("cuda:0")
    inp = workload_inputs(w)
    o, lse = fa_fwd_fp8(*(inp[n].to(dev) for n in ("q", "k", "v")), w.causal,
                        w.scale)
    assert fa_check_device_status(dev) == 0
    heads = sample_heads(w.heads, 3, seed=w.seed)
    flat = lambda t: t.reshape(w.B * w.H, *t.shape[2:])[heads]
    o_ref, lse_ref = ofp8.fwd_fp8(flat(inp["q"]), flat(inp["k"]),
                                  flat(inp["v"]), w.causal, w.scale)
    check_forward(flat(o.cpu()), flat(lse.cpu()), o_ref, lse_ref, w.name)
