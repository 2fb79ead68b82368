"""Pins of the oracle's FP8 (E4M3) quantisation and FP8 forward (CPU only).

The E4M3 value table and the encoder are checked against PyTorch's own
float8_e4m3fn type (an independent implementation of the same format), the
rounding ties and saturation against hand-worked cases, the per-block scales
against their definition's fixed points, and the FP8 forward against the
plain forward in the case where quantisation changes nothing.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_value_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    theirs = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fp8.e4m3_values()
    assert np.array_equal(np.isnan(ours), np.isnan(theirs))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], theirs[ok])


def test_value_table_landmarks():
    v = fp8.e4m3_values()
    assert v[0x38] == 1.0 and v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6   # subnormal, normal
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert np.sum(~np.isnan(v)) == 254


def test_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.uniform(-448.0, 448.0, 20000),
        rng.normal(0.0, 1.0, 20000),
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 20000),      # subnormal range
        fp8.e4m3_values()[:0x7F],                        # exact values
        (fp8.e4m3_values()[1:0x7E] + fp8.e4m3_values()[2:0x7F]) / 2,  # ties
    ]).astype(np.float32)
    ours = fp8.e4m3_encode(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_ties_go_to_even_and_large_values_saturate():
    enc = fp8.e4m3_encode
    assert enc(np.float32(1.0625))[()] == 0x38    # 1.0 | 1.125: even is 1.0
    assert enc(np.float32(1.1875))[()] == 0x3A    # 1.125 | 1.25: even is 1.25
    assert enc(np.float32(3.0 * 2 ** -10))[()] == 0x02   # 1 | 2 (x 2^-9): 2
    assert enc(np.float32(464.0))[()] == 0x7E     # past 448: saturates
    assert enc(np.float32(1e30))[()] == 0x7E
    assert enc(np.float32(-1e30))[()] == 0xFE
    assert enc(np.float32(np.nan))[()] == 0x7F


def test_block_scales_and_codes():
    rng = np.random.default_rng(5)
    x = rng.normal(0.0, 2.0, (2, 3, 50, 64)).astype(np.float32)  # 4 blocks, last partial
    x[0, 0, 16:32] = 0.0                                          # an all-zero block
    codes, scales = fp8.quantize_rowblocks(x)
    assert codes.shape == x.shape and scales.shape == (2, 3, 4)
    assert scales[0, 0, 1] == 1.0 and np.all(codes[0, 0, 16:32] == 0)
    for b in range(4):
        blk = x[..., 16 * b:16 * b + 16, :]
        amax = np.abs(blk).max(axis=(-2, -1))
        nz = amax > 0
        assert np.array_equal(scales[..., b][nz],
                              (amax[nz] / np.float32(448.0)).astype(np.float32))
        # the largest element of each block lands on +-448 exactly
        c = codes[..., 16 * b:16 * b + 16, :]
        assert np.all((np.abs(fp8.e4m3_decode(c)).max(axis=(-2, -1)) == 448.0)[nz])
    # dequantisation error: half a unit in the last place of E4M3 (2^-4
    # relative) for normal values, 2^-10 * scale absolute below them
    xt = fp8.dequantize_rowblocks(codes, scales)
    s = np.repeat(scales.astype(np.float64), 16, axis=-1)[..., :50, None]
    err = np.abs(xt - x)
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s) * (1 + 1e-9))


def test_quantisation_is_idempotent():
    rng = np.random.default_rng(7)
    x = rng.normal(0.0, 1.0, (1, 2, 40, 128)).astype(np.float32)
    c1, s1 = fp8.quantize_rowblocks(x)
    xt = fp8.dequantize_rowblocks(c1, s1).astype(np.float32)
    c2, s2 = fp8.quantize_rowblocks(xt)
    assert np.array_equal(s1, s2) and np.array_equal(c1, c2)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_equals_plain_forward_on_representable_inputs(causal):
    # Every element already an E4M3 value and every block containing +-448:
    # the scale is 1 and quantisation is the identity.
    rng = np.random.default_rng(11)
    vals = fp8.e4m3_values()
    finite = vals[~np.isnan(vals)]
    B, H, N, d = 1, 2, 48, 64
    q = rng.choice(finite, (B, H, N, d)).astype(np.float32)
    k = rng.choice(finite, (B, H, N, d)).astype(np.float32)
    q[..., ::16, 0] = 448.0
    k[..., ::16, 0] = -448.0
    v = rng.normal(0, 1, (B, H, N, d))
    scale = 1e-3
    o1, l1 = oracle.fp8.fwd_fp8(q, k, v, causal, scale)
    o2, l2 = oracle.fwd(q, k, v, causal, scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_fp8_forward_is_close_to_the_exact_forward():
    # Quantisation moves the result by a bounded amount: a sanity pin that
    # a dropped scale or a transposed block would break.
    rng = np.random.default_rng(13)
    q = rng.normal(0, 1, (1, 2, 64, 128)).astype(np.float32)
    k = rng.normal(0, 1, (1, 2, 64, 128)).astype(np.float32)
    v = rng.normal(0, 1, (1, 2, 64, 128))
    scale = 128 ** -0.5
    o1, l1 = oracle.fp8.fwd_fp8(q, k, v, True, scale)
    o2, l2 = oracle.fwd(q, k, v, True, scale)
    assert np.max(np.abs(l1 - l2)) < 0.1
    assert np.linalg.norm(o1 - o2) / np.linalg.norm(o2) < 0.05
