"""FP8 (E4M3) quantisation and the FP8 forward -- TEST INFRASTRUCTURE ONLY.

Follows "GPU Performance Optimization Batch 1 -- Design Spec", Item 3
("FlashAttention-3 Blackwell"), "Optional FP8 path": before the Q K^T
product, Q and K are quantised block by block to E4M3 with one scale factor
per block.  Blocks here are 16 rows by the whole head dimension (the 16-row
granularity of the page; a scale must not vary along the contraction for the
product of two quantised blocks to be rescaled exactly afterwards).

Definitions (all in float32, the precision the CUDA path decides the codes
in, so that both sides produce the same bytes):
  amax  = max |x| over the block (rows past N are not part of any block)
  scale = amax / 448 (448 = largest finite E4M3 value); 1 if amax = 0
  code  = E4M3 round-to-nearest-even of x / scale, saturating at +-448
  x~    = value(code) * scale
The forward is then the plain operation on x~ for Q and K (V unchanged), in
float64 like the rest of the oracle.

E4M3 (the "E4M3FN" layout): 1 sign bit, 4 exponent bits with bias 7, 3
mantissa bits; exponent 0 holds subnormals m * 2^-9; the all-ones pattern
S.1111.111 is NaN and there are no infinities.  The value table below is
built from that description alone.
"""
import numpy as np

E4M3_MAX = 448.0
BLOCK_ROWS = 16


def e4m3_values() -> np.ndarray:
    """float64 value of every byte code 0..255 (NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for b in range(256):
        sign = -1.0 if b & 0x80 else 1.0
        e = (b >> 3) & 0xF
        m = b & 0x7
        if e == 0xF and m == 0x7:
            vals[b] = np.nan
        elif e == 0:
            vals[b] = sign * m * 2.0 ** -9
        else:
            vals[b] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_VALUES = e4m3_values()
_POS_CODES = np.arange(0x00, 0x7F)            # 0 .. 448, increasing
_POS_VALUES = _VALUES[_POS_CODES]


def e4m3_encode(x) -> np.ndarray:
    """Byte codes of float32 values: round to nearest, ties to the even code
    (even mantissa), magnitudes above 448 saturate to 448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    a_sat = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a_sat, side="left")   # first >= a
    hi = np.clip(hi, 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    d_hi = _POS_VALUES[hi] - a_sat
    d_lo = a_sat - _POS_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (_POS_CODES[lo] % 2 == 0))
    code = np.where(pick_lo, _POS_CODES[lo], _POS_CODES[hi]).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)
    return code


def e4m3_decode(code) -> np.ndarray:
    return _VALUES[np.asarray(code, dtype=np.uint8)]


def quantize_rowblocks(x, block_rows: int = BLOCK_ROWS):
    """x: [..., N, d] (any float; bf16 inputs are exact in float32).
    Returns (codes uint8 [..., N, d], scales float32 [..., ceil(N / 16)])."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    x = np.asarray(x, dtype=np.float32)
    *lead, N, d = x.shape
    nb = (N + block_rows - 1) // block_rows
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty((*lead, nb), dtype=np.float32)
    for b in range(nb):
        r0, r1 = b * block_rows, min(N, (b + 1) * block_rows)
        blk = x[..., r0:r1, :]
        amax = np.max(np.abs(blk), axis=(-2, -1)).astype(np.float32)
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX),
                     np.float32(1.0)).astype(np.float32)
        scales[..., b] = s
        codes[..., r0:r1, :] = e4m3_encode(blk / s[..., None, None])
    return codes, scales


def dequantize_rowblocks(codes, scales, block_rows: int = BLOCK_ROWS):
    """float64 x~ = value(code) * scale, per 16-row block."""
    v = e4m3_decode(codes)
    s = np.repeat(np.asarray(scales, dtype=np.float64), block_rows, axis=-1)
    return v * s[..., :v.shape[-2], None]


def fwd_fp8(q, k, v, causal: bool, scale: float):
    """Forward of the FP8 path: Q and K quantised per 16-row block, then the
    plain operation (oracle.fwd) on the dequantised values."""
    from . import fwd
    qc, qs = quantize_rowblocks(q)
    kc, ks = quantize_rowblocks(k)
    return fwd(dequantize_rowblocks(qc, qs), dequantize_rowblocks(kc, ks), v,
               causal, scale)
