"""CPU fp64 attention oracle -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library in
``tiled_attention_bwd_gb300``) never imports, links or calls it, and the two
share no code.

Functions take numpy arrays (any float dtype; bf16 torch tensors should be
converted with ``.double().numpy()``, which is exact) of shape [B, H, N, d]
or [BH, N, d], and return float64 arrays of the same shape (LSE: [..., N]).

What each function follows:
  fwd         -- the definition O = softmax(scale Q K^T [+ causal mask]) V and
                 LSE = ln sum_j exp(scale q_i . k_j), two-pass per row
                 ("RTX Flash Attention Implementation COMPLETE", "Usage
                 Examples": forward(q, k, v, causal, scale) -> output, lse).
  fwd_online  -- the same result by the running-max / running-sum update of
                 "RTX Flash Attention Implementation COMPLETE", "Online
                 Softmax Algorithm", over key tiles, optionally lazy.
  fwd_rows, bwd_rows -- the same computations restricted to a range of
                 query rows (rows are independent), so that long sequences can
                 be checked on rows the oracle finishes quickly.
  fwd_ext, bwd_ext -- grouped / multi-query K/V heads (query head h reads
                 K/V head h // (H // Hkv); dK, dV summed over each group) and
                 a sliding window (key j visible to query i only if
                 |i - j| <= window, and j <= i when causal).  The pages list
                 both as future variants ("Advanced Features (Future)":
                 multi-query / grouped query attention; sliding window).
  fwd_varlen, bwd_varlen -- per-sequence lengths over a padded batch (the
                 "variable sequence lengths" of "GPU Performance Optimization
                 Batch 1 -- Design Spec", Item 1, Constraint): batch entry b
                 is fwd_ext / bwd_ext on its first seq_lens[b] rows alone;
                 the forward's padding rows are NaN, the gradients' zero.
  fp8         -- (submodule) E4M3 quantisation of Q and K per 16-row block
                 with one float32 scale each, and the forward on the
                 dequantised values ("GPU Performance Optimization Batch 1 --
                 Design Spec", Item 3, "Optional FP8 path").
  bwd         -- gradients dQ, dK, dV of L with dL/dO = dout, P recomputed
                 from the row's LSE ("GPU Performance Optimization Batch 1 --
                 Design Spec", Item 3, backward paragraph).  The formulas come
                 from the chain rule; the pages do not print them.

Every function is pinned by tests/test_oracle.py against things other than
itself: torch fp64 autograd, central finite differences, closed forms and
invariants (see that file).
"""
import ctypes

import numpy as np

from .build import build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = build_oracle()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_fwd.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_int,
                                   ctypes.c_double, dp, dp]
        lib.oracle_fwd.restype = None
        lib.oracle_fwd_online.argtypes = [dp, dp, dp, i64, i64, i64,
                                          ctypes.c_int, ctypes.c_double, i64,
                                          ctypes.c_double, dp, dp]
        lib.oracle_fwd_online.restype = None
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, i64, i64, i64,
                                   ctypes.c_int, ctypes.c_double, dp, dp, dp]
        lib.oracle_bwd.restype = None
        lib.oracle_fwd_rows.argtypes = [dp, dp, dp, i64, i64, i64,
                                        ctypes.c_int, ctypes.c_double, i64,
                                        i64, dp, dp]
        lib.oracle_fwd_rows.restype = None
        lib.oracle_bwd_rows.argtypes = [dp, dp, dp, dp, i64, i64, i64,
                                        ctypes.c_int, ctypes.c_double, i64,
                                        i64, dp, dp, dp]
        lib.oracle_bwd_rows.restype = None
        lib.oracle_fwd_ext_rows.argtypes = [dp, dp, dp, i64, i64, i64, i64,
                                            i64, ctypes.c_int, i64,
                                            ctypes.c_double, i64, i64, dp, dp]
        lib.oracle_fwd_ext_rows.restype = None
        lib.oracle_bwd_ext_rows.argtypes = [dp, dp, dp, dp, i64, i64, i64,
                                            i64, i64, ctypes.c_int, i64,
                                            ctypes.c_double, i64, i64, dp, dp,
                                            dp]
        lib.oracle_bwd_ext_rows.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
    return _lib


def _as_f64(x):
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape(q):
    if q.ndim == 4:
        B, H, N, d = q.shape
        return B * H, N, d
    if q.ndim == 3:
        return q.shape
    raise ValueError("expected [B,H,N,d] or [BH,N,d], got %s" % (q.shape,))


def num_threads() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Run later oracle calls (from this thread) on n >= 1 threads."""
    if int(n) < 1:
        raise ValueError("thread count must be >= 1")
    _load().oracle_set_num_threads(int(n))


def fwd(q, k, v, causal: bool, scale: float):
    """Two-pass fp64 forward; returns (O, LSE)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    BH, N, d = _shape(q)
    o = np.empty_like(q)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), BH, N, d, int(bool(causal)),
                       float(scale), _ptr(o), _ptr(lse))
    return o, lse


def fwd_online(q, k, v, causal: bool, scale: float, tile: int = 1,
               tau: float = 0.0):
    """Online-softmax fp64 forward over key tiles of `tile` keys; with
    tau > 0 the reference max is kept until exceeded by more than tau."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    BH, N, d = _shape(q)
    o = np.empty_like(q)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    _load().oracle_fwd_online(_ptr(q), _ptr(k), _ptr(v), BH, N, d,
                              int(bool(causal)), float(scale), int(tile),
                              float(tau), _ptr(o), _ptr(lse))
    return o, lse


def bwd(q, k, v, dout, causal: bool, scale: float):
    """fp64 backward; returns (dQ, dK, dV).  O and D come from the oracle's
    own fp64 forward of the same inputs."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    BH, N, d = _shape(q)
    dq = np.empty_like(q)
    dk = np.empty_like(q)
    dv = np.empty_like(q)
    _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), BH, N, d,
                       int(bool(causal)), float(scale), _ptr(dq), _ptr(dk),
                       _ptr(dv))
    return dq, dk, dv


def fwd_rows(q, k, v, causal: bool, scale: float, r0: int, r1: int):
    """Forward for query rows r0 <= i < r1 only; other rows are NaN."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    BH, N, d = _shape(q)
    if not 0 <= r0 <= r1 <= N:
        raise ValueError("bad row range")
    o = np.full_like(q, np.nan)
    lse = np.full(q.shape[:-1], np.nan, dtype=np.float64)
    _load().oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), BH, N, d,
                            int(bool(causal)), float(scale), int(r0), int(r1),
                            _ptr(o), _ptr(lse))
    return o, lse


def bwd_rows(q, k, v, dout, causal: bool, scale: float, r0: int, r1: int):
    """Backward contributions of query rows r0 <= i < r1 only.  dQ is exact on
    those rows; dK/dV are partial sums over those rows (exact for keys
    j >= r0 when causal and r1 == N)."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    BH, N, d = _shape(q)
    if not 0 <= r0 <= r1 <= N:
        raise ValueError("bad row range")
    dq = np.empty_like(q)
    dk = np.empty_like(q)
    dv = np.empty_like(q)
    _load().oracle_bwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), BH, N, d,
                            int(bool(causal)), float(scale), int(r0), int(r1),
                            _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


def _ext_shapes(q, k):
    if q.ndim != 4 or k.ndim != 4:
        raise ValueError("expected [B,H,N,d] q and [B,Hkv,N,d] k")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or Hkv < 1 or H % Hkv != 0:
        raise ValueError("bad grouped shapes %s / %s" % (q.shape, k.shape))
    return B, H, Hkv, N, d


def fwd_ext(q, k, v, causal: bool, scale: float, window: int = -1,
            r0: int = 0, r1: int = None):
    """Forward with Hkv = k.shape[1] key/value heads and an optional window
    (window < 0: none).  Rows outside [r0, r1) are NaN."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, Hkv, N, d = _ext_shapes(q, k)
    r1 = N if r1 is None else r1
    o = np.full_like(q, np.nan)
    lse = np.full(q.shape[:-1], np.nan, dtype=np.float64)
    _load().oracle_fwd_ext_rows(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, N, d,
                                int(bool(causal)), int(window), float(scale),
                                int(r0), int(r1), _ptr(o), _ptr(lse))
    return o, lse


def bwd_ext(q, k, v, dout, causal: bool, scale: float, window: int = -1,
            r0: int = 0, r1: int = None):
    """Backward of fwd_ext: dQ [B,H,N,d]; dK, dV [B,Hkv,N,d] summed over each
    group of query heads.  Only query rows in [r0, r1) contribute."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, H, Hkv, N, d = _ext_shapes(q, k)
    r1 = N if r1 is None else r1
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(k)
    _load().oracle_bwd_ext_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, H,
                                Hkv, N, d, int(bool(causal)), int(window),
                                float(scale), int(r0), int(r1), _ptr(dq),
                                _ptr(dk), _ptr(dv))
    return dq, dk, dv


def _lengths(seq_lens, B, N):
    lens = [int(x) for x in np.asarray(seq_lens).reshape(-1)]
    if len(lens) != B:
        raise ValueError("seq_lens has %d entries for B = %d" % (len(lens), B))
    return [min(max(x, 0), N) for x in lens]


def fwd_varlen(q, k, v, seq_lens, causal: bool, scale: float,
               window: int = -1):
    """Forward over a padded batch: entry b is fwd_ext on rows [0, L_b) of
    its q, k, v (L_b = seq_lens[b] clamped to [0, N]).  O and LSE rows at or
    past L_b are NaN."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, Hkv, N, d = _ext_shapes(q, k)
    o = np.full_like(q, np.nan)
    lse = np.full(q.shape[:-1], np.nan, dtype=np.float64)
    for b, L in enumerate(_lengths(seq_lens, B, N)):
        if L == 0:
            continue
        ob, lb = fwd_ext(q[b:b + 1, :, :L], k[b:b + 1, :, :L],
                         v[b:b + 1, :, :L], causal, scale, window)
        o[b, :, :L] = ob[0]
        lse[b, :, :L] = lb[0]
    return o, lse


def bwd_varlen(q, k, v, dout, seq_lens, causal: bool, scale: float,
               window: int = -1):
    """Backward of fwd_varlen: entry b is bwd_ext on rows [0, L_b); the
    gradients' rows at or past L_b are zero (padding does not take part)."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, H, Hkv, N, d = _ext_shapes(q, k)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(k)
    for b, L in enumerate(_lengths(seq_lens, B, N)):
        if L == 0:
            continue
        g = bwd_ext(q[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L],
                    dout[b:b + 1, :, :L], causal, scale, window)
        dq[b, :, :L], dk[b, :, :L], dv[b, :, :L] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv
