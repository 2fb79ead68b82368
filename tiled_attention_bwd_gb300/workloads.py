"""Seeded synthetic workloads: shapes and input tensors, nothing else.

This module holds no attention arithmetic.  It is the one piece shared by the
CUDA path's tests/benchmark and the CPU oracle's callers, so both consume the
identical bf16 bytes.

Recipe (the pages run on random tensors of shape [batch, heads, seq_len,
head_dim], "RTX Flash Attention Implementation COMPLETE", "Usage Examples",
and time the shapes of "Validated Performance Gains"):
  * a CPU ``torch.Generator`` seeded with ``seed``;
  * Q, K, V, dO drawn in that order as float32 standard normals;
  * Q and K multiplied by ``qk_mult`` (2.0 for the sharper-softmax workload);
  * each rounded to bfloat16 (round to nearest even);
  * scale = the float32 value of 1/sqrt(head_dim).
"""
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    qk_mult: float
    seed: int

    @property
    def scale(self) -> float:
        return default_scale(self.d)

    @property
    def heads(self) -> int:
        return self.B * self.H

    def fwd_flops(self) -> float:
        """Algorithmic forward FLOPs: two N x N x d contractions per head
        (4 B H N^2 d), halved for causal (only the lower triangle counts)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    def bwd_flops(self) -> float:
        """Backward: five contractions of the same size (2.5 x forward)."""
        return 2.5 * self.fwd_flops()

    def label(self) -> str:
        return "%dx%dx%dx%d %s" % (self.B, self.H, self.N, self.d,
                                   "causal" if self.causal else "non-causal")


# The five workloads: the pages' four timing shapes plus one long sequence.
WORKLOADS = {
    "small_2x8x512x64": Workload("small_2x8x512x64", 2, 8, 512, 64, False, 1.0, 1001),
    "medium_4x32x1024x128_causal": Workload("medium_4x32x1024x128_causal", 4, 32, 1024, 128, True, 1.0, 1002),
    "large_8x64x2048x128_causal_sharp": Workload("large_8x64x2048x128_causal_sharp", 8, 64, 2048, 128, True, 2.0, 1003),
    "xl_4x64x4096x128_causal": Workload("xl_4x64x4096x128_causal", 4, 64, 4096, 128, True, 1.0, 1004),
    "long_1x16x16384x128_causal": Workload("long_1x16x16384x128_causal", 1, 16, 16384, 128, True, 1.0, 1005),
}
HEADLINE = "xl_4x64x4096x128_causal"


def default_scale(d: int) -> float:
    """float32 value of 1/sqrt(d), widened to a Python float."""
    return float(np.float32(1.0) / np.sqrt(np.float32(d)))


def make_inputs(B: int, H: int, N: int, d: int, seed: int,
                qk_mult: float = 1.0):
    """Return dict(q, k, v, do) of contiguous bf16 CPU tensors [B,H,N,d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    out = {}
    for name in ("q", "k", "v", "do"):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if name in ("q", "k") and qk_mult != 1.0:
            x.mul_(qk_mult)
        out[name] = x.to(torch.bfloat16).contiguous()
        del x
    return out


def make_grouped_inputs(B: int, H: int, Hkv: int, N: int, d: int, seed: int,
                        qk_mult: float = 1.0):
    """Inputs with Hkv key/value heads: q, do [B,H,N,d]; k, v [B,Hkv,N,d]
    (same recipe, drawn in the order q, k, v, do)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = {}
    for name in ("q", "k", "v", "do"):
        shape = (B, Hkv if name in ("k", "v") else H, N, d)
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if name in ("q", "k") and qk_mult != 1.0:
            x.mul_(qk_mult)
        out[name] = x.to(torch.bfloat16).contiguous()
        del x
    return out


def make_seq_lens(B: int, N: int, seed: int, fixed=()):
    """int32 [B] per-sequence lengths: the leading entries are `fixed`
    (clamped to [0, N]), the rest drawn uniformly from [1, N]."""
    rng = np.random.default_rng(int(seed))
    lens = [min(max(int(x), 0), N) for x in fixed][:B]
    if len(lens) < B:
        lens += [int(x) for x in rng.integers(1, N + 1, B - len(lens))]
    return torch.tensor(lens, dtype=torch.int32)


def visible_pairs(N: int, causal: bool, window: int, r0: int = 0,
                  r1: int = None) -> int:
    """Number of (query, key) pairs with the query in rows [r0, r1) that a
    query/key length N leaves visible: key j is visible to query i when
    j <= i (causal) and |i - j| <= window (window >= 0).  Used only to count
    the work a band does."""
    r1 = N if r1 is None else r1
    i = np.arange(r0, r1, dtype=np.int64)
    lo = np.maximum(0, i - window) if window >= 0 else np.zeros_like(i)
    if causal:
        hi = i
    elif window >= 0:
        hi = np.minimum(N - 1, i + window)
    else:
        hi = np.full_like(i, N - 1)
    return int((hi - lo + 1).sum())


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)


def sample_heads(n_heads: int, count: int, seed: int):
    """A seeded sample of `count` distinct head indices in [0, n_heads),
    always including the first and the last head."""
    count = max(1, min(count, n_heads))
    if count >= n_heads:
        return list(range(n_heads))
    rng = np.random.default_rng(seed)
    picks = {0, n_heads - 1}
    while len(picks) < count:
        picks.add(int(rng.integers(0, n_heads)))
    return sorted(picks)


__all__ = ["Workload", "WORKLOADS", "HEADLINE", "default_scale", "make_inputs",
           "make_grouped_inputs", "visible_pairs", "workload_inputs",
           "sample_heads"]
