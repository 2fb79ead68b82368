"""Splitting one attention problem over several GPUs by heads.

Every (batch entry, head) of attention is independent in the forward and the
backward pass, and the operation has no parameters to reduce, so a problem
spread over GPUs needs no collective on its data path: each GPU runs the
plain entry points on a contiguous slice of the heads.  (The pages name
multi-GPU operation only as "Distributed attention across devices",
"RTX Flash Attention Implementation COMPLETE", "Platform Expansion".)

The unit of the split is a key/value group: one key/value head with the
H / Hkv query heads that read it (with Hkv = H, simply one head).  Groups
are numbered in memory order over [B, Hkv]; a contiguous range of groups is
then a contiguous range of query heads of the [B, H, N, d] tensors and of
key/value heads of the [B, Hkv, N, d] ones, and is itself a valid problem of
one batch entry with (hi - lo) * H / Hkv query heads and hi - lo key/value
heads.  With per-sequence lengths the unit is a whole batch entry instead,
since its length belongs to all of its heads.

Nothing here touches a GPU; the benchmark and the tests use it on the host.
"""
from dataclasses import dataclass


def unit_range(rank: int, world: int, n_units: int):
    """Contiguous units [lo, hi) of `rank` out of `world`: the first
    n_units % world ranks get one unit more than the others."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank %d outside a world of %d" % (rank, world))
    if n_units < 0:
        raise ValueError("negative unit count")
    base, extra = divmod(n_units, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


@dataclass(frozen=True)
class HeadSlice:
    """Rank's share of a [B, H, N, d] problem with Hkv key/value heads.

    q_lo:q_hi index the flattened B*H query heads (q, o, lse, dout, dq);
    kv_lo:kv_hi the flattened B*Hkv key/value heads (k, v, dk, dv).  As a
    problem of its own the slice has shape (B_s, H_s, Hkv_s): one batch
    entry of all the slice's heads, or, when split by batch entries, the
    slice's entries with every head."""
    q_lo: int
    q_hi: int
    kv_lo: int
    kv_hi: int
    B_s: int
    H_s: int
    Hkv_s: int
    b_lo: int   # first batch entry (by-batch split only, else -1)
    b_hi: int

    @property
    def empty(self) -> bool:
        return self.q_hi <= self.q_lo


def head_slice(rank: int, world: int, B: int, H: int, Hkv: int,
               by_batch: bool = False) -> HeadSlice:
    """The slice of `rank`: whole key/value groups, or whole batch entries
    when `by_batch` (per-sequence lengths)."""
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError("Hkv = %d must divide H = %d" % (Hkv, H))
    g = H // Hkv
    if by_batch:
        b_lo, b_hi = unit_range(rank, world, B)
        n = b_hi - b_lo
        return HeadSlice(b_lo * H, b_hi * H, b_lo * Hkv, b_hi * Hkv,
                         n, H, Hkv, b_lo, b_hi)
    lo, hi = unit_range(rank, world, B * Hkv)
    n = hi - lo
    return HeadSlice(lo * g, hi * g, lo, hi, 1 if n else 0, n * g, n, -1, -1)


def full_slice(B: int, H: int, Hkv: int) -> HeadSlice:
    """The whole problem as one slice, with its own shape (B, H, Hkv)."""
    return HeadSlice(0, B * H, 0, B * Hkv, B, H, Hkv, 0, B)


def slice_heads(t, lo: int, hi: int, B_s: int):
    """Rows [lo, hi) of the flattened leading two dimensions of a [B, X, ...]
    tensor, as a [B_s, (hi - lo) / B_s, ...] view (no copy)."""
    flat = t.reshape(t.shape[0] * t.shape[1], *t.shape[2:])
    part = flat[lo:hi]
    if B_s == 0:
        return part.reshape(0, 0, *t.shape[2:])
    return part.reshape(B_s, (hi - lo) // B_s, *t.shape[2:])


__all__ = ["unit_range", "HeadSlice", "head_slice", "full_slice",
           "slice_heads"]
