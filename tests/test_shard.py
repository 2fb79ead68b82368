"""Splitting one problem over GPUs by heads (host logic, CPU only).

Each rank takes a contiguous range of key/value groups (whole batch entries
with per-sequence lengths) and runs the plain entry points on it, with no
collective on the data path.  Checked here:
  * the ranges of all ranks cover every unit exactly once, ragged counts
    included, both computed per rank in gloo processes (world sizes 2 and
    3) and gathered, and directly;
  * the slices' FLOPs add up to the whole problem's;
  * a slice taken as a problem of its own maps each query head to the same
    key/value head as the whole problem does.
"""
import dataclasses
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from tiled_attention_bwd_gb300.shard import (full_slice, head_slice,  # noqa: E402
                                             slice_heads, unit_range)
from tiled_attention_bwd_gb300.workloads import (WORKLOADS,  # noqa: E402
                                                 make_seq_lens)

CASES = [
    # B, H, Hkv, varlen
    (4, 64, 64, False), (4, 64, 8, False), (1, 16, 16, False),
    (2, 8, 1, False), (3, 5, 5, False), (4, 64, 64, True), (3, 4, 2, True),
]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [dataclasses.astuple(head_slice(rank, world, B, H, Hkv,
                                               by_batch=vl))
                for B, H, Hkv, vl in CASES]
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        out[rank] = gathered
    finally:
        dist.destroy_process_group()


def _covers_once(ranges, n):
    seen = [0] * n
    for lo, hi in ranges:
        assert 0 <= lo <= hi <= n
        for x in range(lo, hi):
            seen[x] += 1
    return all(c == 1 for c in seen)


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_cover_every_head_once(world):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        assert out[r] == out[0]           # every rank sees the same split
    gathered = out[0]
    for x, (B, H, Hkv, vl) in enumerate(CASES):
        slices = [gathered[r][x] for r in range(world)]
        assert _covers_once([(s[0], s[1]) for s in slices], B * H)
        assert _covers_once([(s[2], s[3]) for s in slices], B * Hkv)
        for r in range(world):
            assert dataclasses.astuple(
                head_slice(r, world, B, H, Hkv, by_batch=vl)) == slices[r]


@pytest.mark.parametrize("n", [0, 1, 5, 8, 17, 256])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_unit_ranges_are_contiguous_and_balanced(n, world):
    ranges = [unit_range(r, world, n) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [hi - lo for lo, hi in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_bad_arguments_are_refused():
    with pytest.raises(ValueError):
        unit_range(2, 2, 10)
    with pytest.raises(ValueError):
        head_slice(0, 2, 4, 64, 5)


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_slice_flops_add_up_to_the_whole_problem(name, world):
    w = WORKLOADS[name]
    for hkv, window in ((w.H, -1), (max(1, w.H // 8), -1), (w.H, 100)):
        whole = bench.step_flops(w, window, None)
        parts = [bench.slice_flops(w, window, head_slice(r, world, w.B, w.H, hkv))
                 for r in range(world)]
        assert sum(p[0] for p in parts) == pytest.approx(whole[0], rel=1e-12)
        assert sum(p[1] for p in parts) == pytest.approx(whole[1], rel=1e-12)
    lens = make_seq_lens(w.B, w.N, seed=w.seed)
    whole = bench.step_flops(w, -1, lens)
    parts = [bench.slice_flops(w, -1, head_slice(r, world, w.B, w.H, w.H,
                                                 by_batch=True), lens)
             for r in range(world)]
    assert sum(p[0] for p in parts) == pytest.approx(whole[0], rel=1e-12)
    full = bench.slice_flops(w, -1, full_slice(w.B, w.H, w.H))
    assert full == pytest.approx(bench.step_flops(w, -1, None), rel=1e-12)


@pytest.mark.parametrize("B,H,Hkv", [(4, 8, 8), (4, 8, 2), (3, 6, 1)])
@pytest.mark.parametrize("world", [2, 3, 5])
def test_a_slice_is_a_problem_of_its_own(B, H, Hkv, world):
    # Tensors whose entries name their own (flattened) head.
    q = torch.arange(B * H).reshape(B, H, 1, 1).expand(B, H, 3, 2).contiguous()
    k = torch.arange(B * Hkv).reshape(B, Hkv, 1, 1).expand(B, Hkv, 3, 2).contiguous()
    g = H // Hkv
    q_parts, k_parts = [], []
    for r in range(world):
        s = head_slice(r, world, B, H, Hkv)
        qs = slice_heads(q, s.q_lo, s.q_hi, s.B_s)
        ks = slice_heads(k, s.kv_lo, s.kv_hi, s.B_s)
        assert tuple(qs.shape[:2]) == (s.B_s, s.H_s)
        assert tuple(ks.shape[:2]) == (s.B_s, s.Hkv_s)
        if s.empty:
            continue
        assert s.H_s == s.Hkv_s * g          # whole groups only
        # Inside the slice, query head h reads key/value head h // g (the
        # rule of the entry points); the whole problem has query head
        # b*H + h read b*Hkv + h // g.  They agree.
        for hs in range(s.H_s):
            gq = int(qs[0, hs, 0, 0])
            b, h = divmod(gq, H)
            assert int(ks[0, hs // g, 0, 0]) == b * Hkv + h // g
        q_parts.append(qs.reshape(-1, 3, 2))
        k_parts.append(ks.reshape(-1, 3, 2))
    assert torch.equal(torch.cat(q_parts), q.reshape(-1, 3, 2))
    assert torch.equal(torch.cat(k_parts), k.reshape(-1, 3, 2))


def test_batch_split_keeps_lengths_with_their_entries():
    B, H, Hkv = 5, 4, 2
    for world in (2, 3, 7):
        entries = []
        for r in range(world):
            s = head_slice(r, world, B, H, Hkv, by_batch=True)
            assert s.q_lo == s.b_lo * H and s.q_hi == s.b_hi * H
            assert s.kv_lo == s.b_lo * Hkv and s.kv_hi == s.b_hi * Hkv
            entries += list(range(s.b_lo, s.b_hi))
        assert entries == list(range(B))
