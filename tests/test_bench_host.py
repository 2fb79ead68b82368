"""Host-side logic of bench.py (CPU only).

* The timing reduction across ranks (max over ranks, as the benchmark takes
  the slowest rank's time) is checked with two gloo processes on CPU.
* The committed traffic record is only used while the kernel sources still
  match the fingerprint stored with it.
"""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


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
        bench.barrier(world)
        value = bench.max_over_ranks(1.5 + rank, world)
        out[rank] = value
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_processes():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == pytest.approx(2.5) and out[1] == pytest.approx(2.5)


def test_single_process_timing_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_committed_traffic_requires_matching_sources(tmp_path, monkeypatch):
    rec = bench.committed_traffic("bwd_main_kernel")
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        doc = json.load(f)
    k = doc["kernels"]["bwd_main_kernel"]
    if rec is not None:
        assert rec[0] == k["dram_read_bytes"] + k["dram_write_bytes"]
    # A copy of the repo whose source differs must not report traffic.
    fake = tmp_path / "repo"
    (fake / "profiles").mkdir(parents=True)
    (fake / "profiles" / "traffic.json").write_text(json.dumps(doc))
    for path in k["files"]:
        dst = fake / path
        dst.parent.mkdir(parents=True, exist_ok=True)
        dst.write_bytes(open(os.path.join(ROOT, path), "rb").read() + b"\n// edit")
    monkeypatch.setattr(bench, "ROOT", str(fake))
    assert bench.committed_traffic("bwd_main_kernel") is None


def test_workload_flop_convention():
    from tiled_attention_bwd_gb300.workloads import WORKLOADS
    w = WORKLOADS["xl_4x64x4096x128_causal"]
    assert w.fwd_flops() == pytest.approx(4 * 4 * 64 * 4096 ** 2 * 128 / 2)
    assert w.bwd_flops() == pytest.approx(2.5 * w.fwd_flops())


def test_step_flops_of_the_band():
    from tiled_attention_bwd_gb300.workloads import WORKLOADS, visible_pairs
    w = WORKLOADS["xl_4x64x4096x128_causal"]
    # No window: the N^2 / 2 convention of the base workload.
    assert bench.step_flops(w, -1) == (w.fwd_flops(), w.bwd_flops())
    f, b = bench.step_flops(w, 1024)
    pairs = visible_pairs(w.N, True, 1024)
    # causal band of half-width W: row i sees min(i, W) + 1 keys
    assert pairs == sum(min(i, 1024) + 1 for i in range(w.N))
    assert f == 4.0 * w.B * w.H * w.d * pairs and b == 2.5 * f
    assert visible_pairs(10, False, 2, 3, 7) == 4 * 5


def test_reference_arm_runs_with_a_window():
    import subprocess
    import sys
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
         "reference", "--steps", "1", "--warmup", "0", "--workload",
         "small_2x8x512x64", "--window", "100", "--hkv", "2"],
        capture_output=True, text=True, timeout=300, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["window"] == 100 and line["config"]["Hkv"] == 2


def test_step_flops_with_sequence_lengths():
    from tiled_attention_bwd_gb300.workloads import WORKLOADS
    w = WORKLOADS["xl_4x64x4096x128_causal"]
    # each sequence counts its own visible pairs, L (L + 1) / 2 when causal
    # (full lengths: within 1 / N of the N^2 / 2 convention of the plain run)
    full = [w.N] * w.B
    f, _ = bench.step_flops(w, -1, full)
    assert f == pytest.approx(w.fwd_flops() * (1 + 1 / w.N))
    lens = [4096, 1, 0, 129]
    f, b = bench.step_flops(w, -1, lens)
    pairs = sum(L * (L + 1) // 2 for L in lens)
    assert f == 4.0 * w.H * w.d * pairs and b == 2.5 * f
    f, _ = bench.step_flops(w, 16, [40])
    band = sum(min(i, 16) + 1 for i in range(40))     # causal band of 17
    assert f == 4.0 * w.H * w.d * band
    drawn = bench.bench_lengths(w)
    assert drawn.dtype.is_floating_point is False and len(drawn) == w.B
    assert all(1 <= int(x) <= w.N for x in drawn)
    assert bench.bench_lengths(w).tolist() == drawn.tolist()    # seeded


def test_reference_arm_records_the_lengths():
    import subprocess
    import sys
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
         "reference", "--steps", "1", "--warmup", "0", "--workload",
         "small_2x8x512x64", "--varlen"],
        capture_output=True, text=True, timeout=300, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    from tiled_attention_bwd_gb300.workloads import WORKLOADS
    w = WORKLOADS["small_2x8x512x64"]
    assert line["config"]["seq_lens"] == bench.bench_lengths(w).tolist()


def test_varlen_and_fp8_are_exclusive():
    import subprocess
    import sys
    r = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--varlen", "--fp8",
         "--steps", "1", "--warmup", "3"],
        capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "--varlen" in (r.stderr + r.stdout)
