"""Benchmark: attention forward + backward TFLOP/s on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--hkv HKV] [--window W] [--varlen] [--fp8]
                    [--impl ours|reference] [--replicas] [--no-e2e]
                    [--no-cpu-baseline]

One step = fa_fwd + fa_bwd over the whole workload (default: 4x64x4096x128
causal, the headline shape), inputs resident in HBM.  With several GPUs each
rank takes a contiguous range of the workload's key/value groups (whole
batch entries with --varlen) and runs the plain entry points on it, with no
collective on the data path (strong scaling); --replicas runs the whole
workload on every rank instead (weak scaling).  The reported value is the
algorithmic FLOPs of all ranks divided by the slowest rank's time.  Rank 0
prints one JSON line, with per-kernel rooflines (forward, backward pre, main
and post kernels, each timed by CUDA events on the launching stream) and the
CPU oracle timed on the host cores: on a sample of this workload, on a
sample of every workload (full-workload time extrapolated), and on the
smallest workload with one core.

FLOP convention: forward = 4 B H N^2 d (halved when causal), backward = 2.5 x
forward, step = 3.5 x forward.  With --window the N^2 (or N^2 / 2) becomes
the number of visible (query, key) pairs of the band.  --hkv runs the
grouped-query variant (K/V heads shared by H / HKV query heads); it does not
change the FLOPs.  --varlen gives each batch entry its own length, drawn
uniformly from [1, N] (seeded), through fa_fwd_varlen / fa_bwd_varlen; the
FLOPs then count each sequence's own visible pairs.

--impl reference times the CPU fp64 oracle (the plain definition, no tuning)
on the host cores, each step a bounded sample of the same workload (the last
128 query rows of one head per core, forward + backward), in the same unit.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("attention fwd and fwd+bwd TFLOP/s (bf16) and % of GB300 dense "
          "BF16 peak")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return (float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained",
                                                       p["bf16_tflops"])),
                float(p["hbm_gbs"]), "measured")
    except (OSError, KeyError, ValueError):
        return (FALLBACK_BF16_TFLOPS, 1700.0, FALLBACK_HBM_GBS, "fallback")


def committed_traffic(kernel):
    """DRAM bytes per launch of `kernel` at the headline workload, from the
    committed ncu capture in profiles/traffic.json, if the kernel's sources
    still hash to the fingerprint recorded with it; else None."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)["kernels"][kernel]
        h = hashlib.sha256()
        for path in rec["files"]:
            with open(os.path.join(ROOT, path), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["fingerprint"]:
            return None
        return int(rec["dram_read_bytes"]) + int(rec["dram_write_bytes"]), rec["workload"]
    except (OSError, KeyError, ValueError):
        return None


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, device=None):
    """Max of a float over all ranks (identity for a single process)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu),
                 "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2],
                "sm_max_mhz": max(smax), "power_w_max": max(power),
                "samples": len(sm), "reasons": sorted(reasons)}


def oracle_sample(w, heads, rows, window=-1):
    """Run the CPU oracle (forward + backward) on the last `rows` query rows
    of `heads` heads of workload `w` (with a window: each head as a batch
    entry of its own, which is the per-head arithmetic of the grouped
    operation too).  Returns (algorithmic FLOPs, seconds)."""
    import oracle
    from tiled_attention_bwd_gb300.workloads import make_inputs, visible_pairs
    inp = make_inputs(1, heads, w.N, w.d, seed=w.seed, qk_mult=w.qk_mult)
    r0 = w.N - rows
    if window < 0:
        q, k, v, do = (inp[n].double().numpy()[0] for n in ("q", "k", "v", "do"))
        t0 = time.perf_counter()
        oracle.fwd_rows(q, k, v, w.causal, w.scale, r0, w.N)
        oracle.bwd_rows(q, k, v, do, w.causal, w.scale, r0, w.N)
    else:
        q, k, v, do = (inp[n].double().numpy().transpose(1, 0, 2, 3)
                       for n in ("q", "k", "v", "do"))
        t0 = time.perf_counter()
        oracle.fwd_ext(q, k, v, w.causal, w.scale, window, r0, w.N)
        oracle.bwd_ext(q, k, v, do, w.causal, w.scale, window, r0, w.N)
    dt = time.perf_counter() - t0
    pairs = float(visible_pairs(w.N, w.causal, window, r0, w.N))
    flops = heads * pairs * 4.0 * w.d * 3.5
    return flops, dt


def step_flops(w, window, lens=None):
    """Algorithmic FLOPs of one forward (and of one backward = 2.5 x); with
    per-sequence lengths, each batch entry counts its own visible pairs."""
    from tiled_attention_bwd_gb300.workloads import visible_pairs
    if lens is not None:
        pairs = sum(visible_pairs(int(L), w.causal, window) for L in lens)
        f = 4.0 * w.H * w.d * pairs
        return f, 2.5 * f
    if window < 0:
        return w.fwd_flops(), w.bwd_flops()
    f = 4.0 * w.B * w.H * w.d * visible_pairs(w.N, w.causal, window)
    return f, 2.5 * f


def slice_flops(w, window, sh, lens=None):
    """Algorithmic forward and backward FLOPs of one rank's slice `sh` of
    workload w (a HeadSlice); with per-sequence lengths the slice holds
    whole batch entries and counts their own visible pairs."""
    if lens is not None:
        return step_flops(w, window, lens[sh.b_lo:sh.b_hi])
    f, b = step_flops(w, window, None)
    frac = (sh.q_hi - sh.q_lo) / float(w.B * w.H)
    return f * frac, b * frac


def bench_lengths(w):
    """Per-sequence lengths of --varlen: uniform over [1, N], seeded."""
    from tiled_attention_bwd_gb300.workloads import make_seq_lens
    return make_seq_lens(w.B, w.N, seed=w.seed)


def variant_config(w, args):
    """config keys of the grouped-head / window variant (empty if none)."""
    c = {}
    if args.hkv is not None:
        c["Hkv"] = args.hkv
    if args.window >= 0:
        c["window"] = args.window
    if args.varlen:
        c["seq_lens"] = [int(x) for x in bench_lengths(w)]
        c["seq_lens_recipe"] = "uniform over [1, N], seed = workload seed"
    return c


def run_reference(args, w, rank, world):
    """CPU oracle arm: rank 0 only; other ranks exit without work."""
    if rank != 0:
        return
    import oracle
    cores = oracle.num_threads()
    rows = 128
    for _ in range(args.warmup):
        oracle_sample(w, cores, rows, args.window)
    total_flops, total_s = 0.0, 0.0
    for _ in range(args.steps):
        f, s = oracle_sample(w, cores, rows, args.window)
        total_flops += f
        total_s += s
    value = total_flops / total_s / 1e12
    sample = ("last %d query rows of %d heads (one per core) of %s, fwd+bwd, "
              "per step" % (rows, cores, w.name))
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": dict({"workload": w.name, "B": w.B, "H": w.H, "N": w.N,
                        "d": w.d, "causal": w.causal},
                       **variant_config(w, args)),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def pre_post_bytes(B, H, Hkv, N, d, lens=None):
    """Algorithmic DRAM bytes of the backward's two row passes (None with
    per-sequence lengths).  pre: reads O, dO (2 d bytes each per row) and
    LSE (4), writes D and -LSE log2 e (4 + 4 per padded row) and clears the
    fp32 dQ accumulator (4 d); with a key/value group split over blocks (more
    than 8 query heads per key/value head) also clears the fp32 dK, dV
    accumulators.  post: reads the dQ accumulator (4 d), writes dQ (2 d);
    with a split group also reads the dK, dV accumulators, writes dK, dV."""
    if lens is not None:
        return None, None
    rows = B * H * N
    n_pad = (N + 127) // 128 * 128
    kv_rows = B * Hkv * N if H // Hkv > 8 else 0
    pre = rows * (4 * d + 4 + 4 * d) + B * H * n_pad * 8 + kv_rows * 8 * d
    post = rows * 6 * d + kv_rows * 12 * d
    return float(pre), float(post)


def oracle_whole_heads(w, heads, window=-1):
    """Oracle forward + backward on `heads` whole heads (every row) of
    workload w, in the order of the workload's own inputs.  Returns
    (algorithmic FLOPs, seconds)."""
    import oracle
    from tiled_attention_bwd_gb300.workloads import make_inputs, visible_pairs
    inp = make_inputs(w.B, w.H, w.N, w.d, seed=w.seed, qk_mult=w.qk_mult)
    flat = {n: inp[n].reshape(w.B * w.H, w.N, w.d)[:heads].double().numpy()
            for n in ("q", "k", "v", "do")}
    del inp
    t0 = time.perf_counter()
    oracle.fwd(flat["q"], flat["k"], flat["v"], w.causal, w.scale)
    oracle.bwd(flat["q"], flat["k"], flat["v"], flat["do"], w.causal, w.scale)
    dt = time.perf_counter() - t0
    pairs = float(visible_pairs(w.N, w.causal, window))
    return heads * pairs * 4.0 * w.d * 3.5, dt


def cpu_baselines(w, window):
    """The oracle timed on the host: the workload's own sample (`main`),
    every workload on a bounded sample of whole heads with the full-workload
    time extrapolated (`configs`), and the smallest workload on one core."""
    import oracle
    from tiled_attention_bwd_gb300.workloads import WORKLOADS, visible_pairs
    cores = oracle.num_threads()
    heads = min(w.B * w.H, 2 * cores)
    f, s_ = oracle_sample(w, heads, w.N, window)
    main = {"value": f / s_ / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": "all %d query rows of %d heads of %s, fwd+bwd, %.1f s"
                      % (w.N, heads, w.name, s_)}
    configs = []
    for c in WORKLOADS.values():
        per_head = visible_pairs(c.N, c.causal, -1) * 4.0 * c.d * 3.5
        hs = int(max(1, min(c.B * c.H, round(6e10 / per_head))))
        f, s_ = oracle_whole_heads(c, hs)
        configs.append({
            "workload": c.name, "value": f / s_ / 1e12, "unit": "TFLOP/s",
            "cores": cores, "heads_sampled": hs, "heads_total": c.B * c.H,
            "seconds": s_,
            "full_workload_seconds": s_ * (c.B * c.H) / hs,
            "full_workload_seconds_kind": ("measured" if hs == c.B * c.H
                                           else "extrapolated")})
    small = WORKLOADS["small_2x8x512x64"]
    oracle.set_num_threads(1)
    try:
        f, s_ = oracle_whole_heads(small, small.B * small.H)
    finally:
        oracle.set_num_threads(cores)
    one = {"workload": small.name, "value": f / s_ / 1e12, "unit": "TFLOP/s",
           "cores": 1, "seconds": s_, "heads": small.B * small.H,
           "sample": "the whole workload, fwd+bwd"}
    return main, configs, one


def run_ours(args, w, rank, world, local):
    import torch
    from tiled_attention_bwd_gb300 import (fa_bwd_ext, fa_bwd_set_phase_events,
                                           fa_bwd_ext_workspace_size,
                                           fa_bwd_varlen,
                                           fa_check_device_status, fa_fwd_ext,
                                           fa_fwd_varlen, load_library)
    from tiled_attention_bwd_gb300.shard import (full_slice, head_slice,
                                                 slice_heads)
    from tiled_attention_bwd_gb300.workloads import make_grouped_inputs

    load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak_burst, peak_sust, hbm_peak, peak_src = load_peaks()

    # fa_fwd / fa_bwd are fa_fwd_ext / fa_bwd_ext with Hkv = H and no
    # window; the same draw order makes Hkv = H identical to the base inputs.
    hkv = w.H if args.hkv is None else args.hkv
    window = args.window
    inp_cpu = make_grouped_inputs(w.B, w.H, hkv, w.N, w.d, w.seed, w.qk_mult)
    lens_all = bench_lengths(w) if args.varlen else None
    # This rank's share: whole key/value groups (whole batch entries with
    # lengths) of the one problem, or, with --replicas, all of it.
    if args.replicas or world == 1:
        sh = full_slice(w.B, w.H, hkv)
    else:
        sh = head_slice(rank, world, w.B, w.H, hkv, by_batch=args.varlen)
    Bs, Hs, Hkvs = sh.B_s, sh.H_s, sh.Hkv_s
    part = {n: slice_heads(inp_cpu[n], sh.q_lo, sh.q_hi, Bs) if n in ("q", "do")
            else slice_heads(inp_cpu[n], sh.kv_lo, sh.kv_hi, Bs)
            for n in ("q", "k", "v", "do")}
    part = {n: t.contiguous() for n, t in part.items()}
    del inp_cpu
    q, k, v, do = (part[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq = torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(1, fa_bwd_ext_workspace_size(Bs, Hs, Hkvs, w.N, w.d)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    lens_cpu = lens_all[sh.b_lo:sh.b_hi] if args.varlen else None
    sl = lens_cpu.to(dev) if args.varlen else None
    # FLOPs of the whole problem (all ranks) and of this rank's share.
    fwd_all, bwd_all = step_flops(w, window, lens_all)
    if args.replicas:
        fwd_all, bwd_all = world * fwd_all, world * bwd_all
    fwd_flops, bwd_flops = slice_flops(w, window, sh, lens_all)
    idle = sh.empty

    def fwd():
        if idle:
            return
        if sl is None:
            fa_fwd_ext(q, k, v, w.causal, w.scale, window, out=o, lse=lse)
        else:
            fa_fwd_varlen(q, k, v, sl, w.causal, w.scale, window, out=o,
                          lse=lse)

    def bwd():
        if idle:
            return
        if sl is None:
            fa_bwd_ext(q, k, v, o, lse, do, w.causal, w.scale, window, dq=dq,
                       dk=dk, dv=dv, workspace=ws)
        else:
            fa_bwd_varlen(q, k, v, o, lse, do, sl, w.causal, w.scale, window,
                          dq=dq, dk=dk, dv=dv, workspace=ws)

    def step():
        fwd()
        bwd()

    for _ in range(args.warmup):
        step()
    if fa_check_device_status(dev) != 0:
        raise RuntimeError("device status error during warm-up")

    # -------- timed region.  Two sets of K steps, each step bracketed by
    # its own pair of events on the launching stream.  The first set has
    # nothing else between the four launches and gives the step time; the
    # second also records an event after the forward call and two around
    # the main backward kernel (the library records those two), which time
    # every launch on its own but sit between the kernels (so they add
    # their own cost and keep a kernel from being scheduled behind the one
    # before it).  By default each step is one CUDA graph, captured once per
    # step and set (so every step records its own events): a replay submits
    # the launches at once and no host time falls inside a step.  When the
    # step's inputs (Q, K, V, dO) are smaller than twice L2, a buffer of
    # twice L2 is written before every step, outside its events.
    K = args.steps
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do))
    flush = (torch.empty(max(1, l2 // 2), dtype=torch.float32, device=dev)
             if in_bytes < 2 * l2 else None)
    use_graph = not args.no_graph
    graph_note = None

    def new_event():
        if use_graph:
            return torch.cuda.Event(enable_timing=True, external=True)
        return torch.cuda.Event(enable_timing=True)
    try:
        step_ev = [(new_event(), new_event()) for _ in range(K)]
    except TypeError:            # a torch without external events
        use_graph, graph_note = False, "torch.cuda.Event has no 'external'"
        step_ev = [(new_event(), new_event()) for _ in range(K)]
    ph_ev = [(new_event(), new_event()) for _ in range(K)]
    fwd_end = [new_event() for _ in range(K)]
    main_ev = [(new_event(), new_event()) for _ in range(K)]
    # torch creates the CUDA event lazily and only times events it recorded
    # itself: record each once here; the library re-records them later.
    for a, b in main_ev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)

    def plain_step(i):
        s_ = torch.cuda.current_stream(dev)
        step_ev[i][0].record(s_)
        fwd()
        bwd()
        step_ev[i][1].record(s_)

    def phase_step(i):
        s_ = torch.cuda.current_stream(dev)
        fa_bwd_set_phase_events(*main_ev[i])
        try:
            ph_ev[i][0].record(s_)
            fwd()
            fwd_end[i].record(s_)
            bwd()
            ph_ev[i][1].record(s_)
        finally:
            fa_bwd_set_phase_events(None, None)

    runs = {"plain": plain_step, "phase": phase_step}
    if use_graph:
        try:
            graphs = {}
            for name, fn in runs.items():
                graphs[name] = []
                for i in range(K):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, capture_error_mode="thread_local"):
                        fn(i)
                    graphs[name].append(g)
            for _ in range(args.warmup):
                graphs["plain"][0].replay()
            torch.cuda.synchronize(dev)
            runs = {name: (lambda i, gs=gs: gs[i].replay())
                    for name, gs in graphs.items()}
        except RuntimeError as ex:
            use_graph = False
            graph_note = "capture failed: %s" % str(ex).splitlines()[0]
    if fa_check_device_status(dev) != 0:
        raise RuntimeError("device status error in the graph warm-up")

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    for name in ("plain", "phase"):
        for i in range(K):
            if flush is not None:
                flush.fill_(float(i))
            runs[name](i)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    if fa_check_device_status(dev) != 0:
        raise RuntimeError("device status error in the timed region")

    def mean_ms(pairs):
        return sum(a.elapsed_time(b) for a, b in pairs) / K
    step_ms_local = mean_ms(step_ev)
    phase_step_ms = mean_ms(ph_ev)
    fwd_ms_local = mean_ms([(ph_ev[i][0], fwd_end[i]) for i in range(K)])
    if idle:
        main_ms = pre_ms = post_ms = 0.0
    else:
        main_ms = mean_ms(main_ev)
        pre_ms = mean_ms([(fwd_end[i], main_ev[i][0]) for i in range(K)])
        post_ms = mean_ms([(main_ev[i][1], ph_ev[i][1]) for i in range(K)])
    step_ms = max_over_ranks(step_ms_local, world, dev)
    fwd_ms = max_over_ranks(fwd_ms_local, world, dev)
    del runs

    def ev_pair():
        return (torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True))

    # -------- FP8 forward (optional): Q, K quantised to E4M3 inside the call
    fp8 = None
    if args.fp8 and not idle:
        from tiled_attention_bwd_gb300 import fa_fwd_fp8, fa_fwd_fp8_workspace_size
        ws8 = torch.empty(fa_fwd_fp8_workspace_size(Bs, Hs, w.N, w.d),
                          dtype=torch.uint8, device=dev)
        for _ in range(max(3, args.warmup)):
            fa_fwd_fp8(q, k, v, w.causal, w.scale, out=o, lse=lse, workspace=ws8)
        torch.cuda.synchronize(dev)
        f8_s, f8_e = ev_pair()
        f8_s.record(stream)
        for _ in range(K):
            fa_fwd_fp8(q, k, v, w.causal, w.scale, out=o, lse=lse, workspace=ws8)
        f8_e.record(stream)
        torch.cuda.synchronize(dev)
        if fa_check_device_status(dev) != 0:
            raise RuntimeError("device status error in the FP8 forward")
        f8_ms = max_over_ranks(f8_s.elapsed_time(f8_e) / K, world, dev)
        fp8 = {"value": fwd_all / (f8_ms * 1e-3) / 1e12,
               "unit": "TFLOP/s", "ms": f8_ms,
               "note": "fa_fwd_fp8: E4M3 quantisation of Q and K (two "
                       "launches) + forward with Q K^T on FP8 tensor cores; "
                       "same FLOP convention as fwd"}

    # -------- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        host = {n: part[n].pin_memory() for n in ("q", "k", "v", "do")}
        outs = {n: torch.empty_like(host["q" if n in ("o", "dq") else "k"]).pin_memory()
                for n in ("o", "dq", "dk", "dv")}
        lse_h = torch.empty(tuple(q.shape[:3]), dtype=torch.float32).pin_memory()

        if sl is not None:
            host["seq_lens"] = lens_cpu.pin_memory()
        if variant_config(w, args):
            # grouped heads / window / lengths: copies and compute in turn
            mode = "serial copies around the fa_*_ext or fa_*_varlen calls"

            def e2e_step():
                for n, t in (("q", q), ("k", k), ("v", v), ("do", do)):
                    t.copy_(host[n], non_blocking=True)
                if sl is not None:
                    sl.copy_(host["seq_lens"], non_blocking=True)
                step()
                for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
                    outs[n].copy_(t, non_blocking=True)
                lse_h.copy_(lse, non_blocking=True)
        else:
            # fa_step_host: chunks of heads, copies in both directions
            # overlapped with each other and with the kernels
            from tiled_attention_bwd_gb300 import (fa_step_host,
                                                   fa_step_host_scratch_size)
            mode = "fa_step_host (pinned host buffers, pipelined by head chunks)"
            scratch = torch.empty(
                max(1, fa_step_host_scratch_size(Bs, Hs, w.N, w.d,
                                                 args.chunk_heads)),
                dtype=torch.uint8, device=dev)

            def e2e_step():
                if idle:
                    return
                fa_step_host(host["q"], host["k"], host["v"], host["do"],
                             w.causal, w.scale, outs["o"], lse_h, outs["dq"],
                             outs["dk"], outs["dv"], scratch=scratch,
                             chunk_heads=args.chunk_heads, device=dev)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        s, e = ev_pair()
        K_e2e = max(3, K // 4)
        s.record(stream)
        for _ in range(K_e2e):
            e2e_step()
        e.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_ms = max_over_ranks(s.elapsed_time(e) / K_e2e, world, dev)
        h2d = sum(host[n].numel() * host[n].element_size() for n in host)
        d2h = (sum(outs[n].numel() * outs[n].element_size() for n in outs)
               + lse_h.numel() * 4)
        e2e = {"value": (fwd_all + bwd_all) / (e2e_ms * 1e-3) / 1e12,
               "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "mode": mode}

    plain = not variant_config(w, args)

    def traffic_of(kernel):
        t = committed_traffic(kernel)
        return (t[0] if t and t[1] == w.name and plain and world == 1
                else None)

    value = (fwd_all + bwd_all) / (step_ms * 1e-3) / 1e12
    fwd_tflops = fwd_all / (fwd_ms * 1e-3) / 1e12
    pre_b, post_b = pre_post_bytes(Bs, Hs, Hkvs, w.N, w.d, lens_cpu)

    def tensor_roof(kernel, flop, ms, peak, peak_note):
        a_ = flop / (ms * 1e-3) / 1e12 if ms > 0 else None
        return {"kernel": kernel, "bound": "tensor", "achieved": a_,
                "peak": peak, "unit": "TFLOP/s",
                "frac": a_ / peak if a_ is not None else None,
                "peak_source": peak_note, "ms_per_launch": ms,
                "traffic": traffic_of(kernel),
                "traffic_unit": "bytes per launch (ncu dram read+write)",
                "algorithmic_flop_per_launch": flop}

    def hbm_roof(kernel, nbytes, ms):
        if nbytes is None or ms <= 0:
            return None
        a_ = nbytes / (ms * 1e-3) / 1e9
        return {"kernel": kernel, "bound": "hbm", "achieved": a_,
                "peak": hbm_peak, "unit": "GB/s", "frac": a_ / hbm_peak,
                "peak_source": "%s copy bandwidth" % peak_src,
                "ms_per_launch": ms, "traffic": traffic_of(kernel),
                "traffic_unit": "bytes per launch (ncu dram read+write)",
                "algorithmic_bytes_per_launch": nbytes}

    burst_note = ("%s bf16 burst (each kernel is timed per launch at the "
                  "maximum clock, not in a power-capped loop)" % peak_src)
    roofline = tensor_roof("bwd_main_kernel", bwd_flops, main_ms, peak_burst,
                           burst_note)
    rooflines = {
        "fwd_kernel": tensor_roof("fwd_kernel", fwd_flops, fwd_ms_local,
                                  peak_burst, burst_note),
        "bwd_pre_kernel": hbm_roof("bwd_pre_kernel", pre_b, pre_ms),
        "bwd_post_kernel": hbm_roof("bwd_post_kernel", post_b, post_ms),
    }

    cpu = cpu_configs = cpu_one = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu, cpu_configs, cpu_one = cpu_baselines(w, window)

    if rank != 0:
        return
    if args.replicas:
        per_gpu, scaling = "full workload per rank (replicas)", "weak"
    else:
        per_gpu = ("contiguous key/value groups of the one workload per rank"
                   if not args.varlen else
                   "contiguous batch entries of the one workload per rank")
        scaling = "strong"
    l2_note = ("L2 flushed before every step (a %d MB write; the step's "
               "Q, K, V, dO total %d MB, L2 %d MB)"
               % (2 * l2 // 2**20, in_bytes // 2**20, l2 // 2**20)
               if flush is not None else
               "inputs larger than L2 (Q, K, V, dO total %d MB, L2 %d MB)"
               % (in_bytes // 2**20, l2 // 2**20))
    timing_note = (("one CUDA graph per step (fwd + bwd calls captured), "
                    "events inside the graph" if use_graph else
                    "eager calls, events on the stream"
                    + ("" if graph_note is None else " (%s)" % graph_note))
                   + "; ms_per_step from steps with events only at their "
                   "ends, the per-kernel times (bwd_ms, rooflines) from a "
                   "second set of K steps with events between the kernels")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": scaling,
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict({"workload": w.name, "B": w.B, "H": w.H, "N": w.N,
                        "d": w.d, "causal": w.causal, "scale": w.scale,
                        "qk_mult": w.qk_mult,
                        "per_gpu": per_gpu,
                        "l2": l2_note,
                        "timing": timing_note},
                       **variant_config(w, args)),
        "fwd": {"value": fwd_tflops, "unit": "TFLOP/s", "ms": fwd_ms,
                "frac_of_peak": fwd_tflops / world / peak_burst},
        "fwd_bwd_frac_of_peak": value / world / peak_burst,
        "peak": {"bf16_tflops": peak_burst, "bf16_tflops_sustained": peak_sust,
                 "hbm_gbs": hbm_peak, "source": peak_src},
        "roofline": roofline,
        "rooflines": rooflines,
        "bwd_ms": {"pre": pre_ms, "main": main_ms, "post": post_ms},
        "ms_per_step_with_kernel_events": phase_step_ms,
        "cpu_baseline": cpu,
        "cpu_baseline_configs": cpu_configs,
        "cpu_baseline_1core": cpu_one,
        "e2e": e2e,
        "fwd_fp8": fp8,
        "gpu_launches": 8 * K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    from tiled_attention_bwd_gb300.workloads import HEADLINE, WORKLOADS
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--hkv", type=int, default=None,
                    help="key/value heads (divides H; default H)")
    ap.add_argument("--window", type=int, default=-1,
                    help="sliding window |i - j| <= W (default: none)")
    ap.add_argument("--chunk-heads", type=int, default=0,
                    help="heads per chunk of the host-buffer step (0: B*H/16)")
    ap.add_argument("--varlen", action="store_true",
                    help="per-sequence lengths, uniform over [1, N]")
    ap.add_argument("--fp8", action="store_true",
                    help="also time the FP8 forward (fa_fwd_fp8)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--replicas", action="store_true",
                    help="with several GPUs, run the whole workload on every "
                         "rank instead of splitting its heads")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager calls instead of one CUDA graph per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        raise SystemExit("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.hkv is not None and (args.hkv < 1 or w.H % args.hkv != 0):
        raise SystemExit("--hkv must divide H = %d" % w.H)
    if args.varlen and args.fp8:
        raise SystemExit("--varlen has no FP8 forward")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        run_ours(args, w, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
