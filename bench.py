"""Benchmark of the CSA2 decode step: 1M-token context, 20-layer stack.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
               [--workload 1m|128k|group3|prefill|tiny] [--no-graph]

Workload (default "1m"): batch 8, N = 262144 compressed entries per
sequence (1M tokens at 4 tokens per entry), layer schedule (Full, Reindex,
Reuse, Reuse) x 5, indexer 64 heads x 128 (E4M3 keys, bf16 queries), top-512,
64 heads x 512 FP4-E2M1 main KV, 128-row bf16 window; seeded synthetic data.
A step is one decode step through all 20 layers (csa2_layer_stack), replayed
from a CUDA graph.  One JSON line is printed by rank 0.

N > 1 (torchrun): every rank runs its own replica of the workload (decode
sequences are independent; no data-path collective), so per-GPU work is
fixed ("weak" scaling); value = tokens of all ranks / max-over-ranks time.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode µs/layer & tokens/s at 1M ctx; HBM GB/s vs ~8 TB/s peak"
L2_BYTES = 126 << 20          # B300 L2
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, device="cpu"):
    """Max of a float over all ranks (the slowest rank sets the job time)."""
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world, device="cpu"):
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- peaks, clocks

def measured_peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, which): the machine's measured copy
    bandwidth and cuBLAS bf16 rate, else the recipe's fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6400.0, 1800.0, "fallback"


# E4M3 dense tensor rate over bf16 dense (nominal 4.5 / 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        sm = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def workload_desc(wl):
    """The workload as both arms name it in `config`."""
    pool = f", candidate pool {wl.pool}" if wl.pool else ""
    if wl.page_rows:
        pool += f", paged caches ({wl.page_rows}-entry pages, shuffled block table)"
    if wl.block:
        pool += f", block-level pruning (blocks of {wl.block}, {wl.blocks_kept} kept)"
    q = "" if wl.q_per_seq == 1 else f", {wl.q_per_seq} queries per sequence"
    return (f"{wl.name}: B={wl.B}, N={wl.N}{q}, layers={len(wl.modes)} "
            f"{''.join('FIU'[m] for m in wl.modes)}, indexer {wl.Hi}x{wl.Di} "
            f"{'fp32' if wl.fp32_indexer else 'E4M3'}, top-{wl.k}{pool}, {wl.Hq} heads x {wl.D} "
            f"FP4 KV, window {wl.W} bf16")


# ---------------------------------------------------------------- our arm

def prefill_selects(wl):
    """Whether the layer stack selects this prefill chunk's top-k without its
    score matrix (sampled threshold, candidates, exact selection among them)."""
    return (wl.q_per_seq > 1 and wl.q_per_seq % 4 == 0 and wl.N > 4096 and not wl.pool
            and not wl.block and not wl.fp32_indexer and wl.Hi == 64 and wl.Di == 128
            and wl.k <= 8192)


def fuses_new_rows(wl):
    """Whether a decode Full layer's indexer launch also quantises the step's
    new cache rows (E4M3 keys, one query per sequence, 256-element KV parts,
    no block-level pruning)."""
    return (not wl.fp32_indexer and wl.q_per_seq == 1 and wl.Hi == 64 and wl.Di == 128
            and wl.D % 256 == 0 and not wl.block)


def launches_per_step(wl):
    """Kernels of this library per step (memsets are not counted).  Full:
    new-row quantiser, indexer score, top-k selection and attention; Reindex:
    the same without the new rows; Reuse: attention.  Decode indexer launches
    quantise their queries (and a Full layer's new rows) inside the indexer
    kernel; a prefill chunk runs
    the indexer-Q quantiser as its own kernel and a top-k histogram pass per
    index layer (decode builds the histogram inside the indexer kernel), or,
    when it selects without the score matrix, the kernels of that selection.
    Attention over more than 8 key chunks of 80 adds a merge kernel.  With a
    candidate pool a Full layer selects the pool and then the top-k inside it
    (one kernel more) and a Reindex layer runs the Q quantiser, the pooled
    scores, their selection and attention."""
    # a decode Full layer on the plain path quantises its new rows inside its
    # indexer launch
    per = {0: 3 if fuses_new_rows(wl) else 4, 1: 3, 2: 1}
    n = 0
    for m in wl.modes:
        if wl.block and m == 0:
            # new rows, their block keys, Q quantiser, block scores, block
            # selection (expanded to the pool), pooled scores, selection, attention
            n += 8
        elif m == 1 and (wl.pool or wl.block):
            n += 4  # Q quantiser, pooled scores, their selection, attention
        else:
            n += per[m]
            if m == 0 and wl.pool:
                n += 1  # the pool's selection, then the top-k inside it
            if m != 2 and wl.q_per_seq > 1 and prefill_selects(wl):
                # Q quantiser, sampled scores, two histogram passes and two
                # threshold kernels, the emitting scores; the candidate
                # selector takes the top-k's place
                n += 6
            elif m != 2 and wl.q_per_seq > 1:
                n += 2  # separate Q quantiser, histogram pass
            elif m != 2 and wl.fp32_indexer and wl.N > 4096:
                n += 1  # the fp32 indexer builds no histogram: a histogram pass
        if (wl.k + wl.W + 79) // 80 > 8:
            n += 1
    return n


class L2Flush:
    """Empties L2 between timed iterations: writes a buffer four times the L2,
    then reads another of the same size, so that the lines left in L2 are
    clean.  Without the read the next timed kernel would first write back
    ~126 MB of the flush's own dirty lines (5-12 us measured on a 268 MB
    read stream), work that is not the kernel's."""

    def __init__(self, device="cuda"):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def index_launch_form(wl):
    """How the timed indexer launch takes its queries: "f32" (the CUDA-core
    fp32 indexer), "bf16" (decode: bf16 queries quantised inside the launch,
    the form the layer stack runs) or "q8" (a prefill chunk: queries
    quantised beforehand, so the launch holds only the indexer kernel)."""
    if wl.fp32_indexer:
        return "f32"
    return "bf16" if wl.q_per_seq % 4 != 0 else "q8"


def index_launch_bytes(W):
    """Algorithmic bytes of one timed indexer launch: the keys, the queries
    in the form the launch reads them, the head weights and, over paged
    caches, the block table."""
    wl = W.wl
    q_bytes = {"f32": 4, "bf16": 2, "q8": 1}[index_launch_form(wl)]
    n = W.indexer_bytes_per_layer() + wl.nq * wl.Hi * (wl.Di * q_bytes + 4)
    if wl.page_rows:
        n += wl.B * (-(-wl.N // wl.page_rows)) * 4
    return n


def time_index_kernel(csa2, W, flush, reps=20):
    """Average device time of one launch of the indexer kernel (FP8 tensor
    core, or fp32 CUDA cores for an fp32 indexer) on the workload's first Full
    layer, one kernel per launch (see index_launch_form), with L2 flushed
    before each launch.  A prefill chunk that the stack selects without its
    score matrix is timed in that form (csa2_index_candidates)."""
    L0 = W.layers[0]
    wl = W.wl
    if index_launch_form(wl) == "q8":
        q, c = csa2.quantize_index_q(L0["idx_q"], L0["idx_w"])
    else:
        q, c = L0["idx_q"], L0["idx_w"]
    kw = {} if W.pages is None else {"pages": W.pages, "n": wl.N}
    scores = torch.empty(wl.nq, wl.N, dtype=torch.float32, device=q.device)
    for _ in range(3):
        csa2.index_score(q, c, L0["idxk"], wl.q_per_seq, W.n_valid, scores, **kw)
    launch = lambda: csa2.index_score(q, c, L0["idxk"], wl.q_per_seq, W.n_valid, scores, **kw)
    if wl.q_per_seq > 1 and prefill_selects(wl):
        # the pass the stack runs: no score matrix, the candidates at or above
        # each query's threshold; thresholds at the key of each query's 8k-th
        # largest score, the candidate volume of the stack's sampled threshold
        kth = torch.topk(scores, 8 * wl.k, dim=1).values[:, -1].contiguous()
        u = kth.view(torch.int32).clone()
        u[u == -2147483648] = 0  # -0 counts as +0
        theta = torch.where(u < 0, ~u, u ^ -2147483648)
        cap = 8192
        cand = torch.empty(wl.nq, cap, dtype=torch.int64, device=q.device)
        cnt = torch.zeros(wl.nq, dtype=torch.int32, device=q.device)
        del scores

        def launch():
            csa2.index_candidates(q, c, L0["idxk"], theta, cap, wl.q_per_seq, W.n_valid, cand,
                                  cnt, **kw)
        for _ in range(3):
            cnt.zero_()
            launch()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        flush()
        if wl.q_per_seq > 1 and prefill_selects(wl):
            cnt.zero_()
        a.record(stream)
        launch()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / reps * 1e-3  # seconds


def run_ours(args, world, rank, local):
    from long_context_sparse_27_b300 import csa2, synth
    from long_context_sparse_27_b300.workload import StackWorkload

    torch.cuda.set_device(local)
    wl = synth.WORKLOADS[args.workload]
    W = StackWorkload(wl, seed=100 + rank, gen_device="cuda")
    flush = L2Flush()
    stream = torch.cuda.current_stream()

    # warm-up (also sets kernel attributes before any capture)
    for _ in range(max(args.warmup, 3)):
        W.run()
    torch.cuda.synchronize()
    assert int(W.dev_status.item()) == 0, "device status set during warm-up"

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            W.run()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()

    def step():
        if graph is not None:
            graph.replay()
        else:
            W.run()

    # ---- device-timed steps (L2 flushed before each, outside the events)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for a, b in ev:
            flush()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    dev_s = sum(a.elapsed_time(b) for a, b in ev) * 1e-3
    assert int(W.dev_status.item()) == 0, "device status set during the timed steps"
    t_max = max_over_ranks(dev_s, world, "cuda")

    # ---- end to end: pinned host inputs -> device, step, outputs -> host.
    # Each step's inputs sit in one device block and its outputs in another
    # (one copy each way); two such block pairs alternate, so the copy in of
    # step s + 1 and the copy out of step s - 1 run on their own streams
    # while step s computes, as a serving loop would run them.  Every step's
    # copies are inside the timed region (first copy in .. last copy out).
    ios = [W.make_io() for _ in range(2)]
    host_in = torch.empty(ios[0].dev_in.numel(), dtype=torch.uint8, pin_memory=True)
    host_in.copy_(ios[0].dev_in)
    host_out = [torch.empty(io.dev_out.numel(), dtype=torch.uint8, pin_memory=True) for io in ios]
    io_graphs = []
    for io in ios:
        def run_io(io=io):
            csa2.layer_stack(io.descs, W.sargs, W.workspace)
        run_io()
        torch.cuda.synchronize()
        if args.no_graph:
            io_graphs.append(run_io)
        else:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                run_io()
            io_graphs.append(g.replay)
    torch.cuda.synchronize()
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in ios]
    computed = [torch.cuda.Event() for _ in ios]
    out_read = [torch.cuda.Event() for _ in ios]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    # a step whose bytes do not exceed L2 twice over is flushed out of it
    # before every step here too (inside the timed region)
    flush_e2e = W.algorithmic_bytes() < 2 * L2_BYTES
    barrier(world)
    torch.cuda.synchronize()
    e_start.record(h2d_stream)
    for st in range(args.steps):
        i = st % 2
        io = ios[i]
        with torch.cuda.stream(h2d_stream):
            if st >= 2:
                h2d_stream.wait_event(computed[i])  # step st - 2 no longer reads block i
            io.dev_in.copy_(host_in, non_blocking=True)
            in_ready[i].record(h2d_stream)
        stream.wait_event(in_ready[i])
        if st >= 2:
            stream.wait_event(out_read[i])  # step st - 2's outputs have left block i
        if flush_e2e:
            flush()
        io_graphs[i]()
        computed[i].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(computed[i])
            host_out[i].copy_(io.dev_out, non_blocking=True)
            out_read[i].record(d2h_stream)
    e_end.record(d2h_stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(e_start.elapsed_time(e_end) * 1e-3, world, "cuda")
    assert int(W.dev_status.item()) == 0, "device status set during the end-to-end steps"
    # the outputs that came back are the device-timed steps' outputs, byte for byte
    last = (args.steps - 1) % 2
    for l, L in enumerate(W.layers):
        off = ios[last].layers[l]["out"].data_ptr() - ios[last].dev_out.data_ptr()
        got = host_out[last][off:off + L["out"].numel() * L["out"].element_size()]
        assert torch.equal(got, L["out"].contiguous().view(torch.uint8).flatten().cpu()), \
            f"end-to-end output of layer {l} differs from the device-timed step"
    h2d_bytes, d2h_bytes = ios[0].in_bytes, ios[0].out_bytes

    # ---- dominant kernel, timed live (roofline)
    k_s = time_index_kernel(csa2, W, flush)
    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    k_bytes = index_launch_bytes(W)
    if wl.q_per_seq > 1:
        # a prefill chunk: the indexer is a dense FP8 contraction; algorithmic
        # FLOPs = 2 * Hi * Di per visible (query, entry) pair (causal)
        k_flops = 2.0 * wl.Hi * wl.Di * W.visible_pairs()
        fp8_peak = bf16_peak * FP8_OVER_BF16
        roofline = {
            "kernel": "idx_score_tc_kernel", "bound": "tensor",
            "achieved": round(k_flops / k_s / 1e12, 1), "peak": round(fp8_peak, 1),
            "peak_kind": f"{peak_kind} bf16 x {FP8_OVER_BF16:g} (E4M3 / bf16 nominal)",
            "unit": "TFLOP/s", "frac": round(k_flops / k_s / 1e12 / fp8_peak, 4),
            "traffic": None, "avg_launch_us": round(k_s * 1e6, 3), "flops_per_launch": k_flops,
        }
    else:
        roofline = {
            "kernel": "idx_score_f32_kernel" if wl.fp32_indexer else "idx_score_tc_kernel",
            "bound": "hbm",
            "achieved": round(k_bytes / k_s / 1e9, 1), "peak": hbm_peak, "peak_kind": peak_kind,
            "unit": "GB/s", "frac": round(k_bytes / k_s / 1e9 / hbm_peak, 4), "traffic": None,
            "avg_launch_us": round(k_s * 1e6, 3), "bytes_per_launch": k_bytes,
        }

    tokens = wl.nq * args.steps * world
    value = tokens / t_max
    ms_per_step = t_max / args.steps * 1e3
    n_layers = len(wl.modes)
    alg = W.algorithmic_bytes()
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "us_per_layer": round(ms_per_step * 1e3 / n_layers, 3),
        "hbm_gbs_algorithmic": round(alg / (t_max / args.steps) / 1e9, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic (seeded N(0,1); planted indexer keys)",
        "config": {
            "workload": workload_desc(wl),
            "l2": ("inputs larger than L2 (%.2f GB per step); L2 flushed before every "
                   "device-timed step (512 MB written, then 512 MB read so the lines left are "
                   "clean), not in the pipelined end-to-end loop" % (alg / 1e9))
                  if alg >= 2 * L2_BYTES else
                  ("inputs smaller than L2 (%.2f GB per step); L2 flushed before every step "
                   "(512 MB written, then 512 MB read), device-timed and end-to-end"
                   % (alg / 1e9)),
            "graph": graph is not None,
            "parallelism": f"replicas x{world}",
        },
        "algorithmic_bytes_per_step": alg,
        "roofline": roofline,
        "e2e": {
            "value": round(wl.nq * args.steps * world / e2e_s, 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": h2d_bytes,
            "d2h_bytes_per_step": d2h_bytes,
            "note": ("host-to-device per step: new KV and indexer-K rows, indexer Q and weights, "
                     "attention Q; the caches and the sliding-window rows stay on the device "
                     "(a step's new window rows, %d bytes, are not copied)"
                     % (len(wl.modes) * wl.B * (1 if wl.q_per_seq == 1 else wl.q_per_seq)
                        * wl.D * 2)),
        },
        "gpu_launches": launches_per_step(wl) * args.steps,
        "clocks": clk.summary(),
    }
    # DRAM bytes of one indexer launch from the committed ncu summary, when it
    # was taken on this workload's indexer launch shape
    traffic = os.path.join(ROOT, "profiles", "idx_score_tc_traffic.txt")
    if os.path.exists(traffic):
        kv = {}
        with open(traffic) as f:
            for ln in f:
                if ":" in ln and not ln.startswith("#"):
                    key, val = ln.split(":", 1)
                    kv[key.strip()] = val.strip()
        if kv.get("workload") == wl.name and "bytes_per_launch" in kv:
            line["roofline"]["traffic"] = int(kv["bytes_per_launch"])
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget_s)
    return line


# ---------------------------------------------------------------- oracle arm

def cpu_baseline(wl, budget_s):
    """The fp64 oracle, as it stands, on a bounded sample of the workload:
    whole sequences through the first group of layers (Full, Reindex,
    Reuse, Reuse), one sequence at a time until `budget_s` is spent.  Inputs
    are prepared outside the timed region (the oracle's own E4M3 / FP4
    casts of the seeded bf16 rows); timed: scores, top-k (with the candidate
    pool when the workload has one) and attention."""
    import numpy as np
    from oracle import oracle as orc
    from long_context_sparse_27_b300 import synth
    orc.lib()
    cores = len(os.sched_getaffinity(0))
    group = list(wl.modes[:4]) if len(wl.modes) >= 4 else list(wl.modes)
    scale = 1.0 / math.sqrt(wl.D)
    one = synth.scaled(wl, B=1)
    elapsed = 0.0
    seqs = 0
    table = orc.e4m3_table()
    while elapsed < budget_s and seqs < wl.B:
        s = 9000 + seqs
        kk = synth.index_k_rows(one, s + 1)
        k8 = orc.cast_e4m3(kk.double().numpy())
        kd = table[k8]
        kv = synth.kv_rows(one, s + 2)
        layers = []
        for l, m in enumerate(group):
            layers.append({"q": synth.index_q(one, s + 10 + l).double().numpy(),
                           "w": synth.index_w(one, s + 20 + l).double().numpy(),
                           "aq": synth.attn_q(one, s + 30 + l).double().numpy(),
                           "win": synth.window_rows(one, s + 40 + l).double().numpy()})
        q8c = [None if wl.fp32_indexer else orc.quantize_index_q(L["q"], L["w"]) for L in layers]
        kf = kk.double().numpy()
        t0 = time.perf_counter()
        idx = pool = None
        for l, m in enumerate(group):
            L = layers[l]
            if m in (0, 1):
                if wl.fp32_indexer:
                    sc = orc.index_score(L["q"], L["w"], kf)
                else:
                    q8, c = q8c[l]
                    sc = orc.index_score(table[q8], c, kd)
                if wl.pool and m == 0:
                    pool = orc.topk(sc, wl.pool)   # the candidate pool
                if wl.pool and m == 1:
                    sc = orc.pool_restrict(sc, pool)
                idx = orc.topk(sc, wl.k)
            sel = idx[0][idx[0] >= 0]
            c_rows, s_rows = orc.quantize_fp4(
                kv[0][torch.from_numpy(sel.astype(np.int64))].double().numpy())
            codes = np.zeros((1, wl.N, wl.D // 2), np.uint8)
            scl = np.zeros((1, wl.N, wl.D // 32), np.uint8)
            codes[0, sel], scl[0, sel] = c_rows, s_rows
            orc.sparse_attn(L["aq"], codes, scl, idx, L["win"], scale)
        elapsed += time.perf_counter() - t0
        seqs += 1
    token_steps = seqs * len(group) / len(wl.modes)
    return {"value": round(token_steps / elapsed, 4), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{seqs} of {wl.B} sequences through layers 0-{len(group) - 1} "
                      f"({''.join('FIU'[m] for m in group)}) of {len(wl.modes)}, N={wl.N}; "
                      f"{elapsed:.1f} s of oracle time",
            "seconds": round(elapsed, 2)}


def run_reference(args, world, rank):
    from long_context_sparse_27_b300 import synth
    if rank != 0:
        return None
    wl = synth.WORKLOADS[args.workload]
    budget = max(2.0, args.cpu_budget_s / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        cpu_baseline(wl, budget)
    vals = [cpu_baseline(wl, budget) for _ in range(args.steps)]
    v = statistics.median(x["value"] for x in vals)
    cb = dict(vals[-1])
    cb["value"] = v
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": v,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1); planted indexer keys)",
        "config": {"workload": workload_desc(wl), "sample": cb["sample"]},
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_project(args):
    """The decoder's global-KV projection + FP4 quantiser on its own
    (csa2_project_fp4): a decode step (one new row per sequence, B = 8) and
    a prefill chunk's 1024 entries, hidden 4096, d 512, each timed with CUDA
    events over `steps` launches after `warmup`, L2 flushed before each."""
    from long_context_sparse_27_b300 import csa2, synth
    flush = L2Flush()
    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    hidden, d = 4096, 512
    w = (synth.normal((d, hidden), 300, "cuda") * 0.05).to(torch.bfloat16)
    lines = []
    for rows in (8, 1024):
        h = synth.normal((rows, hidden), 301 + rows, "cuda")
        for _ in range(max(args.warmup, 3)):
            csa2.project_fp4(h, w)
        stream = torch.cuda.current_stream()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for a, b in ev:
            flush()
            a.record(stream)
            csa2.project_fp4(h, w)
            b.record(stream)
        torch.cuda.synchronize()
        t = sum(a.elapsed_time(b) for a, b in ev) / args.steps * 1e-3
        nbytes = (rows + d) * hidden * 2 + rows * (d // 2 + d // 32)
        flops = 2.0 * rows * hidden * d
        lines.append({"op": "csa2_project_fp4", "rows": rows, "hidden": hidden, "d": d,
                      "us": round(t * 1e6, 3), "GB/s": round(nbytes / t / 1e9, 1),
                      "hbm_frac": round(nbytes / t / 1e9 / hbm_peak, 4),
                      "TFLOP/s": round(flops / t / 1e12, 2),
                      "bf16_frac": round(flops / t / 1e12 / bf16_peak, 4), "peak_kind": peak_kind,
                      "steps": args.steps, "warmup": args.warmup})
    return lines


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="1m")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--op", default=None, choices=["project"],
                    help="time one entry point on its own instead of the step")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_env()
    if args.op == "project":
        for line in run_project(args):
            print(json.dumps(line), flush=True)
        return 0
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    init_dist(world, "nccl")
    line = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
