"""Benchmark: INT4 + 2:4 SparseGemv decode linears on one GB300 (or N independent replicas).

Workload (one "step"): the 7B-shaped decode linears at batch 1 -- one sparse GEMV (2:4 "2bit-CSR",
INT4, group 128) of each shape N x K in {4096 x 4096, 11008 x 4096, 4096 x 11008}; W ~ N(0, 0.02^2),
x ~ N(0, 1), synthetic and seeded. Metric: effective HBM GB/s (algorithmic bytes / time) and
microseconds per GEMV.

Dispatch: the three layers of a step are independent (each has its own x), so the step calls the
library's dispatch entry (sgemv_run_stack), which runs them as one grouped launch; --separate launches them
one by one (the per-shape numbers are single launches either way).

Timing: packed weights rotate over 8 distinct copies per shape (about 350 MB, more than twice the L2),
so every step reads its weights from HBM. The timed region is a CUDA-graph replay of K steps on the
launching stream, bracketed by CUDA events with a device synchronize (and, for N > 1, a barrier) on both
sides; W warm-up steps run before it. SM clocks are sampled with nvidia-smi during the timed region.

e2e: the same metric through the Python binding of the C ABI with host buffers: every step copies its
three x vectors (one pinned host buffer) to the device, runs the three GEMVs through sgemv_run_stack, and
reads the three y back (one pinned host buffer). The steps are independent requests, so the reported form
overlaps the copies of neighbouring steps with the GEMVs (three streams ordered by events, double-buffered
x, 32 steps per CUDA graph); e2e.serial is the same loop on one stream, three calls per step from Python.

cpu_baseline / --impl reference: the CPU oracle (plain C++, fp64, OpenMP over rows) on a bounded sample of
the same workload (the first 1024 rows of each shape), timed on this machine's host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "µs per GEMV and effective HBM GB/s (% of GB300 peak) for INT4+2:4 SparseGemv"
SHAPES = ((4096, 4096), (11008, 4096), (4096, 11008))
GROUP = 128
BATCH = 1
ROTATE = 8
E2E_GRAPH = 32  # steps per CUDA graph in the pipelined e2e loop
WORKLOAD = "7B decode linears, batch 1: 4096x4096 + 11008x4096 + 4096x11008, 2:4 sparse INT4 g128"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shapes", default=None,
                    help="profiling: comma-separated NxK list replacing the default workload")
    ap.add_argument("--batch", type=int, default=BATCH, help="profiling: batch (beam width)")
    ap.add_argument("--format", default="sparse", choices=["sparse", "sparse14", "dense"],
                    help="profiling: packed format (2:4, 1:4 or dense INT4)")
    ap.add_argument("--eager", action="store_true", help="profiling: launch eagerly instead of graph replay")
    ap.add_argument("--stack", action="store_true",
                    help="profiling: one decode step of the 224-layer layer-adaptive stack (32 blocks x 7 linears)")
    ap.add_argument("--stack-formats", default="1,2",
                    help="formats the stack policy draws from: 1 = 2:4, 3 = 1:4, 2 = dense (e.g. 1,3,2)")
    ap.add_argument("--separate", action="store_true",
                    help="launch the step's layers one by one instead of through the grouping dispatch")
    ap.add_argument("--beam", action="store_true",
                    help="profiling: the trie-constrained beam-score step (beam 20, vocab 32000, depth-4 trie)")
    ap.add_argument("--skip-extras", action="store_true",
                    help="profiling: time the steps only (no per-shape, e2e or CPU baseline)")
    return ap.parse_args()


# ---------------------------------------------------------------------------------------------- ranks

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Maximum of a per-rank float over all ranks (host collective; not on the data path)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# The sources that define the timed 2:4 GEMV kernel (the streaming kernel, group size 128) and its
# launch (planner, dispatch, public header).
TIMED_KERNEL_SOURCES = ("include/sgemv.h", "int4_weight_only_sgemv_gb300/csrc/abi.cu",
                        "int4_weight_only_sgemv_gb300/csrc/common.cuh",
                        "int4_weight_only_sgemv_gb300/csrc/stream_kernel.cuh",
                        "int4_weight_only_sgemv_gb300/csrc/stream_launch.cuh",
                        "int4_weight_only_sgemv_gb300/csrc/gemv_stream24_g128.cu")


def lib_fingerprint() -> str:
    """Hash of the sources of the timed kernel: identifies the kernel a profile was taken of."""
    h = hashlib.sha256()
    for rel in TIMED_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(rel.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram bytes per launch of the timed kernel from profiles/sgemv_sparse_traffic.txt, if that capture
    was taken of the current sources (its fingerprint line matches); else None."""
    path = os.path.join(ROOT, "profiles", "sgemv_sparse_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for ln in f:
                if ":" in ln and not ln.startswith("#"):
                    k, v = ln.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("fingerprint") != lib_fingerprint():
            return None
        return float(kv["dram_bytes_per_step_launch_avg"])
    except (OSError, KeyError, ValueError):
        return None


def group_launches(formats, max_group: int = 8) -> int:
    """Launches sgemv_run_stack makes for independent layers: runs of the same format, 8 at most each."""
    n, prev, size = 0, None, 0
    for f in formats:
        if f != prev or size == max_group:
            n, prev, size = n + 1, f, 0
        size += 1
    return n


def step_bytes(sg, layouts, batch):
    return sum(sg.algorithmic_bytes(L, batch) for L in layouts)


# ---------------------------------------------------------------------------------------------- CPU oracle

def cpu_oracle_run(seconds: float, single_thread: bool = False):
    """Time the CPU oracle GEMV on the first 1024 rows of each shape (all host cores through OpenMP, or one
    thread: the plain correctness oracle); returns (GB/s, threads, sample, seconds per pass)."""
    import oracle
    rows = 1024
    bufs, xs, nbytes = [], [], 0
    for (n, k) in SHAPES:
        w = synth.weights(rows, k, "bench", n, k)
        bufs.append(oracle.pack(w, oracle.FMT_SPARSE24, GROUP))
        xs.append(synth.activations(BATCH, k, "bench", n, k))
        nbytes += rows * (k // 4 + k // 8 + 4 * k // GROUP) + 2 * BATCH * k + 2 * BATCH * rows
    threads = os.cpu_count() or 1
    if single_thread or not oracle.openmp_available():
        threads = 1
    reps = 0
    t0 = time.perf_counter()
    while True:
        for buf, x in zip(bufs, xs):
            oracle.gemv(buf, x, nthreads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    gbs = nbytes * reps / el / 1e9
    sample = (f"first 1024 rows of each of the 3 shapes (g{GROUP}, batch {BATCH}), {reps} passes in "
              f"{el:.1f} s, {threads} OpenMP thread{'s' if threads > 1 else ''}, fp64 oracle")
    return gbs, threads, sample, el / reps


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    gbs, threads, sample, sec_per_pass = cpu_oracle_run(min(args.cpu_seconds, per_step * args.steps))
    us_per_gemv = sec_per_pass / len(SHAPES) * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec_per_pass * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "us_per_gemv": round(us_per_gemv, 2),
            "config": {"workload": WORKLOAD + " (CPU oracle on a row sample)", "batch": BATCH, "group": GROUP},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------- GPU arm

def run_stack(args, rank, local, world):
    """One decode step of the layer-adaptive stack: 32 blocks x {q, k, v, o, gate, up, down}, each layer
    with its seeded format and group size, run through sgemv_run_stack (one launch per layer). The
    weights of the three distinct shapes are drawn once and packed per layer; x is independent per layer
    (no chaining). The stack (2-4 GB) is far larger than L2, so no rotation is needed."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import int4_weight_only_sgemv_gb300 as sg

    formats = tuple(int(v) for v in args.stack_formats.split(","))
    table = synth.stack_table(formats=formats)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    base = {}
    layers = []
    with torch.cuda.stream(stream):
        for i, (name, n, k, fmt, g) in enumerate(table):
            if (n, k) not in base:
                base[(n, k)] = torch.from_numpy(synth.weights(n, k, "stack-bench", n, k)).to(dev)
            layout, packed = sg.pack(base[(n, k)], fmt, g, status=status)
            x = torch.from_numpy(synth.activations(args.batch, k, "stack-bench", i)).to(dev)
            y = torch.empty((args.batch, n), dtype=torch.float16, device=dev)
            layers.append((layout, packed, x, y))
    torch.cuda.synchronize()
    base.clear()
    if int(status.item()) != 0:
        raise SystemExit(f"packing failed: {sg.sgemv_status_str(int(status.item()))}")
    bytes_step = step_bytes(sg, [L for (L, _, _, _) in layers], args.batch)
    stack_bytes = sum(L.total_bytes for (L, _, _, _) in layers)

    def step():
        sg.sgemv_run_stack(layers, args.batch, status=status, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    if int(status.item()) != 0:
        raise SystemExit(f"kernel reported {sg.sgemv_status_str(int(status.item()))}")
    sec = elapsed_ms / 1e3
    achieved = bytes_step * args.steps / sec / 1e9
    peak, peak_kind = measured_peaks()
    counts = {f: sum(1 for t in table if t[3] == f) for f in formats}
    line = {
        "metric": METRIC, "value": round(world * achieved, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4-f16-f32acc",
        "data": "synthetic", "us_per_gemv": round(elapsed_ms * 1e3 / (args.steps * len(layers)), 3),
        "config": {"workload": f"layer-adaptive stack, one decode step: {len(layers)} layers "
                               f"(formats {counts}, 1 = 2:4, 3 = 1:4, 2 = dense; g in 64/128/256), batch {args.batch}",
                   "batch": args.batch, "bytes_per_step": bytes_step,
                   "l2": f"inputs larger than L2: the stack is {stack_bytes / 1e9:.2f} GB",
                   "timing": "CUDA graph of one step (one launch per layer), replayed; CUDA events"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None, "peak_source": f"{peak_kind} hbm_gbs"},
        "gpu_launches": args.steps * group_launches([L.format for (L, _, _, _) in layers]),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_beam(args, rank, local, world):
    """Trie-constrained decoding of the tree-based verification: one timed unit is a full decode of a
    depth-4 trie (4 beam-score steps, beam 20, vocab 32000) plus the traceback, captured as a CUDA graph
    and run by sgemv_beam_decode (one launch); each step reads its beams from the previous step's output.
    The decoder's log-probabilities are synthetic rows resident on the device (one [20, 32000] block per
    step). Reported per beam step; the same decode as one launch per step (sgemv_beam_step, then
    sgemv_beam_traceback) is reported beside it."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import int4_weight_only_sgemv_gb300 as sg
    from oracle import beam as obeam

    branching, vocab, k = [256, 32, 8, 4], 32000, 20
    ptr, tok, nod = synth.trie(branching, vocab, "bench-beam")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    trie, keep = sg.make_trie(ptr, tok, nod)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    steps = len(branching)
    logps = [torch.from_numpy(synth.log_probs(1 if t == 0 else k, vocab, "bench-beam", t)).to(dev) for t in range(steps)]
    node0 = torch.zeros(1, dtype=torch.int32, device=dev)
    score0 = torch.zeros(1, dtype=torch.float32, device=dev)
    parents = torch.empty((steps, k), dtype=torch.int32, device=dev)  # step t writes row t directly
    toks = torch.empty((steps, k), dtype=torch.int32, device=dev)
    outs = [(torch.empty(k, dtype=torch.int32, device=dev), torch.empty(k, dtype=torch.float32, device=dev),
             parents[t], toks[t], torch.empty(1, dtype=torch.int32, device=dev)) for t in range(steps)]
    seq = torch.empty((k, steps), dtype=torch.int32, device=dev)

    def decode():  # one launch per step, then the traceback
        for t in range(steps):
            nd, sc = (node0, score0) if t == 0 else (outs[t - 1][0], outs[t - 1][1])
            sg.sgemv_beam_step(trie, nd, sc, logps[t], k, outs[t], status=status, stream=stream)
        sg.sgemv_beam_traceback(parents, toks, outs[-1][4], seq, status=status, stream=stream)

    out_f = (torch.empty((steps, k), dtype=torch.int32, device=dev), torch.empty((steps, k), dtype=torch.float32, device=dev),
             torch.empty((steps, k), dtype=torch.int32, device=dev), torch.empty((steps, k), dtype=torch.int32, device=dev),
             torch.empty(steps, dtype=torch.int32, device=dev))
    seq_f = torch.empty((k, steps), dtype=torch.int32, device=dev)

    def decode_fused():  # every step and the traceback in one launch
        sg.sgemv_beam_decode(trie, node0, score0, logps, k, out_f, seq_f, status=status, stream=stream)

    def time_graph(fn, clocks=None):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fn()
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.start()
        barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        clk = clocks.stop() if clocks is not None else None
        return max_over_ranks(ev0.elapsed_time(ev1), world), clk

    elapsed_steps_ms, _ = time_graph(decode)
    clocks = ClockSampler(local)
    elapsed_ms, clk = time_graph(decode_fused, clocks)
    if int(status.item()) != 0:
        raise SystemExit(f"kernel reported {sg.sgemv_status_str(int(status.item()))}")
    # both decodes on the device equal the oracle's (checked once, outside the timed regions)
    nodes, scores = np.array([0], np.int32), np.array([0.0], np.float32)
    for t in range(steps):
        r = obeam.beam_step(ptr, tok, nod, nodes, scores, logps[t].cpu().numpy(), k)
        nodes, scores = r["node"], r["score"]
    assert np.array_equal(outs[-1][0].cpu().numpy()[:r["count"]], r["node"]), "beam decode differs from the oracle"
    assert np.array_equal(out_f[0][-1].cpu().numpy()[:r["count"]], r["node"]), "fused decode differs from the oracle"
    assert np.array_equal(seq_f.cpu().numpy(), seq.cpu().numpy()), "fused traceback differs from the step-by-step one"
    us_step = elapsed_ms * 1e3 / (args.steps * steps)
    cand = [branching[0]] + [k * b for b in branching[1:]]
    # bytes a step must touch: per candidate its edge (token, node) and its log-probability
    bytes_step = sum(12 * c for c in cand) / steps
    achieved = bytes_step / (us_step * 1e3)
    peak, peak_kind = measured_peaks()
    t0 = time.perf_counter()
    reps = 0
    lp_host = [lg.cpu().numpy() for lg in logps]
    while time.perf_counter() - t0 < min(args.cpu_seconds, 3.0) or reps == 0:
        nodes, scores = np.array([0], np.int32), np.array([0.0], np.float32)
        for t in range(steps):
            r = obeam.beam_step(ptr, tok, nod, nodes, scores, lp_host[t], k)
            nodes, scores = r["node"], r["score"]
        reps += 1
    cpu_us = (time.perf_counter() - t0) * 1e6 / (reps * steps)
    line = {
        "metric": "µs per trie-constrained beam-score step (tree-based verification)", "value": round(us_step, 3),
        "unit": "us", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"beam {k}, vocab {vocab}, trie branching {branching} "
                               f"({len(ptr) - 1} nodes), {steps} steps + traceback per decode",
                   "candidates_per_step": cand,
                   "timing": "CUDA graph of one decode (4 steps + traceback in one sgemv_beam_decode launch), "
                             "replayed; CUDA events",
                   "us_per_step_one_launch_per_step": round(elapsed_steps_ms * 1e3 / (args.steps * steps), 3)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 3), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 6), "traffic": None, "peak_source": f"{peak_kind} hbm_gbs",
                     "note": "latency-bound: one CTA per step touches a few KB"},
        "gpu_launches": args.steps,
        "clocks": clk,
        "cpu_baseline": {"value": round(cpu_us, 2), "unit": "us", "cores": 1, "kind": "oracle",
                         "sample": f"{reps} full decodes of the same trie and log-probabilities, numpy oracle"},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, local, world = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.stack or args.beam:
        if args.warmup < 3:
            raise SystemExit("--warmup must be >= 3")
        (run_stack if args.stack else run_beam)(args, rank, local, world)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    shapes = SHAPES
    if args.shapes:
        shapes = tuple(tuple(int(v) for v in item.split("x")) for item in args.shapes.split(","))
    batch = args.batch
    profiling = bool(args.shapes or args.eager or args.skip_extras or batch != BATCH or args.format != "sparse"
                     or args.separate)

    import torch
    import __graft_entry__
    __graft_entry__.build()
    import int4_weight_only_sgemv_gb300 as sg

    fmt = {"sparse": sg.SGEMV_FMT_SPARSE24, "sparse14": sg.SGEMV_FMT_SPARSE14, "dense": sg.SGEMV_FMT_DENSE}[args.format]
    run = sg.sgemv_run_dense if fmt == sg.SGEMV_FMT_DENSE else sg.sgemv_run
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    # ---- workload: weights packed on the GPU, ROTATE distinct copies per shape
    layouts, packs, xs, ys, xs_host = [], [], [], [], []
    for (n, k) in shapes:
        w = synth.weights(n, k, "bench", n, k)
        x = synth.activations(batch, k, "bench", n, k)
        with torch.cuda.stream(stream):
            layout, packed = sg.pack(torch.from_numpy(w).to(dev), fmt, GROUP, status=status)
            copies = [packed] + [packed.clone() for _ in range(ROTATE - 1)]
        layouts.append(layout)
        packs.append(copies)
        xs.append([torch.from_numpy(x).to(dev) for _ in range(ROTATE)])
        ys.append([torch.empty((batch, n), dtype=torch.float16, device=dev) for _ in range(ROTATE)])
        xs_host.append(torch.from_numpy(x).pin_memory())
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise SystemExit(f"packing failed: {sg.sgemv_status_str(int(status.item()))}")
    bytes_step = step_bytes(sg, layouts, batch)
    working_set = sum(L.total_bytes for L in layouts) * ROTATE

    def step(i):
        # the step's layers are independent (each has its own x), so the dispatch runs them as one
        # grouped launch; --separate launches them one by one
        c = i % ROTATE
        if args.separate:
            for s in range(len(shapes)):
                run(layouts[s], packs[s][c], xs[s][c], ys[s][c], status=status, stream=stream)
        else:
            sg.sgemv_run_stack([(layouts[s], packs[s][c], xs[s][c], ys[s][c]) for s in range(len(shapes))], batch,
                               status=status, stream=stream)

    # ---- warm-up (eager), then capture one rotation (ROTATE steps) and the remainder as graphs
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    g_rot = g_tail = None
    if not args.eager:
        g_rot = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rot, stream=stream):
            for i in range(ROTATE):
                step(i)
        tail = args.steps % ROTATE
        if tail:
            g_tail = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_tail, stream=stream):
                for i in range(tail):
                    step(i)
        with torch.cuda.stream(stream):  # warm the graphs themselves
            for _ in range(max(1, args.warmup // ROTATE)):
                g_rot.replay()
        torch.cuda.synchronize()

    # ---- timed region
    clocks = ClockSampler(local)
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    ev0.record(stream)
    with torch.cuda.stream(stream):
        if args.eager:
            for i in range(args.steps):
                step(i)
        else:
            for _ in range(args.steps // ROTATE):
                g_rot.replay()
            if g_tail is not None:
                g_tail.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    if int(status.item()) != 0:
        raise SystemExit(f"kernel reported {sg.sgemv_status_str(int(status.item()))}")
    launches = args.steps * (len(shapes) if args.separate else 1)
    gemvs = args.steps * len(shapes)
    sec = elapsed_ms / 1e3
    value = world * bytes_step * args.steps / sec / 1e9
    us_per_gemv = elapsed_ms * 1e3 / gemvs
    achieved = bytes_step * args.steps / sec / 1e9
    peak, peak_kind = measured_peaks()
    workload = WORKLOAD if not profiling else (
        f"{args.format} INT4 g{GROUP}, batch {batch}: " + " + ".join(f"{n}x{k}" for n, k in shapes))
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int4-f16-f32acc", "data": "synthetic",
        "us_per_gemv": round(us_per_gemv, 3),
        "config": {"workload": workload, "batch": batch, "group": GROUP, "shapes": [f"{n}x{k}" for n, k in shapes],
                   "l2": f"inputs larger than L2: {ROTATE} rotating packed copies, {working_set / 1e6:.0f} MB",
                   "timing": ("eager launches" if args.eager else "CUDA graph replay") +
                             ", CUDA events on the launching stream",
                   "dispatch": ("one launch per layer (sgemv_run)" if args.separate else
                                "sgemv_run_stack: the independent layers of a step run as one grouped launch"),
                   "bytes_per_step": bytes_step},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None if profiling else profiled_traffic(),
                     "peak_source": f"{peak_kind} hbm_gbs", "nominal_frac": round(achieved / 8000.0, 4)},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if args.skip_extras:
        if rank == 0:
            print(json.dumps(line), flush=True)
        return

    # ---- per-shape µs (graph of ROTATE launches of one shape, replayed)
    per_shape = {}
    for s, (n, k) in enumerate(shapes):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in range(ROTATE):
                run(layouts[s], packs[s][c], xs[s][c], ys[s][c], status=status, stream=stream)
        reps = max(10, min(2000, args.steps // ROTATE))
        with torch.cuda.stream(stream):
            for _ in range(5):
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * ROTATE)
        b = sg.algorithmic_bytes(layouts[s], batch)
        per_shape[f"{n}x{k}"] = {"us": round(us, 3), "GB/s": round(b / us / 1e3, 1), "bytes": b}
    line["config"]["per_shape"] = per_shape

    # ---- e2e: host buffers through the binding, copies inside the timed region. The three x vectors
    # sit in one pinned host buffer and one device buffer (one copy in), the three y vectors in one device
    # buffer per weight copy and one pinned host buffer (one copy out); the dispatch tables are
    # marshalled once (sg.Stack), so a step is three calls.
    e2e_steps = max(20, min(args.steps, 3000))
    x_len = [batch * k for (_, k) in shapes]
    y_len = [batch * n for (n, _) in shapes]
    pad8 = lambda v: (v + 7) // 8 * 8  # each vector starts on a 16-byte boundary (the ABI's alignment)
    x_host_all = torch.zeros(sum(pad8(v) for v in x_len), dtype=torch.float16).pin_memory()
    o = 0
    for x, ln in zip(xs_host, x_len):
        x_host_all[o:o + ln] = x.reshape(-1)
        o += pad8(ln)
    x_dev_all = torch.empty_like(x_host_all, device=dev)
    y_host_all = torch.empty(sum(pad8(v) for v in y_len), dtype=torch.float16).pin_memory()
    y_dev_all = [torch.empty_like(y_host_all, device=dev) for _ in range(ROTATE)]

    def views(buf, lens, rows):
        out, o = [], 0
        for ln, (n, k) in zip(lens, rows):
            out.append(buf[o:o + ln].view(batch, ln // batch))
            o += pad8(ln)
        return out

    x_views = views(x_dev_all, x_len, shapes)
    y_views = [views(y_dev_all[c], y_len, shapes) for c in range(ROTATE)]
    stacks = [sg.Stack([(layouts[s], packs[s][c], x_views[s], y_views[c][s]) for s in range(len(shapes))], batch)
              for c in range(ROTATE)]
    h2d = int(x_host_all.numel()) * 2
    d2h = int(y_host_all.numel()) * 2

    def e2e_step(i):
        c = i % ROTATE
        x_dev_all.copy_(x_host_all, non_blocking=True)
        if args.separate:
            for s in range(len(shapes)):
                run(layouts[s], packs[s][c], x_views[s], y_views[c][s], status=status, stream=stream)
        else:
            stacks[c].run(status=status, stream=stream)
        y_host_all.copy_(y_dev_all[c], non_blocking=True)

    def time_e2e(fn):
        with torch.cuda.stream(stream):
            for i in range(5):
                fn(i)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for i in range(e2e_steps):
                fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier(world)
        sec = max_over_ranks(max(wall, e0.elapsed_time(e1) / 1e3), world)
        return round(world * bytes_step * e2e_steps / sec / 1e9, 2)

    serial = time_e2e(e2e_step)

    # Pipelined form of the same loop: steps are independent requests, so the copies of one step overlap
    # the kernels of its neighbours. Three streams ordered by events (x in, GEMVs, y out; x and the host
    # y double-buffered, each y buffer reused only after its copy out), E2E_GRAPH steps captured as one
    # CUDA graph and replayed, so that the host issues one call per E2E_GRAPH steps. Every step still
    # copies its x in from pinned host memory and its y out to pinned host memory.
    e2e_pipe = None
    if not args.separate:
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        x_dev_pp = [x_dev_all, torch.empty_like(x_host_all, device=dev)]
        x_views_pp = [views(x_dev_pp[q], x_len, shapes) for q in range(2)]
        y_host_pp = [y_host_all, torch.empty_like(y_host_all).pin_memory()]
        stacks_pp = [[sg.Stack([(layouts[s], packs[s][c], x_views_pp[q][s], y_views[c][s]) for s in range(len(shapes))],
                               batch) for q in range(2)] for c in range(ROTATE)]
        P = E2E_GRAPH
        ev_in = [torch.cuda.Event() for _ in range(P)]
        ev_k = [torch.cuda.Event() for _ in range(P)]
        ev_out = [torch.cuda.Event() for _ in range(P)]
        ev_fork, ev_in_end, ev_out_end = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()

        def pipelined_steps():
            ev_fork.record(stream)
            s_in.wait_event(ev_fork)
            s_out.wait_event(ev_fork)
            for i in range(P):
                q, c = i % 2, i % ROTATE
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_k[i - 2])  # step i-2's GEMVs have read this x buffer
                    x_dev_pp[q].copy_(x_host_all, non_blocking=True)
                    ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                if i >= ROTATE:
                    stream.wait_event(ev_out[i - ROTATE])  # this y buffer's previous copy out is done
                stacks_pp[c][q].run(status=status, stream=stream)
                ev_k[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_k[i])
                    y_host_pp[q].copy_(y_dev_all[c], non_blocking=True)
                    ev_out[i].record(s_out)
            ev_in_end.record(s_in)
            ev_out_end.record(s_out)
            stream.wait_event(ev_in_end)
            stream.wait_event(ev_out_end)

        torch.cuda.synchronize()
        g_pipe = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pipe, stream=stream):
            pipelined_steps()
        replays = max(1, e2e_steps // P)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g_pipe.replay()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(replays):
                g_pipe.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier(world)
        sec = max_over_ranks(max(wall, e0.elapsed_time(e1) / 1e3), world)
        e2e_pipe = round(world * bytes_step * replays * P / sec / 1e9, 2)

    line["e2e"] = {"value": e2e_pipe if e2e_pipe is not None else serial, "unit": "GB/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                   "form": ("pipelined: copies of neighbouring steps overlap the GEMVs (3 streams, "
                            f"graphs of {E2E_GRAPH} steps)" if e2e_pipe is not None else "serial"),
                   "serial": serial}

    # ---- CPU baseline (rank 0 at N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, threads, sample, _ = cpu_oracle_run(args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample}
        # the same oracle on one core (its plain form, without the OpenMP loop over rows)
        gbs1, _, sample1, _ = cpu_oracle_run(max(1.0, args.cpu_seconds / 4), single_thread=True)
        cpu["single_thread"] = {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1, "sample": sample1}
    line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
