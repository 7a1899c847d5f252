#!/usr/bin/env python3
"""Throughput of the exact per-row top-K on GB300: rows/s, us/row and HBM roofline.

Workload: the decode batch -- 64 requests x next_n = 2 (128 rows), kv_lens
~ U[16384, 524288] uncompressed tokens, compress_ratio 4 (so n up to 131072),
K = 1024, row stride 131072 fp32, scores N(0,1) plus a position-linear bias,
poisoned padding, and three requests at n = K-1, K, K+1.  Synthetic and seeded
(workloads.decode_batch).

One step = one topk_decode_ws call over the whole batch (one kernel launch: the
balanced kernel, which splits the batch's valid scores evenly over the GPU).

* value (cold L2): the timed region replays a CUDA graph that runs the step on
  R distinct device copies of the batch in turn, R * 64 MiB >> L2 (129 MB), so
  no step finds its scores in L2.  Timed with CUDA events on the launching
  stream, a barrier and torch.cuda.synchronize() on both sides, max over ranks.
  The --steps window is repeated until --min-seconds have passed; the line
  reports the median window (clocks are sampled over all of them).
* extra keys (the target configurations, cold/warm, outside the timed region):
  sweep_big (the >= 36 MB sweep cells, decode and prefill), tail (each
  adversarial variant against a normal row of the same shape), single_row
  (one 8192-score row, K = 512) and prefill_tile (4096 rows, K = 2048).
* warm_l2: the same graph over one copy (scores L2-resident after the first).
* e2e: the public API with host buffers: every step copies the batch from
  pinned host memory to the device, selects, and copies the indices back.
* roofline: algorithmic bytes per launch (4 nv per row that needs a selection,
  plus 4 K written per row, plus the kv_lens read) / the cold-L2 time per
  launch, against the measured HBM copy peak.
* cpu_baseline: the CPU oracle (full sort per row) on the host cores.

``--impl reference`` times the CPU oracle alone as the reference arm.
Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no
data-path collective); value = all ranks' rows / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "rows/s and µs/row top-K (cold/warm L2); HBM GB/s vs ~8 TB/s at 1 GB300"
NOMINAL_HBM_GBS = 8000.0
KERNEL_NAME = "gvr_topk_kernel"
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over the default process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def algorithmic_bytes(case, with_values: bool) -> int:
    """Bytes the selection must move: each score of a row that needs a selection read once,
    K indices (and K values) written per row, and one kv_lens entry per request."""
    n = case.row_lengths().astype(np.int64)
    k = case.k
    reads = int(np.where(n > k, 4 * n, 4 * n if with_values else 0).sum())
    writes = case.rows * k * 4 * (2 if with_values else 1)
    return reads + writes + 4 * case.kv_lens.size


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_indexer_exact_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of ``kernel`` on the headline workload, from the ncu
    capture recorded in profiles/traffic.json -- only while the kernel sources still match the
    digest recorded with it (a changed kernel has no measured traffic until it is captured again)."""
    try:
        with open(TRAFFIC_JSON) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != source_digest() or rec.get("kernel") != kernel:
        return None
    return float(rec["dram_bytes_per_launch"])


def measured_peak_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t0 = time.time()
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def time_oracle(case, nthreads: int, repeats: int, min_seconds: float = 0.0, max_runs: int = 1000):
    """Median wall time of one oracle run over the whole batch, over at least `repeats` runs and
    at least `min_seconds` of runs in all (at most `max_runs`); returns (seconds, cores, runs,
    total seconds)."""
    import oracle
    oracle.build()
    cores = oracle.thread_count(nthreads)
    times = []
    while len(times) < max_runs and (len(times) < repeats or sum(times) < min_seconds):
        t0 = time.perf_counter()
        oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k, nthreads=nthreads)
        times.append(time.perf_counter() - t0)
    return statistics.median(times), cores, len(times), sum(times)


CPU_BASELINE_S = 10.0  # the cpu_baseline leg's runs take about this long in all


REFERENCE_BUDGET_S = 90.0  # the reference arm's timed steps take about this long in all


def run_reference(args, case, ws, rank):
    """The CPU oracle as the reference arm: each step selects a bounded sample of whole requests
    of the batch (cycling through it), sized so that all timed steps take about
    REFERENCE_BUDGET_S seconds."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = oracle.thread_count(0)
    t0 = time.perf_counter()
    oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
    t_full = time.perf_counter() - t0
    reqs = case.kv_lens.size
    per_req = t_full / reqs
    nq = int(max(1, min(reqs, REFERENCE_BUDGET_S / (max(args.steps, 1) * per_req))))

    def step(i):
        q0 = (i * nq) % reqs
        q1 = min(q0 + nq, reqs)
        oracle.topk_decode(case.logits[q0 * case.next_n:q1 * case.next_n], case.kv_lens[q0:q1], case.next_n,
                           case.compress_ratio, case.k)
        return (q1 - q0) * case.next_n

    for i in range(args.warmup):
        step(i)
    done = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        done += step(i)
    el = time.perf_counter() - t0
    rows_s = done / el
    sample = (f"{nq} of the batch's {reqs} requests ({nq * case.next_n} rows) per step, cycling through the "
              f"batch, full sort per row, {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": rows_s, "unit": "rows/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "us_per_row": 1e6 * el / max(done, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_block(case, ws),
        "cpu_baseline": {"value": rows_s, "unit": "rows/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": rows_s, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def prefill_algorithmic_bytes(case) -> int:
    """Prefill: each score of a window that needs a selection read once, K indices written,
    and the two window bounds read per row."""
    n = case.window_lengths().astype(np.int64)
    return int(np.where(n > case.k, 4 * n, 0).sum()) + case.rows * case.k * 4 + 8 * case.rows


class ColdWarm:
    """Cold- and warm-L2 timing of one call on the current stream.

    cold: a 512 MiB scrub write before each call (the call then finds none of its inputs in L2);
    per call CUDA events (median / p99 / max of ``reps``; the event clock ticks in ~2 us steps on
    this GPU) and, at finer resolution, the mean over graphs of (scrub + call) minus (scrub) --
    rates use that graph mean.  warm: a graph of ``warm_calls`` back-to-back calls on one input."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.stream = torch.cuda.current_stream()
        self.scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > L2 (129 MB)

    def _graph_us(self, body, calls):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h = torch.cuda.current_stream().cuda_stream
            for i in range(calls):
                body(i, h)
        g.replay()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e3)
        return best / calls

    def __call__(self, launch, reps=32, warm_calls=100):
        torch, stream, scrub = self.torch, self.stream, self.scrub
        for _ in range(3):
            launch(stream.cuda_stream)
        torch.cuda.synchronize()
        cold = []
        for r in range(reps):
            scrub.fill_(r & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch(stream.cuda_stream)
            e1.record(stream)
            torch.cuda.synchronize()
            cold.append(e0.elapsed_time(e1) * 1e3)
        warm = self._graph_us(lambda i, h: launch(h), warm_calls)

        def scrub_then(with_call):
            def body(i, h):
                scrub.fill_(i & 255)
                if with_call:
                    launch(h)
            return body
        cold_mean = self._graph_us(scrub_then(True), 16) - self._graph_us(scrub_then(False), 16)
        cold.sort()
        return {"median": cold[len(cold) // 2], "p99": cold[min(len(cold) - 1, int(0.99 * len(cold)))],
                "max": cold[-1], "graph_mean": cold_mean, "warm": warm}


def _launchers(torch, gvr, dev, wsb):
    """Callables that run one decode / prefill call of a case through the *_ws entry points
    (by default the cluster kernel; flags=1024, GVR_FLAG_SPLIT_KERNEL, asks for the balanced
    kernel where the call fits it)."""

    def decode(case, flags=0):
        lg = torch.from_numpy(case.logits).to(dev)
        kv = torch.from_numpy(case.kv_lens).to(dev)
        idx = torch.empty((case.rows, case.k), dtype=torch.int32, device=dev)
        o = gvr.Options(flags=flags) if flags else None
        return lambda h: gvr.topk_decode_ws_raw(lg.data_ptr(), lg.shape[1], case.rows, kv.data_ptr(), case.next_n,
                                                case.compress_ratio, case.k, idx.data_ptr(), None, wsb.data_ptr(),
                                                wsb.numel(), h, o)

    def prefill(case, flags=0):
        lg = torch.from_numpy(case.logits).to(dev)
        ks = torch.from_numpy(case.row_starts).to(dev)
        ke = torch.from_numpy(case.row_ends).to(dev)
        idx = torch.empty((case.rows, case.k), dtype=torch.int32, device=dev)
        o = gvr.Options(flags=flags) if flags else None
        return lambda h: gvr.topk_prefill_ws_raw(lg.data_ptr(), lg.shape[1], case.rows, ks.data_ptr(), ke.data_ptr(),
                                                 case.k, idx.data_ptr(), wsb.data_ptr(), wsb.numel(), h, o)
    return decode, prefill


def _cell(tag, case, nbytes, t, peak):
    cm = t["graph_mean"]
    return {"cell": tag, "bs": case.rows, "n": int((case.row_lengths() if hasattr(case, "row_lengths") else case.window_lengths()).max()), "k": case.k,
            "cold_us": {k: round(v, 2) for k, v in t.items() if k != "warm"}, "warm_us": round(t["warm"], 2),
            "rows_per_s_cold": case.rows / (cm * 1e-6), "us_per_row_cold": cm / case.rows,
            "algorithmic_bytes": nbytes, "gbs_cold": nbytes / cm / 1e3,
            "frac_of_measured": nbytes / cm / 1e3 / peak, "frac_of_8tbs": nbytes / cm / 1e3 / NOMINAL_HBM_GBS,
            "reachable_60pct": nbytes >= 36e6}


def tail_check(torch, gvr, dev, wsb, timer, peak, emit=None):
    """Each adversarial variant's cold graph-mean time over that of a row of the same shape drawn
    from N(0,1) (the benchmark spec's bound: no rescue-induced tail beyond 2x)."""
    import workloads
    decode, _ = _launchers(torch, gvr, dev, wsb)
    base = workloads.adversarial_row("base")
    g = np.random.default_rng(1049)
    plain = base.logits.copy()
    n0 = int(base.row_lengths()[0])
    plain[0, :n0] = g.standard_normal(n0).astype(np.float32)
    ref_case = workloads.DecodeCase("adversarial_shape_normal", plain, base.kv_lens, 1, base.compress_ratio, base.k,
                                    {"n": n0})
    t_ref = timer(decode(ref_case))
    if emit:
        emit(_cell("tail_reference_normal_row", ref_case, algorithmic_bytes(ref_case, False), t_ref, peak))
    ratios = {}
    for v in workloads.ADVERSARIAL_VARIANTS:
        c = workloads.adversarial_row(v)
        c.meta["n"] = n0
        t = timer(decode(c))
        if emit:
            emit(_cell(f"tail_{v}", c, algorithmic_bytes(c, False), t, peak))
        ratios[v] = round(t["graph_mean"] / t_ref["graph_mean"], 3)
    return {"normal_row_us": round(t_ref["graph_mean"], 2), "ratio_to_normal_row": ratios,
            "within_2x": all(r <= 2.0 for r in ratios.values())}


SWEEP_BIG = [(256, 131072, 512), (256, 131072, 1024), (256, 131072, 2048), (256, 65536, 512)]


def extras(torch, gvr, dev, wsb, peak, head_case=None):
    """The target configurations beside the headline, one call each at a time, cold and warm:
    the >= 36 MB sweep cells (decode and prefill), the tail check, the single decode row and
    the 4096-row prefill tile.  Also the headline batch as one isolated call after an L2 scrub
    (the per-launch figure a profiler that serialises launches reports)."""
    import workloads
    timer = ColdWarm(torch, dev)
    decode, prefill = _launchers(torch, gvr, dev, wsb)
    out = {}
    if head_case is not None:
        t = timer(decode(head_case), reps=16)
        out["isolated_launch"] = {"event_us": {"median": round(t["median"], 2), "p99": round(t["p99"], 2)},
                                  "scrub_graph_us": round(t["graph_mean"], 2),
                                  "note": "one call after a 512 MiB L2 scrub, per-call CUDA events; "
                                          "the headline times back-to-back graph launches"}
    cells = []
    for bs, n, k in SWEEP_BIG:
        dc = workloads.sweep_decode(bs, n, k)
        cells.append(_cell("decode", dc, algorithmic_bytes(dc, False), timer(decode(dc), reps=8), peak))
        pc = workloads.sweep_prefill(bs, n, k)
        cells.append(_cell("prefill", pc, prefill_algorithmic_bytes(pc), timer(prefill(pc), reps=8), peak))
        del dc, pc
        torch.cuda.empty_cache()
    out["sweep_big"] = cells
    out["tail"] = tail_check(torch, gvr, dev, wsb, timer, peak)
    sr = workloads.single_decode_row()
    t = timer(decode(sr))
    out["single_row"] = {"workload": sr.meta["workload"], "cold_us": round(t["graph_mean"], 2),
                         "cold_event_us": {"median": t["median"], "p99": t["p99"], "max": t["max"]},
                         "warm_us": round(t["warm"], 2)}
    pt = workloads.prefill_tile()
    t = timer(prefill(pt), reps=8)
    nb = prefill_algorithmic_bytes(pt)
    out["prefill_tile"] = {"workload": pt.meta.get("workload", "prefill tile"), "rows": pt.rows,
                           "cold_us": round(t["graph_mean"], 2), "warm_us": round(t["warm"], 2),
                           "rows_per_s_cold": pt.rows / (t["graph_mean"] * 1e-6),
                           "us_per_row_cold": t["graph_mean"] / pt.rows, "algorithmic_bytes": nb,
                           "frac_of_measured": nb / t["graph_mean"] / 1e3 / peak}
    return out


def run_sweep(args):
    """Every sweep cell (BS x N x K, decode and prefill), cold and warm L2, one JSON line each;
    the block-skip cells; then the tail check on the adversarial row and its variants."""
    import torch
    import workloads
    import sparse_attention_indexer_exact_gb300 as gvr

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback exists)")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gvr.load_library()
    wsb = torch.zeros(gvr.workspace_size(), dtype=torch.uint8, device=dev)
    peak, _ = measured_peak_hbm()
    timer = ColdWarm(torch, dev)
    decode, prefill = _launchers(torch, gvr, dev, wsb)

    def emit(d):
        print(json.dumps(d), flush=True)

    for n in (16384, 32768, 65536, 131072):
        for bs in (1, 4, 16, 64, 256):
            for k in (512, 1024, 2048):
                dc = workloads.sweep_decode(bs, n, k)
                emit(_cell("decode", dc, algorithmic_bytes(dc, False), timer(decode(dc)), peak))
                pc = workloads.sweep_prefill(bs, n, k)
                emit(_cell("prefill", pc, prefill_algorithmic_bytes(pc), timer(prefill(pc)), peak))
                del dc, pc
            torch.cuda.empty_cache()

    # block-skip: the same selection with exact block maxima given (decode rows)
    def block_max_of(case):
        nb = (case.row_stride + 31) // 32
        out = np.full((case.rows, nb), -np.inf, np.float32)
        n = case.row_lengths()
        for r in range(case.rows):
            if n[r]:
                x = np.full(((n[r] + 31) // 32) * 32, -np.inf, np.float32)
                x[:n[r]] = case.logits[r, :n[r]]
                out[r, :x.size // 32] = x.reshape(-1, 32).max(axis=1)
        return out

    for case in (workloads.decode_batch(), workloads.peaky_decode_batch(), workloads.sweep_decode(64, 131072, 1024),
                 workloads.sweep_decode(256, 131072, 1024), workloads.sweep_decode(256, 65536, 512)):
        lg = torch.from_numpy(case.logits).to(dev)
        kv = torch.from_numpy(case.kv_lens).to(dev)
        bm = torch.from_numpy(block_max_of(case)).to(dev)
        idx = torch.empty((case.rows, case.k), dtype=torch.int32, device=dev)
        case.meta.setdefault("n", int(case.row_lengths().max()))
        runs = (("cluster", lambda h, lg=lg, kv=kv, idx=idx, case=case: gvr.topk_decode_raw(
                    lg.data_ptr(), case.row_stride, case.rows, kv.data_ptr(), case.next_n, case.compress_ratio,
                    case.k, idx.data_ptr(), None, h)),
                ("balanced", decode(case, 1024)),
                ("blockskip_on", lambda h, lg=lg, kv=kv, idx=idx, case=case, bm=bm: gvr.topk_decode_blockskip_raw(
                    lg.data_ptr(), case.row_stride, case.rows, kv.data_ptr(), case.next_n, case.compress_ratio,
                    case.k, bm.data_ptr(), bm.stride(0), idx.data_ptr(), None, h)))
        for tag, launch in runs:
            emit(_cell(f"{tag}:{case.name}", case, algorithmic_bytes(case, False), timer(launch), peak))
        del lg, bm
    t = tail_check(torch, gvr, dev, wsb, timer, peak, emit)
    emit({"tail_check": t})
    return 0


def run_one_workload(args):
    """One workload alone, for profiling it (not the headline): the 4096-row prefill tile through
    topk_prefill, or the single 8192-score decode row (K = 512) through topk_decode; --steps
    graph-replayed calls rotating over --copies device copies, CUDA events on the launching
    stream; one JSON line."""
    import torch
    import workloads
    import sparse_attention_indexer_exact_gb300 as gvr

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback exists)")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gvr.load_library()
    tile = args.workload == "prefill_tile"
    case = workloads.prefill_tile() if tile else workloads.single_decode_row()
    copies = max(1, args.copies)
    bufs = [torch.from_numpy(case.logits).to(dev) for _ in range(copies)]
    idx = torch.empty((case.rows, case.k), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    if tile:
        ks = torch.from_numpy(case.row_starts).to(dev)
        ke = torch.from_numpy(case.row_ends).to(dev)

        def launch(buf, h):
            gvr.topk_prefill_raw(buf.data_ptr(), case.row_stride, case.rows, ks.data_ptr(), ke.data_ptr(), case.k,
                                 idx.data_ptr(), h)
    else:
        kv = torch.from_numpy(case.kv_lens).to(dev)

        def launch(buf, h):
            gvr.topk_decode_raw(buf.data_ptr(), case.row_stride, case.rows, kv.data_ptr(), case.next_n,
                                case.compress_ratio, case.k, idx.data_ptr(), None, h)

    for i in range(args.warmup):
        launch(bufs[i % copies], stream.cuda_stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(copies):
            launch(bufs[i], h)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // copies)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    per = e0.elapsed_time(e1) * 1e3 / (reps * copies)
    nbytes = prefill_algorithmic_bytes(case) if tile else algorithmic_bytes(case, False)
    peak, peak_kind = measured_peak_hbm()
    print(json.dumps({"workload": case.meta.get("workload", args.workload), "rows": case.rows, "k": case.k,
                      "calls": reps * copies, "copies": copies, "us_per_call": per,
                      "rows_per_s": case.rows / (per * 1e-6), "algorithmic_bytes": nbytes,
                      "frac_of_measured": nbytes / per / 1e3 / peak, "peak_kind": peak_kind}))
    return 0


def config_block(case, ws):
    return {"workload": f"decode batch: {case.meta['workload']}", "rows_per_gpu": case.rows,
            "global_rows": case.rows * ws, "k": case.k, "row_stride": case.row_stride,
            "valid_scores_per_step": int(case.row_lengths().sum()),
            "l2": "cold: graph steps rotate over distinct input copies whose total exceeds L2 "
                  "(warm_l2 reuses one copy)",
            "parallelism": f"{ws} GPU(s), each selecting its own batch; no data-path collective"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["gvr", "reference"], default="gvr")
    ap.add_argument("--copies", type=int, default=16, help="distinct device copies of the batch (cold L2)")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the --steps window until this much time has passed; report the median window")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--values", action="store_true", help="also write the fp32 values output")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the sweep_big / tail / single_row / prefill_tile keys")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the headline line: every sweep cell and the adversarial tail check")
    ap.add_argument("--workload", choices=["decode_batch", "prefill_tile", "single_row"], default="decode_batch",
                    help="prefill_tile / single_row: one line for the 4096-row prefill tile or the single "
                         "8192-score decode row alone (for profiling it)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.sweep:
        return run_sweep(args)
    if args.workload in ("prefill_tile", "single_row"):
        return run_one_workload(args)

    import workloads
    ws, rank, local = dist_env()
    case = workloads.decode_batch()

    if args.impl == "reference":
        return run_reference(args, case, ws, rank)

    import torch
    import torch.distributed as dist
    import sparse_attention_indexer_exact_gb300 as gvr

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback exists)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)

    gvr.load_library()
    k, rows, stride = case.k, case.rows, case.row_stride
    copies = max(1, args.copies)
    host = torch.from_numpy(case.logits)
    bufs = [host.to(dev) for _ in range(copies)]
    kv = torch.from_numpy(case.kv_lens).to(dev)
    idx = torch.empty((rows, k), dtype=torch.int32, device=dev)
    vals = torch.empty((rows, k), dtype=torch.float32, device=dev) if args.values else None
    vptr = vals.data_ptr() if vals is not None else None
    # the workspace of the balanced kernel (zero-filled once; every call leaves it zero-filled)
    wsb = torch.zeros(gvr.workspace_size(), dtype=torch.uint8, device=dev)

    def launch(buf, stream_handle, options=None):
        gvr.topk_decode_ws_raw(buf.data_ptr(), stride, rows, kv.data_ptr(), case.next_n, case.compress_ratio, k,
                               idx.data_ptr(), vptr, wsb.data_ptr(), wsb.numel(), stream_handle, options)

    stream = torch.cuda.current_stream()
    for i in range(args.warmup):  # eager warm-up also performs the one-time device set-up
        launch(bufs[i % copies], stream.cuda_stream)
    # which kernel the library chose for this call: its per-row path codes (untimed call)
    st = torch.full((rows, 4), -1, dtype=torch.int32, device=dev)
    launch(bufs[0], stream.cuda_stream, gvr.Options(row_stats=st.data_ptr()))
    torch.cuda.synchronize()
    paths = st[:, 0]
    kernel = ("gvr_split_kernel" if bool(((paths == 7) | (paths == 8)).any()) else
              "gvr_short_kernel" if bool(((paths == 10) | (paths == 11)).any()) else "gvr_topk_kernel")

    def make_graph(buffers):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h = torch.cuda.current_stream().cuda_stream
            for b in buffers:
                launch(b, h)
        return g

    cold_graph = make_graph(bufs)
    warm_graph = make_graph([bufs[0]] * copies)
    cold_graph.replay()  # graph upload
    warm_graph.replay()
    torch.cuda.synchronize()

    def window(graph, steps):
        """Exactly `steps` steps, bracketed by a barrier and a synchronize on both sides; device
        seconds from CUDA events on the launching stream, and wall seconds."""
        reps, rem = divmod(steps, copies)
        barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        for i in range(rem):
            launch(bufs[i % copies] if graph is cold_graph else bufs[0], stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3, time.perf_counter() - t_wall

    def windows(graph):
        """Repeat the window until --min-seconds of wall time (the same count on every rank);
        returns the median window's device seconds, the window count and the wall seconds."""
        first, wall0 = window(graph, args.steps)
        n = max(3, int(np.ceil(args.min_seconds / max(wall0, 1e-6))))
        n = int(max_over_ranks(float(n), dev))
        times, wall = [first], wall0
        for _ in range(n - 1):
            t, w = window(graph, args.steps)
            times.append(t)
            wall += w
        return statistics.median(times), len(times), wall

    with ClockSampler(local) as clk:
        cold_s, n_windows, cold_wall = windows(cold_graph)
    warm_s, _, _ = windows(warm_graph)

    # end to end through the public API with host buffers
    pinned = host.pin_memory()
    kv_host = torch.from_numpy(case.kv_lens).pin_memory()
    idx_host = torch.empty((rows, k), dtype=torch.int32).pin_memory()
    dlog = bufs[0]
    e2e_steps = max(1, args.e2e_steps)
    for _ in range(3):
        dlog.copy_(pinned, non_blocking=True)
        kv.copy_(kv_host, non_blocking=True)
        gvr.topk_decode(dlog, kv, case.next_n, case.compress_ratio, k, indices=idx)
        idx_host.copy_(idx, non_blocking=True)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        dlog.copy_(pinned, non_blocking=True)
        kv.copy_(kv_host, non_blocking=True)
        gvr.topk_decode(dlog, kv, case.next_n, case.compress_ratio, k, indices=idx)
        idx_host.copy_(idx, non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_s = f0.elapsed_time(f1) / 1e3
    barrier()

    cold_max = max_over_ranks(cold_s, dev)
    warm_max = max_over_ranks(warm_s, dev)
    e2e_max = max_over_ranks(e2e_s, dev)
    total_rows = sum_over_ranks(float(rows), dev)

    if rank == 0:
        per_launch = cold_s / args.steps
        nbytes = algorithmic_bytes(case, args.values)
        achieved = nbytes / per_launch / 1e9
        peak, peak_kind = measured_peak_hbm()
        warm_per = warm_s / args.steps
        del bufs
        torch.cuda.empty_cache()
        extra = None if args.no_extras else extras(torch, gvr, dev, wsb, peak, head_case=case)
        cpu = None
        if not args.no_cpu_baseline:
            secs, cores, runs, total = time_oracle(case, 0, 5, CPU_BASELINE_S)
            sub = workloads.DecodeCase(case.name, case.logits[:16], case.kv_lens[:16 // case.next_n], case.next_n,
                                       case.compress_ratio, case.k)
            secs1, _, runs1, total1 = time_oracle(sub, 1, 5, CPU_BASELINE_S / 4)
            cpu = {"value": rows / secs, "unit": "rows/s", "cores": cores, "kind": "oracle",
                   "sample": f"all {rows} rows of the batch per run (one step), full sort per row, median of "
                             f"{runs} runs ({total:.1f} s)",
                   "single_thread": {"value": sub.rows / secs1, "unit": "rows/s", "cores": 1,
                                     "sample": f"the batch's first 16 rows per run, one thread, median of {runs1} "
                                               f"runs ({total1:.1f} s)"}}
        clocks = clk.summary()
        line = {
            "metric": METRIC,
            "value": total_rows * args.steps / cold_max,
            "unit": "rows/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": 1e3 * cold_max / args.steps,
            "us_per_row": 1e6 * cold_max / (args.steps * rows),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": config_block(case, ws),
            "timing": {"windows": n_windows, "steps_per_window": args.steps, "window_s": "median",
                       "wall_s": round(cold_wall, 3)},
            "warm_l2": {"value": total_rows * args.steps / warm_max, "unit": "rows/s",
                        "us_per_call": 1e6 * warm_per, "us_per_row": 1e6 * warm_per / rows,
                        "effective_gbs": nbytes / warm_per / 1e9},
            "hbm_gbs_vs_nominal": {"achieved": achieved, "nominal": NOMINAL_HBM_GBS,
                                   "frac": achieved / NOMINAL_HBM_GBS},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": profiled_traffic(kernel), "algorithmic_bytes_per_launch": nbytes,
                         "us_per_launch": 1e6 * per_launch, "kernel": kernel},
            "e2e": {"value": total_rows * e2e_steps / e2e_max, "unit": "rows/s",
                    "h2d_bytes_per_step": int(pinned.numel() * 4 + kv_host.numel() * 4),
                    "d2h_bytes_per_step": int(idx_host.numel() * 4)},
            "gpu_launches": args.steps * n_windows,
            "cpu_baseline": cpu,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"], "samples": clocks["samples"],
                       "window_s": round(cold_wall, 3)},
        }
        if extra:
            line.update(extra)
        print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
