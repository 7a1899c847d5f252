#!/usr/bin/env python3
"""Throughput of the exact per-row top-K on GB300: rows/s, us/row and HBM roofline.

Workload: the decode batch -- 64 requests x next_n = 2 (128 rows), kv_lens
~ U[16384, 524288] uncompressed tokens, compress_ratio 4 (so n up to 131072),
K = 1024, row stride 131072 fp32, scores N(0,1) plus a position-linear bias,
poisoned padding, and three requests at n = K-1, K, K+1.  Synthetic and seeded
(workloads.decode_batch).

One step = one topk_decode call over the whole batch (one kernel launch).

* value (cold L2): the timed region replays a CUDA graph that runs the step on
  R distinct device copies of the batch in turn, R * 64 MiB >> L2 (129 MB), so
  no step finds its scores in L2.  Timed with CUDA events on the launching
  stream, a barrier and torch.cuda.synchronize() on both sides, max over ranks.
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
import re
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
PROFILE_NOTE = os.path.join(ROOT, "profiles", "gvr_topk_kernel_decode_batch.md")


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


def profiled_traffic():
    """dram bytes per launch from the committed ncu summary, if it matches the current kernel."""
    try:
        text = open(PROFILE_NOTE).read()
    except OSError:
        return None
    src = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    tb = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not src or not tb or src.group(1) != source_digest():
        return None
    return float(tb.group(1))


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


def run_sweep(args):
    """Every sweep cell (BS x N x K, decode and prefill), cold and warm L2, one JSON line each;
    then the tail check on the adversarial row and its variants.

    cold: a 512 MiB scrub write before each call; per call CUDA events (median / p99 / max of
    32) and, at finer resolution, the mean over graphs of (scrub + call) minus (scrub) -- the
    rates use the graph mean.  warm: a graph of 100 back-to-back calls on one input."""
    import torch
    import workloads
    import sparse_attention_indexer_exact_gb300 as gvr

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback exists)")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gvr.load_library()
    stream = torch.cuda.current_stream()
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > L2: evicts the scores
    peak, _ = measured_peak_hbm()

    def measure(launch, reps=32, warm_calls=100):
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
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h = torch.cuda.current_stream().cuda_stream
            for _ in range(warm_calls):
                launch(h)
        g.replay()
        torch.cuda.synchronize()
        warm = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            warm.append(e0.elapsed_time(e1) * 1e3 / warm_calls)
        # the event clock ticks in ~2 us steps here, so the cold mean is also taken from graphs:
        # (scrub + call) x R minus (scrub) x R, over R calls
        def graph_of(with_call, r=16):
            gg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gg):
                h = torch.cuda.current_stream().cuda_stream
                for i in range(r):
                    scrub.fill_(i & 255)
                    if with_call:
                        launch(h)
            gg.replay()
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                gg.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1) * 1e3)
            return best / r
        cold_mean = graph_of(True) - graph_of(False)
        cold.sort()
        return (cold[len(cold) // 2], cold[min(len(cold) - 1, int(0.99 * len(cold)))], cold[-1], min(warm),
                cold_mean)

    def emit(tag, case, nbytes, launch):
        med, p99, mx, warm, cmean = measure(launch)
        print(json.dumps({
            "sweep": tag, "bs": case.rows, "n": int(case.meta.get("n", 0)), "k": case.k,
            "cold_us": {"median": med, "p99": p99, "max": mx, "graph_mean": cmean}, "warm_us": warm,
            "rows_per_s_cold": case.rows / (cmean * 1e-6), "us_per_row_cold": cmean / case.rows,
            "algorithmic_bytes": nbytes, "gbs_cold": nbytes / cmean / 1e3, "gbs_warm_effective": nbytes / warm / 1e3,
            "frac_of_8tbs": nbytes / cmean / 1e3 / NOMINAL_HBM_GBS, "frac_of_measured": nbytes / cmean / 1e3 / peak,
            "reachable_60pct": nbytes >= 36e6}), flush=True)
        return cmean

    for n in (16384, 32768, 65536, 131072):
        for bs in (1, 4, 16, 64, 256):
            dcase = workloads.sweep_decode(bs, n, 512)
            lg = torch.from_numpy(dcase.logits).to(dev)
            for k in (512, 1024, 2048):
                dc = workloads.DecodeCase(dcase.name, dcase.logits, dcase.kv_lens, 1, 1, k, {"n": n})
                kv = torch.from_numpy(dc.kv_lens).to(dev)
                idx = torch.empty((bs, k), dtype=torch.int32, device=dev)
                emit("decode", dc, algorithmic_bytes(dc, False),
                     lambda h, lg=lg, kv=kv, idx=idx, k=k: gvr.topk_decode_raw(
                         lg.data_ptr(), lg.stride(0), bs, kv.data_ptr(), 1, 1, k, idx.data_ptr(), None, h))
                ks = torch.from_numpy((np.arange(bs) % 4).astype(np.int32)).to(dev)
                ke = torch.full((bs,), n, dtype=torch.int32, device=dev)
                pc = workloads.PrefillCase(dcase.name, dcase.logits, (np.arange(bs) % 4).astype(np.int32),
                                           np.full(bs, n, np.int32), k, {"n": n})
                emit("prefill", pc, prefill_algorithmic_bytes(pc),
                     lambda h, lg=lg, ks=ks, ke=ke, idx=idx, k=k: gvr.topk_prefill_raw(
                         lg.data_ptr(), lg.stride(0), bs, ks.data_ptr(), ke.data_ptr(), k, idx.data_ptr(), h))
            del lg
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
        for tag, fn in (("blockskip_off", None), ("blockskip_on", bm)):
            if fn is None:
                launch = (lambda h, lg=lg, kv=kv, idx=idx, case=case: gvr.topk_decode_raw(
                    lg.data_ptr(), case.row_stride, case.rows, kv.data_ptr(), case.next_n, case.compress_ratio,
                    case.k, idx.data_ptr(), None, h))
            else:
                launch = (lambda h, lg=lg, kv=kv, idx=idx, case=case, bm=bm: gvr.topk_decode_blockskip_raw(
                    lg.data_ptr(), case.row_stride, case.rows, kv.data_ptr(), case.next_n, case.compress_ratio,
                    case.k, bm.data_ptr(), bm.stride(0), idx.data_ptr(), None, h))
            emit(f"{tag}:{case.name}", case, algorithmic_bytes(case, False), launch)
        del lg, bm
    # tail check: each adversarial variant against a row of the same shape drawn from N(0,1)
    base = workloads.adversarial_row("base")
    g = np.random.default_rng(1049)
    plain = base.logits.copy()
    n0 = int(base.row_lengths()[0])
    plain[0, :n0] = g.standard_normal(n0).astype(np.float32)
    ref_case = workloads.DecodeCase("adversarial_shape_normal", plain, base.kv_lens, 1, base.compress_ratio, base.k,
                                    {"n": n0})

    def adv_launch(case):
        lg = torch.from_numpy(case.logits).to(dev)
        kv = torch.from_numpy(case.kv_lens).to(dev)
        idx = torch.empty((case.rows, case.k), dtype=torch.int32, device=dev)
        return lambda h: gvr.topk_decode_raw(lg.data_ptr(), lg.stride(0), case.rows, kv.data_ptr(), case.next_n,
                                             case.compress_ratio, case.k, idx.data_ptr(), None, h)

    ref_med = emit("tail_reference_normal_row", ref_case, algorithmic_bytes(ref_case, False), adv_launch(ref_case))
    for v in workloads.ADVERSARIAL_VARIANTS:
        c = workloads.adversarial_row(v)
        c.meta["n"] = n0
        med = emit(f"tail_{v}", c, algorithmic_bytes(c, False), adv_launch(c))
        print(json.dumps({"tail_check": v, "ratio_to_normal_row": med / ref_med, "within_2x": med <= 2 * ref_med}),
              flush=True)
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
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["gvr", "reference"], default="gvr")
    ap.add_argument("--copies", type=int, default=16, help="distinct device copies of the batch (cold L2)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--values", action="store_true", help="also write the fp32 values output")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the headline line: every sweep cell and the adversarial tail check")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.sweep:
        return run_sweep(args)

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

    def launch(buf, stream_handle):
        gvr.topk_decode_raw(buf.data_ptr(), stride, rows, kv.data_ptr(), case.next_n, case.compress_ratio, k,
                            idx.data_ptr(), vptr, stream_handle)

    stream = torch.cuda.current_stream()
    for i in range(args.warmup):  # eager warm-up also performs the one-time device set-up
        launch(bufs[i % copies], stream.cuda_stream)
    torch.cuda.synchronize()

    def make_graph(buffers):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h = torch.cuda.current_stream().cuda_stream
            for b in buffers:
                launch(b, h)
        return g

    cold_graph = make_graph(bufs)
    warm_graph = make_graph([bufs[0]] * copies)
    torch.cuda.synchronize()

    def timed(graph, steps):
        reps, rem = divmod(steps, copies)
        graph.replay()  # one untimed replay: graph upload
        torch.cuda.synchronize()
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

    with ClockSampler(local) as clk:
        cold_s, cold_wall = timed(cold_graph, args.steps)
    warm_s, _ = timed(warm_graph, args.steps)

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
            "warm_l2": {"value": total_rows * args.steps / warm_max, "unit": "rows/s",
                        "us_per_call": 1e6 * warm_per, "us_per_row": 1e6 * warm_per / rows,
                        "effective_gbs": nbytes / warm_per / 1e9},
            "hbm_gbs_vs_nominal": {"achieved": achieved, "nominal": NOMINAL_HBM_GBS,
                                   "frac": achieved / NOMINAL_HBM_GBS},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": profiled_traffic(), "algorithmic_bytes_per_launch": nbytes,
                         "us_per_launch": 1e6 * per_launch, "kernel": KERNEL_NAME},
            "e2e": {"value": total_rows * e2e_steps / e2e_max, "unit": "rows/s",
                    "h2d_bytes_per_step": int(pinned.numel() * 4 + kv_host.numel() * 4),
                    "d2h_bytes_per_step": int(idx_host.numel() * 4)},
            "gpu_launches": args.steps,
            "cpu_baseline": cpu,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"], "samples": clocks["samples"],
                       "window_s": round(cold_wall, 3)},
        }
        print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
