"""CUDA-graph capture and replay with the row lengths growing in place.

One launch is captured with fixed buffers; between replays the device-resident kv_lens
(and the scores) change in place, so rows cross the short-row boundary nv = K, the ring
residency boundary and the full stride while the graph stays the same.  Every replay is
compared with the oracle for the lengths of that step, which shows that the call reads
nothing on the host and takes every per-row decision on the device ("Self-sampling GVR
V2", CUDA-graph-safe per-row decisions; MTP window formula of run_varlen).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tiecheck import compare_rows, decode_windows

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def gvr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_indexer_exact_gb300 import _build
    _build.build_library()
    import sparse_attention_indexer_exact_gb300 as mod
    mod.load_library()
    torch.cuda.set_device(0)
    return mod


def _kv_schedule(k, cr, next_n, stride, steps):
    """Per-request kv_len at each step: rows start below K and grow past K, past one ring stage
    per CTA and up to the stride (clamped there)."""
    starts = np.array([cr * (k - 4) + next_n - 1, cr * (k - 1) + next_n - 1, cr * 4096, 1, next_n - 1,
                       cr * (stride - 40)], np.int64)
    grow = np.array([cr, cr, cr * 4096, cr * 3000, 7, cr * 64], np.int64)
    return [np.minimum(starts + s * grow, cr * stride + next_n).astype(np.int32) for s in range(steps)]


@pytest.mark.parametrize("stride,flags", [(65536, 0), (65536, 32), (16384, 0)])
def test_graph_replay_with_growing_kv_lens(gvr, stride, flags):
    """The cluster kernel (65536-score rows) and, for 16384-score rows, the short-row kernel."""
    k, cr, next_n = 1024, 4, 2
    sched = _kv_schedule(k, cr, next_n, stride, steps=6)
    reqs = len(sched[0])
    rows = reqs * next_n
    g = np.random.default_rng(2024)
    lg = torch.empty((rows, stride), dtype=torch.float32, device=DEV)
    kv = torch.empty((reqs,), dtype=torch.int32, device=DEV)
    idx = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    vals = torch.empty((rows, k), dtype=torch.float32, device=DEV)
    opts = gvr.Options(flags=flags)

    def host_step(step):
        x = g.standard_normal((rows, stride)).astype(np.float32)
        if step % 2:
            x = np.round(x * 2).astype(np.float32)  # tie-heavy steps
        case = workloads.DecodeCase("graph", x, sched[step], next_n, cr, k)
        n = case.row_lengths()
        for r in range(rows):
            x[r, n[r]:] = workloads.DECODE_POISON[np.arange(n[r], stride) % 3]
        return case

    first = host_step(0)
    lg.copy_(torch.from_numpy(first.logits))
    kv.copy_(torch.from_numpy(first.kv_lens))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up launch outside the capture
        gvr.topk_decode(lg, kv, next_n, cr, k, indices=idx, values=vals, options=opts)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert (gvr.plan(stride, rows, k, opts)["threads"] == 1024) == (stride <= 16384)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gvr.topk_decode(lg, kv, next_n, cr, k, indices=idx, values=vals, options=opts)
    seen_short = seen_long = False
    for step in range(len(sched)):
        case = host_step(step)
        lg.copy_(torch.from_numpy(case.logits))
        kv.copy_(torch.from_numpy(case.kv_lens))
        idx.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        got, gv = idx.cpu().numpy(), vals.cpu().numpy()
        ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, next_n, cr, k)
        n = case.row_lengths()
        seen_short |= bool((n <= k).any())
        seen_long |= bool((n > k).any())
        if flags & gvr.FLAG_SORTED:
            assert np.array_equal(got, ref), f"step {step}: sorted output differs from the oracle"
        bad, why = compare_rows(decode_windows(case.logits, case.kv_lens, next_n, cr), k, got, ref, got_values=gv)
        assert bad == 0, f"step {step}: {why}"
    assert seen_short and seen_long
