"""GPU parity of the balanced (split) kernel behind topk_decode_ws / topk_prefill_ws.

The balanced kernel cuts the batch's valid scores into equal chunks on the device, publishes the
scores at or above each row's sampled floor to a workspace and lets the last chunk of a row
select it.  These cases force it (GVR_FLAG_SPLIT_KERNEL) or its exact lone path
(GVR_FLAG_SPLIT_ALONE) and compare with the CPU oracle tie-aware, 0 inexact rows, covering:
chunk boundaries inside a row (every lead, the partial last vector in the last chunk), rows of
very different lengths, short / empty / boundary rows, tie-heavy and -inf rows that the
published scores cannot decide, repeated calls and CUDA-graph replay (the workspace must come
back zero-filled), and the host's fall back to the cluster kernel for calls it does not fit.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tiecheck import compare_rows, decode_windows, prefill_windows

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SPLIT, ALONE, CLUSTER = 1024, 512 | 1024, 256


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


@pytest.fixture(scope="module")
def ws(gvr):
    return torch.zeros(gvr.workspace_size(), dtype=torch.uint8, device=DEV)


def decode(gvr, ws, case, flags, values=True):
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    idx = torch.full((case.rows, case.k), -9, dtype=torch.int32, device=DEV)
    vals = torch.empty((case.rows, case.k), dtype=torch.float32, device=DEV) if values else None
    st = torch.full((case.rows, 4), -7, dtype=torch.int32, device=DEV)
    opts = gvr.Options(flags=flags, row_stats=st.data_ptr())
    gvr.topk_decode_ws_raw(lg.data_ptr(), lg.shape[1], case.rows, kv.data_ptr(), case.next_n, case.compress_ratio,
                           case.k, idx.data_ptr(), vals.data_ptr() if values else None, ws.data_ptr(), ws.numel(),
                           torch.cuda.current_stream().cuda_stream, opts)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (vals.cpu().numpy() if values else None), st.cpu().numpy()


def prefill(gvr, ws, case, flags):
    lg = torch.from_numpy(case.logits).to(DEV)
    ks = torch.from_numpy(case.row_starts).to(DEV)
    ke = torch.from_numpy(case.row_ends).to(DEV)
    idx = torch.full((case.rows, case.k), -9, dtype=torch.int32, device=DEV)
    st = torch.full((case.rows, 4), -7, dtype=torch.int32, device=DEV)
    opts = gvr.Options(flags=flags, row_stats=st.data_ptr())
    gvr.topk_prefill_ws_raw(lg.data_ptr(), lg.shape[1], case.rows, ks.data_ptr(), ke.data_ptr(), case.k,
                            idx.data_ptr(), ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream, opts)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), st.cpu().numpy()


def workspace_is_clean(ws):
    return int(ws[:2048].count_nonzero().item()) == 0  # the per-row arrival counters


def check_decode(gvr, ws, case, flags, values=True):
    got, vals, st = decode(gvr, ws, case, flags, values)
    ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
    bad, why = compare_rows(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio), case.k,
                            got, ref, got_values=vals)
    assert bad == 0, f"{case.name} flags={flags}: {bad} inexact rows: {why}"
    assert workspace_is_clean(ws), "the workspace must come back zero-filled"
    return st


def check_prefill(gvr, ws, case, flags):
    got, st = prefill(gvr, ws, case, flags)
    ref, _ = oracle.topk_prefill(case.logits, case.row_starts, case.row_ends, case.k)
    bad, why = compare_rows(prefill_windows(case.logits, case.row_starts, case.row_ends), case.k, got, ref)
    assert bad == 0, f"{case.name} flags={flags}: {bad} inexact rows: {why}"
    assert workspace_is_clean(ws), "the workspace must come back zero-filled"
    return st


def long_paths(case, st):
    return set(np.unique(st[case.row_lengths() > case.k, 0]).tolist())


# ----------------------------------------------------------------------------- workloads
def test_decode_batch_full_size(gvr, ws):
    case = workloads.decode_batch()
    st = check_decode(gvr, ws, case, SPLIT)
    assert long_paths(case, st) == {7}, st[:, 0]
    assert (st[case.row_lengths() <= case.k, 0] == 0).all()
    assert st[:, 2].max() > 1, "long rows span several chunks"


def test_decode_batch_lone_path(gvr, ws):
    case = workloads.decode_batch(seed=11, requests=24, stride=32768, kv_lo=1, kv_hi=131072)
    st = check_decode(gvr, ws, case, ALONE)
    assert long_paths(case, st) <= {8}


@pytest.mark.parametrize("flags", [SPLIT, ALONE])
def test_single_rows(gvr, ws, flags):
    check_decode(gvr, ws, workloads.single_decode_row(), flags)
    check_decode(gvr, ws, workloads.single_decode_row(seed=5, n=100000, k=2048), flags, values=False)


@pytest.mark.parametrize("variant", workloads.ADVERSARIAL_VARIANTS)
def test_adversarial_rows(gvr, ws, variant):
    check_decode(gvr, ws, workloads.adversarial_row(variant), SPLIT)


@pytest.mark.parametrize("bs,n,k", [(4, 16384, 512), (16, 65536, 2048), (64, 131072, 1024), (256, 32768, 512),
                                    (2, 131072, 2048)])
def test_sweep_cells(gvr, ws, bs, n, k):
    check_decode(gvr, ws, workloads.sweep_decode(bs, n, k), SPLIT, values=False)
    check_prefill(gvr, ws, workloads.sweep_prefill(bs, n, k), SPLIT)


def test_prefill_tile_subset(gvr, ws):
    full = workloads.prefill_tile()
    sel = np.r_[np.arange(0, 4096, 16), np.arange(4090, 4096)]  # 262 rows incl. nv = K-1, K, K+1
    case = workloads.PrefillCase("tile_subset", np.ascontiguousarray(full.logits[sel]), full.row_starts[sel],
                                 full.row_ends[sel], full.k)
    check_prefill(gvr, ws, case, SPLIT)


# ----------------------------------------------------------------------------- chunk geometry
def test_uneven_rows_every_lead(gvr, ws):
    """Rows from just above K to the full stride, window starts at every lead, partial last
    vectors: chunk boundaries fall inside rows, the lead sits in chunk 0, the tail in the last."""
    g = np.random.default_rng(41)
    k, stride = 1024, 98304
    starts, ends, rows = [], [], []
    for lead in range(4):
        for nv in (k + 1, 3 * k + 5, 4096, 4097, 20000, 65535, 98304 - 8, 98304 - lead):
            ks = lead if nv + lead <= stride else 0
            ke = min(stride, ks + nv)
            row = workloads.PREFILL_POISON[np.arange(stride) % 4].copy()
            row[ks:ke] = (g.standard_normal(ke - ks) + np.linspace(0, 2, ke - ks)).astype(np.float32)
            rows.append(row)
            starts.append(ks)
            ends.append(ke)
    case = workloads.PrefillCase("uneven_leads", np.stack(rows), np.array(starts, np.int32), np.array(ends, np.int32),
                                 k)
    st = check_prefill(gvr, ws, case, SPLIT)
    assert set(st[:, 0].tolist()) <= {7, 8}
    check_prefill(gvr, ws, case, ALONE)


def test_short_empty_and_boundary_rows(gvr, ws):
    g = np.random.default_rng(42)
    for k in (512, 2048):
        ns = [0, 1, k - 1, k, k + 1, 2 * k, 5000, 0, k + 2]
        stride = 8192
        lg = g.standard_normal((len(ns), stride)).astype(np.float32)
        for r, n in enumerate(ns):
            lg[r, n:] = workloads.DECODE_POISON[np.arange(n, stride) % 3]
        check_decode(gvr, ws, workloads.DecodeCase("short", lg, np.array(ns, np.int32), 1, 1, k), SPLIT)


def test_all_rows_short(gvr, ws):
    g = np.random.default_rng(43)
    lg = g.standard_normal((40, 1024)).astype(np.float32)
    check_decode(gvr, ws, workloads.DecodeCase("all_short", lg, g.integers(0, 1025, 40).astype(np.int32), 1, 1,
                                               1024), SPLIT)


def test_tie_heavy_and_neg_inf_rows(gvr, ws):
    """Rows the published scores cannot decide (ties in the crossing bin, fewer than K finite
    scores, one value everywhere) take the lone path; the rest of the batch is unaffected."""
    g = np.random.default_rng(44)
    rows, stride, k = 8, 32768, 1024
    lg = g.standard_normal((rows, stride)).astype(np.float32)
    lg[1] = 3.0
    lg[2] = np.where(g.random(stride) < 0.5, 1.0, 2.0).astype(np.float32)
    lg[3, g.choice(stride, stride - k + 9, replace=False)] = -np.inf
    lg[4] = np.round(lg[4] * 2) / 2
    lg[5, g.choice(stride, 3000, replace=False)] = np.inf
    lg[6] = -0.0
    lg[6, g.choice(stride, 500, replace=False)] = 0.0
    case = workloads.DecodeCase("ties", lg, np.full(rows, stride, np.int32), 1, 1, k)
    st = check_decode(gvr, ws, case, SPLIT)
    assert st[0, 0] == 7 and st[7, 0] == 7 and st[1, 0] == 8


def test_nan_inside_window_is_safe(gvr, ws):
    g = np.random.default_rng(45)
    rows, stride, k = 4, 8192, 512
    lg = g.standard_normal((rows, stride)).astype(np.float32)
    lg[0, g.choice(stride, 50, replace=False)] = np.nan
    lg[1, :] = np.nan
    lg[2, g.choice(stride, stride - 100, replace=False)] = np.nan
    lg[3, ::2] = np.nan
    case = workloads.DecodeCase("nan", lg, np.full(rows, stride, np.int32), 1, 1, k)
    got, _, _ = decode(gvr, ws, case, SPLIT, values=False)
    for r in range(rows):
        assert got[r].min() >= 0 and got[r].max() < stride and np.unique(got[r]).size == k
    assert workspace_is_clean(ws)


# ----------------------------------------------------------------------------- calls and dispatch
def test_repeated_calls_and_graph_replay(gvr, ws):
    """The last chunk of each row resets its counter: back-to-back calls and graph replays with
    kv_lens changed in place stay exact."""
    case = workloads.decode_batch(seed=46, requests=32, stride=65536, kv_lo=8192, kv_hi=262144)
    for _ in range(3):
        check_decode(gvr, ws, case, SPLIT)
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    idx = torch.empty((case.rows, case.k), dtype=torch.int32, device=DEV)
    opts = gvr.Options(flags=SPLIT)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gvr.topk_decode_ws_raw(lg.data_ptr(), lg.shape[1], case.rows, kv.data_ptr(), case.next_n,
                               case.compress_ratio, case.k, idx.data_ptr(), None, ws.data_ptr(), ws.numel(),
                               torch.cuda.current_stream().cuda_stream, opts)
    rng = np.random.default_rng(47)
    for rep in range(4):
        # any length up to the one the scores were drawn for (beyond it lies the poisoned pad)
        kv_h = rng.integers(1, case.kv_lens.astype(np.int64) + 1).astype(np.int32)
        kv_h[0] = case.k * case.compress_ratio + case.next_n - 1 + 2 * rep  # crosses nv = K
        kv.copy_(torch.from_numpy(kv_h))
        g.replay()
        torch.cuda.synchronize()
        c2 = workloads.DecodeCase("replay", case.logits, kv_h, case.next_n, case.compress_ratio, case.k)
        ref, _, _ = oracle.topk_decode(c2.logits, kv_h, c2.next_n, c2.compress_ratio, c2.k)
        bad, why = compare_rows(decode_windows(c2.logits, kv_h, c2.next_n, c2.compress_ratio), c2.k,
                                idx.cpu().numpy(), ref)
        assert bad == 0, why
        assert workspace_is_clean(ws)


def test_calls_the_balanced_kernel_does_not_fit(gvr, ws):
    """More rows than the balanced grid can hold, or cluster tuning, run the other kernels as a
    plain call would (and leave the workspace alone); GVR_FLAG_CLUSTER_KERNEL the cluster kernel."""
    case = workloads.decode_batch(seed=48, requests=300, next_n=2, stride=8192, kv_lo=1, kv_hi=32768)
    st = check_decode(gvr, ws, case, SPLIT, values=False)  # 600 rows > 512: a plain call's kernel
    assert long_paths(case, st) <= {10, 11}  # the short-row kernel, for rows this short
    small = workloads.decode_batch(seed=49, requests=8, stride=16384, kv_lo=1, kv_hi=65536)
    st = check_decode(gvr, ws, small, CLUSTER)
    assert long_paths(small, st) <= {1, 2, 3, 5, 6}


def test_workspace_errors(gvr, ws):
    case = workloads.decode_batch(seed=50, requests=4, stride=8192, kv_lo=1, kv_hi=32768)
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    idx = torch.empty((case.rows, case.k), dtype=torch.int32, device=DEV)
    h = torch.cuda.current_stream().cuda_stream
    for ptr, size in ((0, ws.numel()), (ws.data_ptr() + 4, ws.numel() - 4), (ws.data_ptr(), ws.numel() - 1)):
        with pytest.raises(gvr.GvrError) as e:
            gvr.topk_decode_ws_raw(lg.data_ptr(), lg.shape[1], case.rows, kv.data_ptr(), case.next_n,
                                   case.compress_ratio, case.k, idx.data_ptr(), None, ptr, size, h,
                                   gvr.Options(flags=SPLIT))
        assert e.value.status == 7
