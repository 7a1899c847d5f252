"""Seeded randomized parity: many small decode and prefill batches against the oracle.

Every case draws its own shape (rows, row stride, K, next_n, compress ratio, windows with every
lead and with clamped bounds), its own score distribution per row (normal, heavy-tailed, a few
distinct values, two values, one value, plateaus of equal scores above the rest, signed zeros
at the top, +inf / -inf classes, rows with fewer than K finite scores, hot blocks over a low
background) and its own options (cluster size, deterministic or sorted output, compact lists,
forced paths, the opt-in kernels, per-block score bounds for block skipping: tight, loose, +inf or
with NaN entries).  The comparison is the tie-aware one of ``tiecheck``; sorted
and deterministic calls must equal the oracle's arrays.  The draws are seeded: a failure names
its case number and reproduces.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from test_blockskip_gpu import block_bounds
from tiecheck import compare_rows, decode_windows, prefill_windows

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# option draws: (cluster_size, flags); 16/32 deterministic / sorted, 128 compact lists, 8 radix
# refine, 2 no floor, 4 zero candidate capacity, 64 streamed rescue, 1 forced rescue,
# 256 cluster kernel, 1024 balanced split kernel, 4096 short-row kernel, 8192 block-skip gate always on
OPTION_DRAWS = [(0, 0), (0, 0), (0, 0), (0, 16), (0, 32), (0, 128), (0, 8), (0, 2), (0, 4), (0, 4 | 64), (0, 1),
                (0, 256), (0, 4096), (1, 0), (2, 0), (4, 0), (8, 0), (2, 128), (4, 16), (0, 128 | 32),
                (0, 1024), (0, 1024 | 16), (0, 8192), (2, 8192 | 128), (0, 8192 | 2)]


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


def draw_row(g, n: int, k: int) -> np.ndarray:
    """n scores of one of the distributions above (fp32)."""
    kind = int(g.integers(0, 11))
    x = g.standard_normal(n).astype(np.float32)
    if kind == 1:  # heavy tail
        sel = g.random(n) < 0.01
        x[sel] += (g.random(sel.sum()) ** (-1 / 1.5)).astype(np.float32)
    elif kind == 2:  # a few distinct values
        x = np.round(x * 2) / 2
    elif kind == 3:  # two values
        x = np.where(g.random(n) < 0.5, np.float32(1.0), np.float32(2.0)).astype(np.float32)
    elif kind == 4:  # one value
        x[:] = np.float32(g.standard_normal())
    elif kind == 5:  # a plateau above the rest holding tau, or wholly above it
        m = int(g.integers(1, 3 * k)) if n > 1 else 1
        x[g.choice(n, min(m, n), replace=False)] = np.float32(7.5)
    elif kind == 6:  # signed zeros at the top
        x = -(np.abs(x) + 1)
        z = g.choice(n, min(n, int(g.integers(1, 2 * k))), replace=False)
        x[z] = np.where(np.arange(z.size) % 2 == 0, np.float32(-0.0), np.float32(0.0))
    elif kind == 7:  # +inf and -inf classes
        x[g.random(n) < 0.05] = np.inf
        x[g.random(n) < 0.2] = -np.inf
    elif kind == 8:  # fewer than k finite scores (tau = -inf)
        x[g.choice(n, max(0, n - int(g.integers(0, k))), replace=False)] = -np.inf
    elif kind == 9:  # hot blocks over a low background, hot ends
        hot = np.repeat(g.random((n + 31) // 32) < 0.03, 32)[:n]
        x = x - 4 + 5 * hot.astype(np.float32)
        x[:64] += 5
        x[-64:] += 5
    elif kind == 10:  # a linear position bias
        x = x + np.float32(g.random() * 3) * np.arange(n, dtype=np.float32) / max(n, 1)
    return x.astype(np.float32)


def decode_case(g, idx: int):
    k = int(g.choice([512, 1024, 2048]))
    next_n = int(g.integers(1, 4))
    cr = int(g.choice([1, 1, 4]))
    requests = int(g.integers(1, 7))
    rows = requests * next_n
    stride = 4 * int(g.integers(16, 10001))
    # lengths around k and up to past the stride (clamped), some requests with kv_len < next_n
    kv = np.empty(requests, np.int64)
    for q in range(requests):
        c = int(g.integers(0, 5))
        if c == 0:
            kv[q] = int(g.integers(0, next_n + 1))
        elif c == 1:
            kv[q] = cr * (k + int(g.integers(-2, 3))) + next_n - 1
        else:
            kv[q] = int(g.integers(next_n, cr * stride + 2 * next_n + 1))
    kv = kv.astype(np.int32)
    lg = np.empty((rows, stride), np.float32)
    case = workloads.DecodeCase(f"fuzz_decode_{idx}", lg, kv, next_n, cr, k)
    n = case.row_lengths()
    for r in range(rows):
        lg[r, :n[r]] = draw_row(g, int(n[r]), k)
        lg[r, n[r]:] = workloads.DECODE_POISON[np.arange(n[r], stride) % 3]
    return case


def prefill_case(g, idx: int):
    k = int(g.choice([512, 1024, 2048]))
    rows = int(g.integers(1, 13))
    stride = 4 * int(g.integers(16, 8001))
    ks = np.empty(rows, np.int64)
    ke = np.empty(rows, np.int64)
    lg = np.empty((rows, stride), np.float32)
    for r in range(rows):
        a = int(g.integers(-8, stride))
        b = a + int(g.integers(-4, stride + 8))
        ks[r], ke[r] = a, b
        lg[r] = workloads.PREFILL_POISON[np.arange(stride) % 4]
        lo, hi = max(a, 0), min(max(b, 0), stride)
        if hi > lo:
            lg[r, lo:hi] = draw_row(g, hi - lo, k)
    return workloads.PrefillCase(f"fuzz_prefill_{idx}", lg, ks.astype(np.int32), ke.astype(np.int32), k)


def exact_equal(got, ref, n, k):
    """Rows that differ from the oracle's arrays (deterministic / sorted calls)."""
    bad = []
    for r in range(got.shape[0]):
        if n[r] <= k:
            if not np.array_equal(got[r], ref[r]):
                bad.append(r)
        elif not np.array_equal(np.sort(got[r]), np.sort(ref[r])):
            bad.append(r)
    return bad


@pytest.mark.parametrize("case_no", range(120))
def test_fuzz_decode(gvr, case_no):
    g = np.random.default_rng(7000 + case_no)
    case = decode_case(g, case_no)
    cs, flags = OPTION_DRAWS[int(g.integers(0, len(OPTION_DRAWS)))]
    values = bool(g.integers(0, 2))
    # block bounds on every call of the always-skip option and on a quarter of the others; that
    # entry point takes no workspace, so the balanced kernel's options are dropped there
    bm = None
    if flags & 8192 or g.random() < 0.25:
        kind = ["exact", "exact", "loose", "inf", "nan"][int(g.integers(0, 5))]
        bm = torch.from_numpy(block_bounds(case, kind, seed=case_no)).to(DEV)
        flags &= ~(512 | 1024)
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    idx, vals = gvr.topk_decode(lg, kv, case.next_n, case.compress_ratio, case.k, want_values=values,
                                options=gvr.Options(cluster_size=cs, flags=flags), block_max=bm)
    torch.cuda.synchronize()
    got = idx.cpu().numpy()
    gv = vals.cpu().numpy() if vals is not None else None
    ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
    bad, why = compare_rows(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio), case.k,
                            got, ref, got_values=gv)
    assert bad == 0, f"{case.name} (cs={cs}, flags={flags}, values={values}, bounds={bm is not None}): {why}"
    if flags & (16 | 32):
        n = case.row_lengths()
        rows = exact_equal(got, ref, n, case.k) if flags & 16 and not flags & 32 else \
            [r for r in range(got.shape[0]) if not np.array_equal(got[r], ref[r])]
        assert not rows, f"{case.name} (flags={flags}): rows {rows[:8]} differ from the oracle's arrays"


@pytest.mark.parametrize("case_no", range(80))
def test_fuzz_prefill(gvr, case_no):
    g = np.random.default_rng(9000 + case_no)
    case = prefill_case(g, case_no)
    cs, flags = OPTION_DRAWS[int(g.integers(0, len(OPTION_DRAWS)))]
    flags &= ~8192  # prefill takes no block bounds
    lg = torch.from_numpy(case.logits).to(DEV)
    ks = torch.from_numpy(case.row_starts).to(DEV)
    ke = torch.from_numpy(case.row_ends).to(DEV)
    idx = gvr.topk_prefill(lg, ks, ke, case.k, options=gvr.Options(cluster_size=cs, flags=flags))
    torch.cuda.synchronize()
    got = idx.cpu().numpy()
    ref, _ = oracle.topk_prefill(case.logits, case.row_starts, case.row_ends, case.k)
    bad, why = compare_rows(prefill_windows(case.logits, case.row_starts, case.row_ends), case.k, got, ref)
    assert bad == 0, f"{case.name} (cs={cs}, flags={flags}): {why}"
    if flags & (16 | 32):
        n = np.maximum(np.minimum(case.row_ends, case.logits.shape[1]) - np.maximum(case.row_starts, 0), 0)
        rows = exact_equal(got, ref, n, case.k) if flags & 16 and not flags & 32 else \
            [r for r in range(got.shape[0]) if not np.array_equal(got[r], ref[r])]
        assert not rows, f"{case.name} (flags={flags}): rows {rows[:8]} differ from the oracle's arrays"
