"""GPU parity: the CUDA path through the C ABI against the CPU oracle, tie-aware.

Every case runs the library on cuda:0 and the oracle on the host over the same
seeded inputs, then compares row by row with tests/tiecheck.py (short rows by
exact equality; long rows by the set of winners above tau, the exact selected
value multiset and index validity).  The bar is 0 inexact rows.

Cases: the five workloads (single decode row, the 128-row decode batch at full
size, the 4096-row prefill tile, the adversarial row and its variants, sweep
cells), every launch geometry including streamed shares, every forced path of
the method (rescue on an invalid bracket, rescue on overflow, no floor, radix
refine), and the edge cases: empty and short rows at nv in {0, 1, K-1, K, K+1},
misaligned prefill windows with the -inf tie class, clamped windows, MTP rows
with kv_len < next_n, more than 65535 rows, and NaN inside a window (safety
only: K distinct in-window indices).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tiecheck import compare_rows, decode_windows, prefill_windows

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


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


DEV = "cuda:0"


def run_decode(gvr, case, *, values=True, options=None, stats=False):
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    st = None
    if stats:
        st = torch.full((case.rows, 4), -7, dtype=torch.int32, device=DEV)
        options = options or gvr.Options()
        options.row_stats = st.data_ptr()
    idx, vals = gvr.topk_decode(lg, kv, case.next_n, case.compress_ratio, case.k, want_values=values,
                                options=options)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (vals.cpu().numpy() if vals is not None else None), \
        (st.cpu().numpy() if st is not None else None)


def run_prefill(gvr, case, *, options=None, stats=False):
    lg = torch.from_numpy(case.logits).to(DEV)
    ks = torch.from_numpy(case.row_starts).to(DEV)
    ke = torch.from_numpy(case.row_ends).to(DEV)
    st = None
    if stats:
        st = torch.full((case.rows, 4), -7, dtype=torch.int32, device=DEV)
        options = options or gvr.Options()
        options.row_stats = st.data_ptr()
    idx = gvr.topk_prefill(lg, ks, ke, case.k, options=options)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (st.cpu().numpy() if st is not None else None)


def assert_decode_exact(gvr, case, **kw):
    got, vals, st = run_decode(gvr, case, **kw)
    ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
    bad, why = compare_rows(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio), case.k,
                            got, ref, got_values=vals)
    assert bad == 0, f"{case.name}: {bad} inexact rows: {why}"
    return st


def assert_prefill_exact(gvr, case, **kw):
    got, st = run_prefill(gvr, case, **kw)
    ref, _ = oracle.topk_prefill(case.logits, case.row_starts, case.row_ends, case.k)
    bad, why = compare_rows(prefill_windows(case.logits, case.row_starts, case.row_ends), case.k, got, ref)
    assert bad == 0, f"{case.name}: {bad} inexact rows: {why}"
    return st


# ----------------------------------------------------------------------------- the workloads
@pytest.mark.parametrize("values", [False, True])
def test_single_decode_row(gvr, values):
    assert_decode_exact(gvr, workloads.single_decode_row(), values=values)


def test_decode_batch_full_size(gvr):
    st = assert_decode_exact(gvr, workloads.decode_batch(), stats=True)
    n = workloads.decode_batch().row_lengths()
    assert (st[n <= 1024, 0] == 0).all() and (st[n > 1024, 0] >= 1).all()


def test_decode_batch_with_empty_request(gvr):
    case = workloads.decode_batch(requests=64, empty_request=True, stride=32768, kv_hi=131072)
    assert_decode_exact(gvr, case)


@pytest.mark.parametrize("kernel", [0, 4096])
def test_prefill_tile_full_size(gvr, kernel):
    # the cluster kernel by default, the short-row kernel (stride 14848 fits it) when asked for
    st = assert_prefill_exact(gvr, workloads.prefill_tile(), stats=True, options=gvr.Options(flags=kernel))
    assert np.isin(st[:, 0], [0, 1, 10]).all(), "an ordinary N(0,1) tile should never need the rescue"


@pytest.mark.parametrize("variant", workloads.ADVERSARIAL_VARIANTS)
def test_adversarial_row(gvr, variant):
    st = assert_decode_exact(gvr, workloads.adversarial_row(variant), stats=True)
    path = int(st[0, 0])
    if variant == "all_equal":
        assert path == 2  # GMIN == GMAX: invalid bracket
    if variant == "two_valued":
        assert path == 3  # the top bin holds ~n/2 candidates: overflow
    if variant == "neg_inf_tau":
        assert path == 9  # fewer than k finite scores: decided by the first pass (-inf fill)


@pytest.mark.parametrize("bs,n,k", [(1, 16384, 512), (4, 32768, 1024), (16, 65536, 2048), (4, 131072, 512),
                                    (1, 131072, 2048), (64, 16384, 1024), (64, 131072, 512), (16, 65536, 512)])
def test_sweep_cells_decode(gvr, bs, n, k):
    assert_decode_exact(gvr, workloads.sweep_decode(bs, n, k))


@pytest.mark.parametrize("bs,n,k", [(4, 16384, 512), (16, 32768, 2048), (4, 131072, 1024)])
def test_sweep_cells_prefill(gvr, bs, n, k):
    assert_prefill_exact(gvr, workloads.sweep_prefill(bs, n, k))


# ----------------------------------------------------------------------------- geometry and paths
@pytest.mark.parametrize("cs", [1, 2, 4, 8, 16])
def test_every_cluster_size(gvr, cs):
    """Every cluster size: shares from a fraction of one ring stage to many stages."""
    case = workloads.decode_batch(seed=77, requests=6, next_n=2, cr=1, k=1024, stride=40960, kv_lo=900,
                                  kv_hi=40960, boundary=False)
    assert_decode_exact(gvr, case, options=gvr.Options(cluster_size=cs))
    pc = workloads.prefill_tile(seed=78, rows=24, k=512, lengths=(700, 2100, 5000, 9000))
    assert_prefill_exact(gvr, pc, options=gvr.Options(cluster_size=cs))


@pytest.mark.parametrize("stages", [3, 4, 5, 7, 16])
def test_every_ring_depth(gvr, stages):
    """Ring depths wrap the per-slot barrier phases differently; results must not change."""
    case = workloads.decode_batch(seed=79, requests=5, next_n=2, cr=2, k=512, stride=65536, kv_lo=2000,
                                  kv_hi=131072, boundary=False)
    for cs in (1, 8, 16):
        assert_decode_exact(gvr, case, options=gvr.Options(cluster_size=cs, ring_stages=stages))
        assert_decode_exact(gvr, case, options=gvr.Options(cluster_size=cs, ring_stages=stages, flags=1))


@pytest.mark.parametrize("cs", [1, 2, 4])
def test_stage_holding_only_the_partial_vector(gvr, cs):
    """Windows whose last ring stage holds nothing but the partial last vector (every lead)."""
    g = np.random.default_rng(31)
    k, stride = 512, 16384
    rows = []
    for lead in range(4):
        for nfull in (512, 1024, 1536, 2048, 3584):  # whole vectors per CTA share multiple of a stage
            for tailn in (1, 2, 3):
                span = 4 * nfull * cs + tailn
                if span > stride:
                    continue
                ks = lead
                ke = span  # window [lead, span): span - lead scores
                row = workloads.PREFILL_POISON[np.arange(stride) % 4].copy()
                row[ks:ke] = g.standard_normal(ke - ks).astype(np.float32)
                rows.append((row, ks, ke))
    lg = np.stack([r[0] for r in rows])
    case = workloads.PrefillCase("tail_stage", lg, np.array([r[1] for r in rows], np.int32),
                                 np.array([r[2] for r in rows], np.int32), k)
    assert_prefill_exact(gvr, case, options=gvr.Options(cluster_size=cs))
    assert_prefill_exact(gvr, case, options=gvr.Options(cluster_size=cs, flags=1))


@pytest.mark.parametrize("flags,expect", [(1, {4}), (4, {3, 5, 6}), (2, {1}), (8, {1}), (2 | 8, {1}),
                                          (2 | 4, {3, 5, 6}), (4 | 64, {3}), (2 | 4 | 64, {3})])
def test_forced_paths(gvr, flags, expect):
    case = workloads.decode_batch(seed=5, requests=8, next_n=2, cr=4, k=1024, stride=131072,
                                  boundary=False)
    st = assert_decode_exact(gvr, case, options=gvr.Options(flags=flags), stats=True)
    long_rows = case.row_lengths() > case.k
    assert set(np.unique(st[long_rows, 0]).tolist()) <= expect, st[:, 0]
    adv = workloads.adversarial_row("base")
    assert_decode_exact(gvr, adv, options=gvr.Options(flags=flags))
    pc = workloads.prefill_tile(seed=9, rows=32, k=512, lengths=(600, 1800, 3000, 6000))
    assert_prefill_exact(gvr, pc, options=gvr.Options(flags=flags))


def test_radix_refine_large_candidate_sets(gvr):
    """Coarse plateaus give crossing bins with hundreds to thousands of members."""
    g = np.random.default_rng(21)
    rows, stride, k = 12, 65536, 2048
    lg = np.round(g.standard_normal((rows, stride)) * (2.0 + np.arange(rows)[:, None] * 3)).astype(np.float32)
    case = workloads.DecodeCase("plateaus", lg, np.full(rows, stride, np.int32), 1, 1, k)
    st = assert_decode_exact(gvr, case, stats=True)
    assert (st[:, 1] > 256).any(), st


# ----------------------------------------------------------------------------- edge cases
@pytest.mark.parametrize("k", [512, 1024, 2048])
def test_short_row_boundaries(gvr, k):
    ns = [0, 1, k - 1, k, k + 1, k + 2, 2 * k + 3]
    stride = workloads.roundup(2 * k + 8, 64)
    g = np.random.default_rng(k)
    lg = np.empty((len(ns), stride), np.float32)
    for r, n in enumerate(ns):
        lg[r] = g.standard_normal(stride).astype(np.float32)
        lg[r, n:] = workloads.DECODE_POISON[np.arange(n, stride) % 3]
    case = workloads.DecodeCase("short", lg, np.array(ns, np.int32), 1, 1, k)
    assert_decode_exact(gvr, case)


def test_prefill_misaligned_neg_inf_class(gvr):
    """ks % 4 in {0,1,2,3} crossed with a -inf tie class that holds tau; poison all around."""
    g = np.random.default_rng(3)
    k, stride = 512, 8192
    rows = []
    for s in range(4):
        for nv in (513, 700, 3000, 7000):
            ks = 4 * int(g.integers(0, 50)) + s
            nv = min(nv, stride - ks)
            row = workloads.PREFILL_POISON[np.arange(stride) % 4].copy()
            w = g.standard_normal(nv).astype(np.float32)
            w[g.choice(nv, nv - k + 40, replace=False)] = -np.inf
            row[ks:ks + nv] = w
            rows.append((row, ks, ks + nv))
    lg = np.stack([r[0] for r in rows])
    case = workloads.PrefillCase("neg_inf_lead", lg, np.array([r[1] for r in rows], np.int32),
                                 np.array([r[2] for r in rows], np.int32), k)
    got, _ = run_prefill(gvr, case)
    assert got.min() >= 0
    long_rows = case.window_lengths() > k
    st = assert_prefill_exact(gvr, case, stats=True, options=gvr.Options(flags=256))
    assert (st[long_rows, 0] == 9).all(), st[:, 0]  # cluster kernel, tau = -inf: the -inf fill
    st = assert_prefill_exact(gvr, case, stats=True)
    assert (st[long_rows, 0] == 11).all(), st[:, 0]  # by default the short-row kernel: radix over the row
    st = assert_prefill_exact(gvr, case, stats=True, options=gvr.Options(flags=4096))
    assert (st[long_rows, 0] == 11).all(), st[:, 0]  # short-row kernel: radix over the row


def test_prefill_clamped_windows(gvr):
    g = np.random.default_rng(4)
    k, stride = 512, 4096
    lg = g.standard_normal((6, stride)).astype(np.float32)
    ks = np.array([-5, 3000, 100, 2000, -100, 4090], np.int32)
    ke = np.array([1000, 5000, 50, 2000, 9000, 4100], np.int32)
    case = workloads.PrefillCase("clamped", lg, ks, ke, k)
    assert_prefill_exact(gvr, case)


@pytest.mark.parametrize("next_n", [1, 2, 3, 4])
@pytest.mark.parametrize("cr", [1, 4])
def test_mtp_rows(gvr, next_n, cr):
    g = np.random.default_rng(100 * next_n + cr)
    reqs, stride, k = 9, 16384, 512
    kv = g.integers(0, stride * cr, reqs).astype(np.int32)
    kv[0], kv[1], kv[2] = next_n - 1, next_n, cr * k + next_n - 1  # empty, tiny, boundary
    rows = reqs * next_n
    lg = g.standard_normal((rows, stride)).astype(np.float32)
    case = workloads.DecodeCase("mtp", lg, kv, next_n, cr, k)
    n = case.row_lengths()
    for r in range(rows):
        lg[r, n[r]:] = workloads.DECODE_POISON[np.arange(n[r], stride) % 3]
    assert_decode_exact(gvr, case)


def test_more_than_65535_rows(gvr):
    rows, stride, k = 70000, 64, 512
    g = np.random.default_rng(6)
    lg = g.standard_normal((rows, stride)).astype(np.float32)
    kv = g.integers(0, stride + 1, rows).astype(np.int32)
    case = workloads.DecodeCase("many_rows", lg, kv, 1, 1, k)
    assert_decode_exact(gvr, case, values=False)


def test_mixed_row_independence(gvr):
    """304 rows of random, full-length, short, empty and boundary lengths under next_n = 4."""
    g = np.random.default_rng(304)
    next_n, cr, k, stride = 4, 4, 1024, 65536
    kv = g.integers(1, stride * cr, 76).astype(np.int32)
    kv[:6] = [stride * cr, 3, 4, cr * k + 3, cr * (k + 1) + 3, 4 * stride * cr]
    rows = 76 * next_n
    lg = np.empty((rows, stride), np.float32)
    n = workloads.DecodeCase("x", lg, kv, next_n, cr, k).row_lengths()
    for r in range(rows):
        lg[r] = g.standard_normal(stride).astype(np.float32) * (1 + r % 7)
        lg[r, n[r]:] = workloads.DECODE_POISON[np.arange(n[r], stride) % 3]
    assert_decode_exact(gvr, workloads.DecodeCase("mixed", lg, kv, next_n, cr, k))


def test_nan_inside_window_is_safe(gvr):
    g = np.random.default_rng(8)
    rows, stride, k = 4, 8192, 512
    lg = g.standard_normal((rows, stride)).astype(np.float32)
    lg[0, g.choice(stride, 50, replace=False)] = np.nan
    lg[1, :] = np.nan
    lg[2, g.choice(stride, stride - 100, replace=False)] = np.nan
    lg[3, ::2] = np.nan
    lg_t = torch.from_numpy(lg).to(DEV)
    kv = torch.full((rows,), stride, dtype=torch.int32, device=DEV)
    idx, _ = gvr.topk_decode(lg_t, kv, 1, 1, k)
    got = idx.cpu().numpy()
    for r in range(rows):
        assert got[r].min() >= 0 and got[r].max() < stride and np.unique(got[r]).size == k


def test_empty_batch_and_side_stream(gvr):
    lg = torch.zeros((0, 1024), device=DEV)
    kv = torch.zeros((1,), dtype=torch.int32, device=DEV)
    idx, _ = gvr.topk_decode(lg, kv, 1, 1, 512)
    assert idx.shape == (0, 512)
    case = workloads.single_decode_row(seed=55)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lg = torch.from_numpy(case.logits).to(DEV)
        kv = torch.from_numpy(case.kv_lens).to(DEV)
        idx, _ = gvr.topk_decode(lg, kv, 1, 1, case.k)
    s.synchronize()
    ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, 1, 1, case.k)
    bad, why = compare_rows(decode_windows(case.logits, case.kv_lens, 1, 1), case.k, idx.cpu().numpy(), ref)
    assert bad == 0, why


def test_signed_zero_and_inf_classes(gvr):
    for variant in ("signed_zero_tau", "pos_inf_class", "neg_inf_tau"):
        case = workloads.adversarial_row(variant)
        for flags in (0, 1, 4):
            assert_decode_exact(gvr, case, options=gvr.Options(flags=flags))


@pytest.mark.parametrize("cs", [0, 2, 8])
def test_large_crossing_bins(gvr, cs):
    """Crossing bins larger than the candidate buffer whose members every CTA still listed.

    Row families: a plateau of P equal scores on top (tau is the plateau), winners above a
    plateau that holds tau, and a narrow band of distinct values around tau.  Up to 512 members
    per ring stage (1536 with the 3-stage ring forced here), rank 0 collects them in its idle
    ring and refines them alone (path 1 with m > 512); beyond, the cluster's digit passes run
    over the per-CTA lists (path 5), seeded with the crossing bin.  With the automatic ring
    depth the same rows are exact, and a deeper ring takes larger bins on rank 0.
    """
    g = np.random.default_rng(500 + cs)
    k, stride = 512, 65536
    rows = []
    for p in (600, 1000, 1500, 2500, 3500):
        r = g.standard_normal(stride).astype(np.float32)
        r[g.choice(stride, p, replace=False)] = 3.5
        rows.append(r)
    for above, plateau in ((300, 900), (100, 1200), (511, 700), (200, 2600)):
        r = g.standard_normal(stride).astype(np.float32)
        pos = g.choice(stride, above + plateau, replace=False)
        r[pos[:above]] = 5.0 + g.random(above).astype(np.float32)
        r[pos[above:]] = 3.25
        rows.append(r)
    for width in (1e-3, 1e-5):
        r = g.standard_normal(stride).astype(np.float32)
        r[g.choice(stride, 1400, replace=False)] = (4.0 + width * g.random(1400)).astype(np.float32)
        rows.append(r)
    lg = np.stack(rows)
    case = workloads.DecodeCase("plateau_lists", lg, np.full(len(rows), stride, np.int32), 1, 1, k)
    st = assert_decode_exact(gvr, case, options=gvr.Options(cluster_size=cs, ring_stages=3), stats=True)
    if cs != 2:  # two CTAs per row: the lists hold too few of the ~2K above-floor scores
        assert ((st[:, 0] == 1) & (st[:, 1] > 512)).any(), st  # rank 0 refined a large bin
        assert (st[:, 0] == 5).any(), st  # the cluster refined a larger one over the lists
    assert (st[st[:, 0] == 5, 1] > 512).all(), st
    assert (st[(st[:, 0] == 1) & (st[:, 2] == 1), 1] <= 3 * 512).all(), st
    nst = gvr.plan(stride, len(rows), k, gvr.Options(cluster_size=cs))["ring_stages"]
    st = assert_decode_exact(gvr, case, options=gvr.Options(cluster_size=cs), stats=True)
    assert (st[(st[:, 0] == 1) & (st[:, 2] == 1), 1] <= nst * 512).all(), (nst, st)


@pytest.mark.parametrize("cs", [0, 4, 16])
def test_tie_class_fills_the_crossing_bin(gvr, cs):
    """A tie class too large for the lists fills the crossing bin: alone, below a few hundred
    winners, and with a few scores one ulp above it in the same bin (early in a share, where
    they are listed, or late, where the lists are full).  Rows with fewer than K finite scores
    (tau = -inf), and a -inf class that shares its top key digit with finite scores near
    -FLT_MAX."""
    g = np.random.default_rng(601 + cs)
    k, n = 512, 131072
    up = np.nextafter(np.float32(2.0), np.float32(3.0))
    rows = []
    r = np.where(g.random(n) < 0.5, 1.0, 2.0).astype(np.float32)  # two-valued
    rows.append(r)
    r = (0.3 * g.standard_normal(n)).astype(np.float32)  # below 1.6: no score in 2.0's bin
    pos = g.choice(n, n // 2 + 300, replace=False)
    r[pos[:n // 2]] = 2.0
    r[pos[n // 2:]] = (5.0 + g.random(300)).astype(np.float32)  # winners above the tie class
    rows.append(r)
    for where in (slice(n - 8, n - 3), slice(3, 8)):  # one more key in the bin: late, then early
        r = np.where(g.random(n) < 0.5, 1.0, 2.0).astype(np.float32)
        r[where] = up
        rows.append(r)
    r = np.full(n, -np.inf, np.float32)  # tau = -inf
    r[g.choice(n, k - 100, replace=False)] = g.standard_normal(k - 100).astype(np.float32)
    rows.append(r)
    r = np.full(n, -np.inf, np.float32)  # -inf shares its top digit with scores near -FLT_MAX
    pos = g.choice(n, k + 50, replace=False)
    r[pos[:k - 60]] = g.standard_normal(k - 60).astype(np.float32)
    r[pos[k - 60:]] = np.float32(-3.0e38) * (1.0 + g.random(110).astype(np.float32) * 0.1)
    rows.append(r)
    lg = np.stack(rows)
    case = workloads.DecodeCase("tie_class_bins", lg, np.full(len(rows), n, np.int32), 1, 1, k)
    assert_decode_exact(gvr, case, options=gvr.Options(cluster_size=cs))
    for flags in (16, 32):
        assert_decode_deterministic(gvr, case, flags, cluster_size=cs)


def test_big_collect_with_an_overflowed_list(gvr):
    """A crossing bin of ~1K equal scores that all sit in rank 1's first stage: rank 1's list
    overflows, rank 0's does not, so rank 0 still collects the bin in its ring (path 1) while
    rank 1 reads its share again for the collect."""
    g = np.random.default_rng(77)
    k, stride, cs = 512, 65536, 4
    rows = []
    for plateau in (3.0, 3.0, 2.75):
        r = g.standard_normal(stride).astype(np.float32)
        r[1024:2048] = plateau  # stage 1: rank 1 of 4
        r[g.choice(np.arange(4096, stride), 300, replace=False)] = (5.0 + g.random(300)).astype(np.float32)
        rows.append(r)
    lg = np.stack(rows)
    case = workloads.DecodeCase("plateau_in_one_share", lg, np.full(len(rows), stride, np.int32), 1, 1, k)
    st = assert_decode_exact(gvr, case, options=gvr.Options(cluster_size=cs, ring_stages=3), stats=True)
    assert ((st[:, 0] == 1) & (st[:, 1] > 512)).all(), st
    for flags in (16, 32):
        assert_decode_deterministic(gvr, case, flags, cluster_size=cs, ring_stages=3)


def test_relist_after_list_overflow(gvr):
    """No floor (every score listed, so long shares overflow their lists) and no candidate
    buffer: overflowing rows read their share again and select over the re-built lists."""
    case = workloads.decode_batch(seed=15, requests=16, next_n=2, cr=4, k=1024, stride=131072, boundary=False)
    st = assert_decode_exact(gvr, case, options=gvr.Options(flags=2 | 4), stats=True)
    long_rows = case.row_lengths() > case.k
    assert (st[long_rows, 0] == 6).any(), st[:, 0]
    assert ((st[st[:, 0] == 6, 2] // 10) >= 1).any(), st  # some shares were read again
    for flags in (16, 32):
        assert_decode_deterministic(gvr, case, flags, 2 | 4)


def test_far_outlier_samples_trim_the_bins(gvr):
    """Heavy-tailed rows whose samples include a far spike (Pareto tail up to ~10^3 sigma): the
    bins end at a robust sample rank instead of the sampled maximum, so the crossing bin stays
    small (no list refine, no rescue); the spikes above it clamp into the top bin as winners."""
    case = workloads.sweep_decode(64, 32768, 2048)
    st = assert_decode_exact(gvr, case, stats=True)
    assert (st[:, 0] == 1).all() and (st[:, 1] <= 512).all(), st
    g = np.random.default_rng(91)
    k, n = 2048, 32768
    lg = g.standard_normal((4, n)).astype(np.float32)
    nblk = 2048 // 64  # 2048 samples on these rows
    for r in range(4):  # a spike inside a sampled run, plus unsampled spikes elsewhere
        st0 = (5 + r) * (n - 64) // (nblk - 1)
        lg[r, st0 + 7] = 1e3 * (r + 1)
        lg[r, g.choice(n, 50, replace=False)] = (20.0 + 100.0 * g.random(50)).astype(np.float32)
    case = workloads.DecodeCase("sampled_spike", lg, np.full(4, n, np.int32), 1, 1, k)
    for flags in (0, 8):
        st = assert_decode_exact(gvr, case, options=gvr.Options(flags=flags), stats=True)
        assert (st[:, 0] == 1).all() and (st[:, 1] <= 512).all(), st
    for flags in (16, 32):
        assert_decode_deterministic(gvr, case, flags)


def test_second_pass_block_concentrated(gvr):
    """Sink, recent tokens and hot blocks: the block64 runs at both row ends over-represent the
    top, the sampled floor of the plain path is too high and the rows need the second counting
    pass (scores below the floor), then the collect reads the share again.  (Through the
    block-skip entry point the floor is taken again from the interior runs: see
    test_blockskip_gpu.py.)"""
    case = workloads.peaky_decode_batch(requests=24)
    st = assert_decode_exact(gvr, case, stats=True)
    long_rows = case.row_lengths() > case.k
    assert ((st[long_rows, 2] % 10) == 2).sum() >= long_rows.sum() // 2, st
    assert_decode_deterministic(gvr, case, 16)


def test_second_pass_ties_below_floor(gvr):
    """Half of K scores at 10.0 exactly where the block64 runs fall, every other score 0.0: the
    floor sits at 10.0, fewer than K scores reach it, and the second pass counts a warp of equal
    scores at a time (tau = 0.0, a tie class of about n - K/2 members)."""
    k, nv, rows = 1024, 131072, 4
    lg = np.zeros((rows, nv), np.float32)
    nblk = k // 64  # 1024 samples on these rows: k * samples / nv = 8
    for b in range(nblk):
        st0 = b * (nv - 64) // (nblk - 1)
        lg[:, st0:st0 + 32] = 10.0
    lg[1, 5] = -1.0   # a few distinct scores below the tie class
    lg[2, 77777] = 3.0  # one more winner above it
    case = workloads.DecodeCase("ties_below_floor", lg, np.full(rows, nv, np.int32), 1, 1, k)
    for flags in (0, 8):
        st = assert_decode_exact(gvr, case, options=gvr.Options(flags=flags), stats=True)
        assert ((st[:, 2] % 10) == 2).all(), st
    for flags in (16, 32):
        assert_decode_deterministic(gvr, case, flags)


def test_crossing_in_the_floor_bin(gvr):
    """tau inside the bin that holds the sampled floor: one counting pass, candidates >= the floor.

    Each row has a few hundred scores far on top, then a dense class (one histogram bin wide)
    that holds the K-th score and enough block64 samples to put the floor in its bin, and the
    rest far below.
    """
    g = np.random.default_rng(71)
    k, stride = 1024, 131072
    rows = []
    for top, dense, width in ((600, 1500, 0.0), (600, 3000, 1e-3), (300, 5000, 1e-4), (1000, 2500, 0.0)):
        r = (g.standard_normal(stride) - 9.0).astype(np.float32)
        pos = g.choice(stride, top + dense, replace=False)
        r[pos[:top]] = 10.0 + g.random(top).astype(np.float32)
        r[pos[top:]] = (2.0 + width * g.random(dense)).astype(np.float32)
        rows.append(r)
    lg = np.stack(rows)
    case = workloads.DecodeCase("floor_bin", lg, np.full(len(rows), stride, np.int32), 1, 1, k)
    for flags in (0, 8):
        st = assert_decode_exact(gvr, case, options=gvr.Options(flags=flags), stats=True)
        assert (st[:, 2] % 10 == 1).all(), st  # one counting pass per row
        assert set(st[:, 0].tolist()) <= {1, 5, 6}, st


# ----------------------------------------------------------------------------- deterministic mode
def _exact_vs_oracle(got, ref, n, k, ordered):
    """Rows with nv <= k: the identity; long rows: the oracle's set (ordered: its sequence)."""
    bad = []
    for r in range(got.shape[0]):
        if n[r] <= k or ordered:
            ok = np.array_equal(got[r], ref[r])
        else:
            ok = np.array_equal(np.sort(got[r]), np.sort(ref[r]))
        if not ok:
            bad.append(r)
    return bad


def assert_decode_deterministic(gvr, case, flags, extra=0, **opt):
    got, vals, st = run_decode(gvr, case, values=True, options=gvr.Options(flags=flags | extra, **opt),
                               stats=True)
    ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
    n = case.row_lengths()
    bad = _exact_vs_oracle(got, ref, n, case.k, ordered=bool(flags & gvr.FLAG_SORTED))
    assert not bad, f"{case.name}: rows {bad[:8]} differ from the oracle (paths {st[bad[:8], 0]})"
    # values stay the scores at the returned indices
    nbad, why = compare_rows(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio), case.k,
                             got, ref, got_values=vals)
    assert nbad == 0, why
    return st


def assert_prefill_deterministic(gvr, case, flags, extra=0, **opt):
    got, _ = run_prefill(gvr, case, options=gvr.Options(flags=flags | extra, **opt))
    ref, _ = oracle.topk_prefill(case.logits, case.row_starts, case.row_ends, case.k)
    n = np.maximum(np.minimum(case.row_ends, case.logits.shape[1]) - np.maximum(case.row_starts, 0), 0)
    bad = _exact_vs_oracle(got, ref, n, case.k, ordered=bool(flags & gvr.FLAG_SORTED))
    assert not bad, f"{case.name}: rows {bad[:8]} differ from the oracle"


DET_MODES = [16, 32]  # GVR_FLAG_DETERMINISTIC, GVR_FLAG_SORTED


@pytest.mark.parametrize("flags", DET_MODES)
def test_deterministic_workloads(gvr, flags):
    assert_decode_deterministic(gvr, workloads.single_decode_row(), flags)
    assert_decode_deterministic(gvr, workloads.decode_batch(), flags)
    assert_decode_deterministic(gvr, workloads.decode_batch(requests=64, empty_request=True, stride=32768,
                                                           kv_hi=131072), flags)
    assert_prefill_deterministic(gvr, workloads.prefill_tile(), flags)


@pytest.mark.parametrize("flags", DET_MODES)
@pytest.mark.parametrize("variant", workloads.ADVERSARIAL_VARIANTS)
def test_deterministic_ties(gvr, flags, variant):
    """Tie classes at tau far larger than the free slots: the smallest indices must win."""
    case = workloads.adversarial_row(variant)
    for extra in (0, 1, 4):  # histogram path, forced rescue, overflow
        assert_decode_deterministic(gvr, case, flags, extra)


@pytest.mark.parametrize("flags", DET_MODES)
@pytest.mark.parametrize("extra", [0, 1, 4, 8, 2 | 4, 4 | 64])
def test_deterministic_every_path(gvr, flags, extra):
    g = np.random.default_rng(900 + extra)
    rows, stride, k = 10, 65536, 1024
    lg = np.round(g.standard_normal((rows, stride)) * (1.0 + np.arange(rows)[:, None])).astype(np.float32)
    lg[0] = 1.0                      # one class
    lg[1, ::3] = 7.0                 # a class of ~21845 on top
    lg[2, g.choice(stride, 700, replace=False)] = 9.0
    case = workloads.DecodeCase("det_paths", lg, np.full(rows, stride, np.int32), 1, 1, k)
    assert_decode_deterministic(gvr, case, flags, extra)
    assert_decode_deterministic(gvr, case, flags, extra, cluster_size=2)


@pytest.mark.parametrize("flags", DET_MODES)
def test_deterministic_list_refine_and_prefill_leads(gvr, flags):
    g = np.random.default_rng(77)
    k, stride = 512, 65536
    rows = []
    for p in (600, 1500):
        r = g.standard_normal(stride).astype(np.float32)
        r[g.choice(stride, p, replace=False)] = 3.5
        rows.append(r)
    case = workloads.DecodeCase("det_lists", np.stack(rows), np.full(2, stride, np.int32), 1, 1, k)
    st = assert_decode_deterministic(gvr, case, flags)
    assert (st[:, 0] == 5).all(), st
    rows, ks, ke = [], [], []
    for s in range(4):
        row = workloads.PREFILL_POISON[np.arange(8192) % 4].copy()
        w = np.round(g.standard_normal(7000)).astype(np.float32)
        row[s:s + 7000] = w
        rows.append(row)
        ks.append(s)
        ke.append(s + 7000)
    pc = workloads.PrefillCase("det_prefill", np.stack(rows), np.array(ks, np.int32), np.array(ke, np.int32), 512)
    for extra in (0, 1):
        assert_prefill_deterministic(gvr, pc, flags, extra)


# ----------------------------------------------------------------------------- compact lists
CL = 128  # GVR_FLAG_COMPACT_LISTS: (score, 16-bit share position) lists, 16 samples above tau


def test_compact_lists_chosen_for_two_wave_launches(gvr):
    """256 rows of 64K scores at K=1024 would take two waves of 8-CTA clusters; the host halves
    the cluster and takes the compact lists (their instantiation runs by default here)."""
    for bs, n, k in ((256, 65536, 1024), (256, 32768, 2048)):
        case = workloads.sweep_decode(bs, n, k)
        st = assert_decode_exact(gvr, case, stats=True)
        assert (st[:, 0] == 1).all() and (st[:, 2] % 10 == 1).all(), st
        assert gvr.plan(case.row_stride, case.rows, case.k)["cluster_size"] == 4


@pytest.mark.parametrize("flags,expect", [(4, {3, 5, 6}), (2, {1}), (8, {1}), (2 | 4, {3, 5, 6}), (0, {1})])
def test_compact_lists_forced_paths(gvr, flags, expect):
    case = workloads.decode_batch(seed=5, requests=8, next_n=2, cr=4, k=1024, stride=131072,
                                  boundary=False)
    st = assert_decode_exact(gvr, case, options=gvr.Options(flags=flags | CL), stats=True)
    long_rows = case.row_lengths() > case.k
    assert set(np.unique(st[long_rows, 0]).tolist()) <= expect, st[:, 0]
    assert_decode_exact(gvr, workloads.adversarial_row("base"), options=gvr.Options(flags=flags | CL))
    pc = workloads.prefill_tile(seed=9, rows=32, k=512, lengths=(600, 1800, 3000, 6000))
    assert_prefill_exact(gvr, pc, options=gvr.Options(flags=flags | CL))


@pytest.mark.parametrize("cs", [1, 4, 16])
def test_compact_lists_workloads(gvr, cs):
    """The compact format through every list consumer: collect, rank-0 ring collect, the
    cluster selection over lists, the relist, deterministic ties and sorting, prefill windows
    with lead lanes, and shares longer than 64 stages (no 16-bit positions: read again)."""
    o = dict(flags=CL, cluster_size=cs)
    assert_decode_exact(gvr, workloads.decode_batch(requests=16), options=gvr.Options(**o))
    assert_decode_exact(gvr, workloads.single_decode_row(), options=gvr.Options(**o))
    for bs, n, k in ((16, 65536, 512), (4, 131072, 2048), (8, 32768, 1024)):
        assert_decode_exact(gvr, workloads.sweep_decode(bs, n, k), options=gvr.Options(**o))
        assert_prefill_exact(gvr, workloads.sweep_prefill(bs, n, k), options=gvr.Options(**o))
    assert_prefill_exact(gvr, workloads.prefill_tile(seed=11, rows=64, k=2048), options=gvr.Options(**o))
    relist = workloads.decode_batch(seed=15, requests=8, next_n=2, cr=4, k=1024, stride=131072, boundary=False)
    assert_decode_exact(gvr, relist, options=gvr.Options(flags=CL | 2 | 4, cluster_size=cs))
    for flags in (16, 32):
        assert_decode_deterministic(gvr, workloads.decode_batch(requests=8), flags, CL, cluster_size=cs)
        assert_decode_deterministic(gvr, relist, flags, CL | 2 | 4, cluster_size=cs)


def test_compact_lists_large_bins_and_long_shares(gvr):
    """Large crossing bins (rank-0 ring collect, cluster selection over lists) with compact
    lists, and one CTA per 512K-score row: 128 stages, beyond 16-bit positions, so the lists
    are not used and the collect reads the share again."""
    g = np.random.default_rng(123)
    k, stride = 512, 65536
    rows = []
    for p in (600, 1500, 3500):
        r = g.standard_normal(stride).astype(np.float32)
        r[g.choice(stride, p, replace=False)] = 3.5
        rows.append(r)
    case = workloads.DecodeCase("plateau_compact", np.stack(rows), np.full(3, stride, np.int32), 1, 1, k)
    st = assert_decode_exact(gvr, case, options=gvr.Options(flags=CL, cluster_size=4, ring_stages=3), stats=True)
    assert (st[:, 1] > 512).all(), st
    big = workloads.sweep_decode(2, 1 << 19, 1024)
    st = assert_decode_exact(gvr, big, options=gvr.Options(flags=CL, cluster_size=1), stats=True)
    # no list is used: the collect reads the share again, or an overflowing bin goes to the rescue
    assert ((st[:, 0] == 3) | ((st[:, 0] == 1) & (st[:, 2] >= 10))).all(), st


def test_binding_refuses_narrowed_views(gvr):
    # The row stride passed to the library bounds every window; a narrowed view would let a
    # window run past the view's columns, so the binding refuses it.
    buf = torch.zeros((4, 2048), dtype=torch.float32, device=DEV)
    kv = torch.full((4,), 2048, dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError, match="packed"):
        gvr.topk_decode(buf[:, :1024], kv, 1, 1, 512)
    ks = torch.zeros((4,), dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError, match="packed"):
        gvr.topk_prefill(buf[:, :1024], ks, kv, 512)


def test_device_error_reporting(gvr):
    """The failure path, driven by a diagnostic flag instead of a failure: the first row's cluster
    reports a give-up after its first pass completed; that row reads -2 with the device-error
    path, every other row is exact."""
    case = workloads.decode_batch(seed=61, requests=12, next_n=2, cr=4, k=1024, stride=65536,
                                  kv_lo=8192, kv_hi=262144, boundary=False)
    for flags in (2048, 2048 | 16, 2048 | 2):
        got, _, st = run_decode(gvr, case, values=False, options=gvr.Options(flags=flags), stats=True)
        assert (got[0] == -2).all() and st[0, 0] == -1, (flags, got[0][:8], st[0])
        ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
        wins = list(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio))[1:]
        bad, why = compare_rows(iter(wins), case.k, got, ref)  # rows 1.. (row indices kept)
        assert bad == 0, why
        assert (st[1:, 0] >= 0).all()


# ----------------------------------------------------------------------------- dense shares
@pytest.mark.parametrize("flags", [0, 128])  # 128: the compact lists
@pytest.mark.parametrize("cs", [1, 2])
def test_dense_shares(gvr, flags, cs):
    """K = 2048 on windows of a few thousand scores with one or two CTAs per row: the floor lets
    about half of every share through, more than a CTA's list holds, so the first pass only
    counts (hits added one by one, tie runs by popcount), the collect reads the share again
    (winners told from candidates by the crossing bin's edges) and rank 0's candidates go to its
    list area.  Decode with values -- plain, few distinct values, a tie class at the top -- and
    prefill with every lead."""
    g = np.random.default_rng(95 + cs)
    stride, k = 8192, 2048
    kv = np.array([2049, 2500, 3000, 4096, 4097, 5000, 6000, 7000, 8000, 8191, 8192, 2052], np.int32)
    lg = g.standard_normal((kv.size, stride)).astype(np.float32)
    lg[3] = np.round(lg[3] * 2) / 2  # a handful of distinct values: tie runs in the count-only pass
    lg[7, g.choice(7000, 2600, replace=False)] = 9.0  # a tie class above the rest holds tau
    for r, n in enumerate(kv):
        lg[r, n:] = workloads.DECODE_POISON[np.arange(n, stride) % 3]
    case = workloads.DecodeCase("dense_decode", lg, kv, 1, 1, k)
    opts = gvr.Options(cluster_size=cs, flags=flags)
    assert_decode_exact(gvr, case, values=True, options=opts)
    assert_decode_exact(gvr, case, options=opts)
    rows = []
    for r in range(8):
        ks = 4 * int(g.integers(0, 100)) + r % 4
        ke = ks + int(g.integers(2100, 7600))
        row = workloads.PREFILL_POISON[np.arange(stride) % 4].copy()
        row[ks:ke] = g.standard_normal(ke - ks).astype(np.float32)
        rows.append((row, ks, ke))
    pcase = workloads.PrefillCase("dense_prefill", np.stack([x[0] for x in rows]), np.array([x[1] for x in rows], np.int32),
                                  np.array([x[2] for x in rows], np.int32), k)
    assert_prefill_exact(gvr, pcase, options=opts)


# ----------------------------------------------------------------------------- one value above the floor
def test_one_value_above_the_floor(gvr):
    """Rows whose scores at or above the sampled floor are all one value: the tie slots come from
    the first pass's lists when they hold k of them (half the row one value; a top class of signed
    zeros), else from the digit passes (3072 ties, all in the share of one CTA of the cluster,
    more than its lists hold).  Exact with values, and in deterministic mode."""
    g = np.random.default_rng(81)
    stride, k = 131072, 2048
    half = g.standard_normal(stride).astype(np.float32)
    half[g.random(stride) < 0.5] = 7.0
    packed = g.standard_normal(stride).astype(np.float32)
    for s0 in (0, 16384, 32768):  # stage s0 / 1024 of the row: rank 0's for any cluster of <= 16
        packed[s0:s0 + 1024] = 7.0
    zeros = -(np.abs(g.standard_normal(stride)) + 1).astype(np.float32)
    z = g.choice(stride, 5000, replace=False)
    zeros[z] = np.where(np.arange(z.size) % 2 == 0, np.float32(-0.0), np.float32(0.0))
    lg = np.stack([half, packed, zeros])
    case = workloads.DecodeCase("one_value", lg, np.full(3, stride, np.int32), 1, 1, k)
    st = assert_decode_exact(gvr, case, stats=True)
    assert (st[:2, 0] == 3).all(), st  # overflow: the lists cannot hold the crossing bin
    assert st[2, 0] in (1, 5, 6), st  # 5000 ties over every CTA: the lists hold them
    assert_decode_exact(gvr, case, values=True)
    assert_decode_exact(gvr, case, options=gvr.Options(flags=16))


# ----------------------------------------------------------------------------- short-row kernel
SHORT, CLUSTER = 4096, 256


@pytest.mark.parametrize("kernel", [SHORT, CLUSTER])
@pytest.mark.parametrize("bs,n,k", [(1, 16384, 512), (4, 16384, 2048), (16, 16384, 1024), (256, 16384, 512),
                                    (64, 8192, 2048), (3, 4100, 1024)])
def test_short_stride_cells(gvr, kernel, bs, n, k):
    """Rows that fit one CTA's shared memory, through the short-row kernel and the cluster
    kernel: decode and prefill (every lead), heavy-tailed scores."""
    st = assert_decode_exact(gvr, workloads.sweep_decode(bs, n, k), options=gvr.Options(flags=kernel), stats=True)
    if kernel == SHORT:
        assert np.isin(st[:, 0], [0, 10, 11]).all(), st[:, 0]
    assert_prefill_exact(gvr, workloads.sweep_prefill(bs, n, k), options=gvr.Options(flags=kernel))


@pytest.mark.parametrize("values", [False, True])
def test_short_kernel_single_row(gvr, values):
    st = assert_decode_exact(gvr, workloads.single_decode_row(), values=values, stats=True,
                             options=gvr.Options(flags=SHORT))
    assert st[0, 0] == 10
    st = assert_decode_exact(gvr, workloads.single_decode_row(), values=values, stats=True)
    assert st[0, 0] == 10  # the default for a row this short
    st = assert_decode_exact(gvr, workloads.single_decode_row(), values=values, stats=True,
                             options=gvr.Options(flags=CLUSTER))
    assert st[0, 0] in (1, 5, 6)


def test_short_kernel_tie_heavy_rows(gvr):
    """Rows the histogram cannot decide take the exact radix over the staged row:
    one value, two values, a -inf class holding tau, a +inf class, signed zero at tau, plateaus."""
    g = np.random.default_rng(71)
    rows, stride, k = 9, 16384, 1024
    lg = g.standard_normal((rows, stride)).astype(np.float32)
    lg[1] = 2.5
    lg[2] = np.where(g.random(stride) < 0.5, 1.0, 2.0).astype(np.float32)
    lg[3, g.choice(stride, stride - k + 30, replace=False)] = -np.inf
    lg[4, g.choice(stride, k - 3, replace=False)] = np.inf
    lg[5] = -(np.abs(lg[5]) + 1)
    z = g.choice(stride, 3 * k, replace=False)
    lg[5, z[:k // 2]] = np.abs(lg[5, z[:k // 2]]) + 1
    lg[5, z[k // 2:]] = np.where(np.arange(z.size - k // 2) % 2 == 0, np.float32(-0.0), np.float32(0.0))
    lg[6] = np.round(lg[6] * 3)
    lg[7] = np.round(lg[7] * 40) / 40
    lg[8, g.choice(stride, 40, replace=False)] = 1e30  # far outliers stretch the bins
    case = workloads.DecodeCase("short_ties", lg, np.full(rows, stride, np.int32), 1, 1, k)
    for kernel in (SHORT, CLUSTER):
        st = assert_decode_exact(gvr, case, options=gvr.Options(flags=kernel), stats=True)
        if kernel == SHORT:
            assert st[1, 0] == 11 and st[2, 0] == 11 and st[3, 0] == 11, st[:, 0]


def test_short_kernel_device_error_reporting(gvr):
    """The short-row kernel's failure path, driven by the diagnostic flag: row 0 reports a give-up
    once its window has landed; it reads -2 with the device-error path, every other row is exact."""
    case = workloads.sweep_decode(8, 16384, 1024)
    for flags in (SHORT | 2048, SHORT | 2048 | 1):
        got, _, st = run_decode(gvr, case, values=False, options=gvr.Options(flags=flags), stats=True)
        assert (got[0] == -2).all() and st[0, 0] == -1, (flags, got[0][:8], st[0])
        ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
        wins = list(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio))[1:]
        bad, why = compare_rows(iter(wins), case.k, got, ref)  # rows 1.. (row indices kept)
        assert bad == 0, why
        assert np.isin(st[1:, 0], [10, 11]).all(), st[:, 0]


def test_short_kernel_list_overflow(gvr):
    """A cluster of high scores that the block64 samples never see: the floor lets through more
    scores than the kernel lists (4096), and the row takes the exact radix over the window."""
    g = np.random.default_rng(73)
    stride, k = 16384, 512
    lg = g.standard_normal((2, stride)).astype(np.float32)
    nsamp, nv = 512, stride  # K samples in K/64 runs of 64 (the row needs no more)
    nblk = nsamp // 64
    sampled = np.zeros(stride, bool)
    for b in range(nblk):
        st0 = b * (nv - 64) // (nblk - 1)
        sampled[st0:st0 + 64] = True
    hidden = np.flatnonzero(~sampled)[:6000]
    lg[0, hidden] = (5.0 + g.random(hidden.size)).astype(np.float32)
    lg[1, hidden[:3000]] = (5.0 + g.random(3000)).astype(np.float32)  # below the list's capacity
    case = workloads.DecodeCase("hidden_cluster", lg, np.full(2, stride, np.int32), 1, 1, k)
    st = assert_decode_exact(gvr, case, values=True, stats=True)
    assert st[0, 0] == 11, st[:, 0]


def test_short_kernel_boundaries_and_nan(gvr):
    g = np.random.default_rng(72)
    for k in (512, 2048):
        ns = [0, 1, k - 1, k, k + 1, k + 2, 4097, 16384]
        stride = 16384
        lg = g.standard_normal((len(ns), stride)).astype(np.float32)
        for r, n in enumerate(ns):
            lg[r, n:] = workloads.DECODE_POISON[np.arange(n, stride) % 3]
        assert_decode_exact(gvr, workloads.DecodeCase("short_b", lg, np.array(ns, np.int32), 1, 1, k),
                            options=gvr.Options(flags=SHORT))
    lg = g.standard_normal((3, 8192)).astype(np.float32)
    lg[0, ::3] = np.nan
    lg[1, :] = np.nan
    lt = torch.from_numpy(lg).to(DEV)
    idx, _ = gvr.topk_decode(lt, torch.full((3,), 8192, dtype=torch.int32, device=DEV), 1, 1, 512)
    got = idx.cpu().numpy()
    for r in range(3):
        assert got[r].min() >= 0 and got[r].max() < 8192 and np.unique(got[r]).size == 512
