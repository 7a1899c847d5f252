"""Block-skip first pass (topk_decode_blockskip) against the oracle.

The block-maxima side tensor bounds every 32-score block of a row's window ("Block-skip fast
path for self-sampling GVR top-K decode", opt-in row pass); the first counting pass reads
only the blocks whose bound reaches the sampled floor.  For any valid bounds the selection is
the exact one: exact maxima, loose bounds, +inf (nothing skipped) and NaN bounds (read), on
every workload, every forced path and in deterministic / sorted mode -- through the per-row gate
and with blocks skipped on every row.
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


def block_bounds(case, kind, seed=0):
    """fp32 [rows, ceil(stride / 32) + 2]: per 32-column block, a bound of the window's scores."""
    nb = (case.row_stride + 31) // 32
    out = np.full((case.rows, nb + 2), -np.inf, np.float32)
    n = case.row_lengths()
    g = np.random.default_rng(seed)
    for r in range(case.rows):
        if n[r] == 0:
            continue
        x = np.full(((n[r] + 31) // 32) * 32, -np.inf, np.float32)
        x[:n[r]] = case.logits[r, :n[r]]
        m = x.reshape(-1, 32).max(axis=1)
        if kind == "loose":
            m = m + np.abs(g.standard_normal(m.size)).astype(np.float32)
        elif kind == "inf":
            m[:] = np.inf
        elif kind == "nan":
            m[g.random(m.size) < 0.1] = np.nan
        out[r, :m.size] = m
    return out


ALWAYS = 8192  # GVR_FLAG_BLOCKSKIP_ALWAYS: skip blocks whatever the samples' estimate


def assert_blockskip_exact(gvr, case, kind="exact", flags=0, seed=0):
    """Exact with the gate (the samples decide per row between skipping and the staged pass)
    and with blocks skipped on every row."""
    bm = torch.from_numpy(block_bounds(case, kind, seed)).to(DEV)
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
    for f in (flags, flags | ALWAYS):
        st = torch.full((case.rows, 4), -7, dtype=torch.int32, device=DEV)
        opts = gvr.Options(flags=f)
        opts.row_stats = st.data_ptr()
        idx, vals = gvr.topk_decode(lg, kv, case.next_n, case.compress_ratio, case.k, want_values=True, options=opts,
                                    block_max=bm)
        torch.cuda.synchronize()
        got, gv = idx.cpu().numpy(), vals.cpu().numpy()
        bad, why = compare_rows(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio), case.k,
                                got, ref, got_values=gv)
        assert bad == 0, f"{case.name}/{kind}/{f}: {bad} inexact rows: {why}"
        if f & 32:
            assert np.array_equal(got, ref)
    return st.cpu().numpy()


@pytest.mark.parametrize("kind", ["exact", "loose", "inf", "nan"])
def test_blockskip_decode_batch(gvr, kind):
    assert_blockskip_exact(gvr, workloads.decode_batch(), kind, seed=3)


@pytest.mark.parametrize("kind", ["exact", "loose"])
def test_blockskip_peaky_batch(gvr, kind):
    """Block-concentrated rows, where most blocks fall below the floor and are never read."""
    assert_blockskip_exact(gvr, workloads.peaky_decode_batch(), kind, seed=8)
    assert_blockskip_exact(gvr, workloads.peaky_decode_batch(requests=8, next_n=3, hot_frac=0.002), kind, 32)


def test_blockskip_block_concentrated_floor(gvr):
    """On block-concentrated rows the two end runs (sink, recent tokens) hold most of the samples
    at or above the floor while their neighbours hold few: the block-skip instantiation takes the
    floor again from the interior runs, and most rows need no second counting pass."""
    case = workloads.peaky_decode_batch(requests=24)
    st = assert_blockskip_exact(gvr, case, "exact", seed=9)
    long_rows = case.row_lengths() > case.k
    assert ((st[long_rows, 2] % 10) == 2).sum() <= long_rows.sum() // 4, st


@pytest.mark.parametrize("variant", workloads.ADVERSARIAL_VARIANTS)
def test_blockskip_adversarial(gvr, variant):
    case = workloads.adversarial_row(variant)
    for kind in ("exact", "loose"):
        assert_blockskip_exact(gvr, case, kind, seed=4)


@pytest.mark.parametrize("flags", [1, 2, 4, 8, 16, 32, 2 | 4, 4 | 64, 128, 128 | 4, 128 | 32])
def test_blockskip_forced_paths_and_modes(gvr, flags):  # 128: the compact lists
    case = workloads.decode_batch(seed=6, requests=10, next_n=3, cr=4, k=512, stride=65536, boundary=True)
    assert_blockskip_exact(gvr, case, "exact", flags)


@pytest.mark.parametrize("bs,n,k", [(4, 131072, 512), (16, 65536, 2048), (1, 16384, 1024), (8, 100003, 1024)])
def test_blockskip_sweep_cells(gvr, bs, n, k):
    if n % 64:  # a window that ends inside a block and inside a vector
        case = workloads.sweep_decode(bs, 131072, k)
        case = workloads.DecodeCase("odd_n", case.logits, np.full(bs, n, np.int32), 1, 1, k)
        lg = case.logits
        for r in range(bs):
            lg[r, n:] = workloads.DECODE_POISON[np.arange(n, lg.shape[1]) % 3]
    else:
        case = workloads.sweep_decode(bs, n, k)
    assert_blockskip_exact(gvr, case, "exact")
    assert_blockskip_exact(gvr, case, "loose", seed=5)


def test_blockskip_rejects_bad_bounds(gvr):
    case = workloads.single_decode_row()
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    with pytest.raises(ValueError):
        gvr.topk_decode(lg, kv, 1, 1, case.k, block_max=torch.zeros((1, 3), dtype=torch.float32, device=DEV))
    with pytest.raises(ValueError):
        gvr.topk_decode(lg, kv, 1, 1, case.k, block_max=torch.zeros((1, 256), dtype=torch.float32, device=DEV),
                        pre_idx=torch.zeros((1, 512), dtype=torch.int32, device=DEV))
