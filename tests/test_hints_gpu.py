"""Hinted sampling (topk_decode_hinted) against the oracle: exact whatever the hints hold.

The hints are a request's previous-step selection, shared by its next_n rows ("Block-skip
fast path for self-sampling GVR top-K decode", request-level pre_idx taken as-is).  They only
choose sample positions, so every hint pattern must give the exact selection: the current
step's own top-K, a drifted previous step, all zero, all the same, all at INT32_MAX, half
duplicated, -1 padded (a short previous row), negative and out-of-window garbage.
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


HINTS = ["current", "previous", "zero", "same", "int_max", "half_dup", "neg_pad", "garbage"]


def make_hints(case, kind, seed):
    """int32 [requests, k + 3] hint rows (3 spare columns exercise the stride)."""
    g = np.random.default_rng(seed)
    k = case.k
    reqs = len(case.kv_lens)
    h = np.zeros((reqs, k + 3), np.int32)
    n = case.row_lengths()
    if kind in ("current", "previous", "half_dup", "neg_pad"):
        lg = case.logits
        if kind == "previous":  # last step: the same rows drifted a little, one token shorter
            lg = lg + 0.3 * g.standard_normal(lg.shape).astype(np.float32)
        kv_prev = case.kv_lens - (1 if kind == "previous" else 0)
        ref, _, _ = oracle.topk_decode(lg, np.maximum(kv_prev, 0).astype(np.int32), case.next_n,
                                       case.compress_ratio, k)
        h[:, :k] = ref[::case.next_n]  # the request's first row
        if kind == "half_dup":
            h[:, k // 2:k] = h[:, :k - k // 2]
        if kind == "neg_pad":
            h[:, k // 3:k] = -1
    elif kind == "same":
        h[:] = 5
    elif kind == "int_max":
        h[:] = np.iinfo(np.int32).max
    elif kind == "garbage":
        h[:] = g.integers(-(1 << 31), (1 << 31) - 1, h.shape, dtype=np.int64).astype(np.int32)
        h[:, ::4] = g.integers(0, max(int(n.max()), 1), (reqs, (k + 3 + 3) // 4))
    return h


def run_hinted(gvr, case, hints, flags=0, stats=False):
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    pre = torch.from_numpy(hints).to(DEV)
    opts = gvr.Options(flags=flags)
    st = None
    if stats:
        st = torch.full((case.rows, 4), -7, dtype=torch.int32, device=DEV)
        opts.row_stats = st.data_ptr()
    idx, vals = gvr.topk_decode(lg, kv, case.next_n, case.compress_ratio, case.k, want_values=True,
                                options=opts, pre_idx=pre)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), vals.cpu().numpy(), (st.cpu().numpy() if st is not None else None)


def assert_hinted_exact(gvr, case, kind, flags=0, seed=0):
    hints = make_hints(case, kind, seed)
    got, vals, st = run_hinted(gvr, case, hints, flags, stats=True)
    ref, _, _ = oracle.topk_decode(case.logits, case.kv_lens, case.next_n, case.compress_ratio, case.k)
    bad, why = compare_rows(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio), case.k,
                            got, ref, got_values=vals)
    assert bad == 0, f"{case.name}/{kind}: {bad} inexact rows: {why}"
    if flags & 32:
        assert np.array_equal(got, ref)
    return st


@pytest.mark.parametrize("kind", HINTS)
def test_hinted_decode_batch(gvr, kind):
    st = assert_hinted_exact(gvr, workloads.decode_batch(), kind, seed=11)
    if kind in ("current", "previous"):
        n = workloads.decode_batch().row_lengths()
        assert np.isin(st[n > 1024, 0], (1, 5)).all(), st[:, 0]  # good hints: no rescue


@pytest.mark.parametrize("kind", HINTS)
def test_hinted_single_and_adversarial(gvr, kind):
    assert_hinted_exact(gvr, workloads.single_decode_row(), kind, seed=12)
    for variant in ("base", "all_equal", "two_valued", "neg_inf_tau", "signed_zero_tau", "pos_inf_class"):
        assert_hinted_exact(gvr, workloads.adversarial_row(variant), kind, seed=13)


@pytest.mark.parametrize("kind", ["previous", "zero", "neg_pad"])
@pytest.mark.parametrize("flags", [16, 32, 1, 4, 128, 128 | 32])
def test_hinted_modes_and_forced_paths(gvr, kind, flags):  # 128: the compact lists
    case = workloads.decode_batch(seed=5, requests=12, next_n=3, cr=4, k=512, stride=65536, boundary=True)
    assert_hinted_exact(gvr, case, kind, flags, seed=14)


def test_hinted_rejects_bad_buffers(gvr):
    case = workloads.single_decode_row()
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    with pytest.raises(ValueError):
        gvr.topk_decode(lg, kv, 1, 1, case.k, pre_idx=torch.zeros((1, case.k - 1), dtype=torch.int32, device=DEV))
    with pytest.raises(ValueError):
        gvr.topk_decode(lg, kv, 1, 1, case.k, pre_idx=torch.zeros((1, case.k), dtype=torch.int64, device=DEV))
