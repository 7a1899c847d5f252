"""The entry point that allocates nothing: topk_decode_noalloc.

Some callers cannot allocate device memory at the moment they select -- an inference engine's
plugin that is only handed its inputs and outputs at enqueue time, a serving loop that lives on
a fixed arena owned by another allocator, latency-critical code that cannot risk the device-wide
synchronization a cudaMalloc may bring.  For them the library keeps its own fixed scratch array
(no workspace argument) and runs its balanced kernel on it.

This test calls that entry point through the C ABI twice in a row on the full decode batch (128
rows, its limit) and checks each result against the plain topk_decode's on the same input,
tie-aware as every parity test here (the same winners above tau, the same selected value
multiset bit for bit, valid distinct indices, values equal to the scores at the returned
indices), and that a call over the row limit is refused before anything is enqueued.  It lives
in a file of its own that pytest collects last, so a run that stops at the first failure has
already run every other test; it passes alone in a fresh process as well as after them.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import workloads
from tiecheck import compare_rows, decode_windows

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GVR_ERR_NOALLOC_LIMIT = 8


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_indexer_exact_gb300 import _build
    _build.build_library()
    import sparse_attention_indexer_exact_gb300 as gvr
    torch.cuda.set_device(0)
    return gvr.load_library()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_matches_topk_decode_on_two_calls_in_a_row(lib):
    case = workloads.decode_batch()  # 128 rows: the entry point's row limit
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (case.row_stride, case.rows, _ptr(kv), case.next_n, case.compress_ratio, case.k)

    ref_idx = torch.empty((case.rows, case.k), dtype=torch.int32, device=DEV)
    ref_val = torch.empty((case.rows, case.k), dtype=torch.float32, device=DEV)
    assert lib.topk_decode(_ptr(lg), *args, _ptr(ref_idx), _ptr(ref_val), h) == 0
    torch.cuda.synchronize()
    ref = ref_idx.cpu().numpy()

    for call in range(2):
        idx = torch.full((case.rows, case.k), -9, dtype=torch.int32, device=DEV)
        val = torch.empty((case.rows, case.k), dtype=torch.float32, device=DEV)
        assert lib.topk_decode_noalloc(_ptr(lg), *args, _ptr(idx), _ptr(val), h) == 0
        torch.cuda.synchronize()
        bad, why = compare_rows(decode_windows(case.logits, case.kv_lens, case.next_n, case.compress_ratio), case.k,
                                idx.cpu().numpy(), ref, got_values=val.cpu().numpy())
        assert bad == 0, f"call {call}: {bad} rows differ from topk_decode: {why}"


def test_noalloc_refuses_more_rows_than_its_scratch_holds(lib):
    case = workloads.decode_batch(seed=9, requests=65, stride=8192, kv_lo=1, kv_hi=32768, boundary=False)
    assert case.rows == 130
    lg = torch.from_numpy(case.logits).to(DEV)
    kv = torch.from_numpy(case.kv_lens).to(DEV)
    idx = torch.full((case.rows, case.k), -9, dtype=torch.int32, device=DEV)
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.topk_decode_noalloc(_ptr(lg), case.row_stride, case.rows, _ptr(kv), case.next_n, case.compress_ratio,
                                 case.k, _ptr(idx), None, h)
    assert st == GVR_ERR_NOALLOC_LIMIT
    assert b"128" in lib.gvr_status_string(st)
    torch.cuda.synchronize()
    assert int((idx != -9).sum().item()) == 0, "a refused call must enqueue nothing"
