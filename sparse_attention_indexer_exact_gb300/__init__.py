"""Exact per-row top-K for a DSA sparse-attention indexer on one GB300 (sm_103a).

A thin Python binding over the C ABI of ``libgvrtopk.so`` (declared in
``include/gvr_topk.h``).  Every step of the selection runs in the library's
CUDA kernel; this module only checks tensor types, takes device pointers and
the current CUDA stream, and forwards them.  PyTorch is used for device
memory and streams only.  There is no CPU fallback: if the library has not
been built (``python -m sparse_attention_indexer_exact_gb300._build`` or
``__graft_entry__.build()``), every call raises.

Entry points (same names as the C ABI):

* ``topk_decode(logits, kv_lens, next_n, compress_ratio, k, ...)`` -- decode
  rows, n = (kv_len - next_n + row % next_n + 1) // compress_ratio valid
  scores per row ("Block-skip fast path for self-sampling GVR top-K decode",
  TensorRT-LLM PR #18122, commit "run_varlen");
* ``topk_prefill(logits, row_starts, row_ends, k, ...)`` -- per-row windows
  [row_starts, row_ends) written in the local frame with a -1 pad
  ("Self-sampling GVR V2 prefill indexer top-K", PR #18702, "Kernel").
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["topk_decode", "topk_prefill", "topk_decode_raw", "topk_decode_hinted_raw", "topk_decode_blockskip_raw",
           "topk_prefill_raw", "topk_decode_ws_raw", "topk_prefill_ws_raw", "topk_decode_noalloc_raw",
           "workspace_size", "workspace", "plan",
           "Options",
           "GvrError", "library_path", "load_library", "FLAG_FORCE_RESCUE", "FLAG_NO_FLOOR", "FLAG_ZERO_CAP",
           "FLAG_RADIX_REFINE", "FLAG_DETERMINISTIC", "FLAG_SORTED", "FLAG_STREAM_RESCUE", "FLAG_COMPACT_LISTS",
           "FLAG_CLUSTER_KERNEL", "FLAG_SPLIT_ALONE", "FLAG_SPLIT_KERNEL", "FLAG_DIAG_FAIL_ROW0", "FLAG_SHORT_KERNEL",
           "FLAG_BLOCKSKIP_ALWAYS", "PATH_NAMES", "SUPPORTED_K"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libgvrtopk.so")
_lock = threading.Lock()
_lib = None

FLAG_FORCE_RESCUE, FLAG_NO_FLOOR, FLAG_ZERO_CAP, FLAG_RADIX_REFINE = 1, 2, 4, 8
FLAG_DETERMINISTIC, FLAG_SORTED, FLAG_STREAM_RESCUE, FLAG_COMPACT_LISTS = 16, 32, 64, 128
FLAG_CLUSTER_KERNEL, FLAG_SPLIT_ALONE, FLAG_SPLIT_KERNEL, FLAG_DIAG_FAIL_ROW0, FLAG_SHORT_KERNEL = 256, 512, 1024, 2048, 4096
FLAG_BLOCKSKIP_ALWAYS = 8192
PATH_NAMES = {-1: "device_error", 0: "short", 1: "refine", 2: "rescue_bracket", 3: "rescue_overflow",
              4: "rescue_forced", 5: "refine_cluster", 6: "refine_relist", 7: "split", 8: "split_alone",
              9: "neg_inf_fill", 10: "short_kernel", 11: "short_radix"}
SUPPORTED_K = (512, 1024, 2048)
EXPORTED_SYMBOLS = ("topk_decode", "topk_prefill", "topk_decode_ex", "topk_prefill_ex", "topk_decode_hinted",
                    "topk_decode_blockskip", "topk_decode_ws", "topk_prefill_ws", "gvr_workspace_size",
                    "topk_decode_noalloc", "gvr_status_string", "gvr_plan")


class GvrError(RuntimeError):
    """A non-zero gvr_status returned by the library."""

    def __init__(self, status: int, message: str):
        super().__init__(f"gvr status {status}: {message}")
        self.status = status


class Options(ctypes.Structure):
    """Mirror of ``gvr_options`` (tuning and diagnostics of the *_ex entry points)."""
    _fields_ = [("cluster_size", ctypes.c_int32), ("ring_stages", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("row_stats", ctypes.c_void_p)]


def library_path() -> str:
    return _LIB_PATH


def _declare(lib):
    i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.topk_decode.argtypes = [p, i64, i64, p, i32, i32, i32, p, p, p]
    lib.topk_decode_ex.argtypes = [p, i64, i64, p, i32, i32, i32, p, p, p, ctypes.POINTER(Options)]
    lib.topk_decode_hinted.argtypes = [p, i64, i64, p, i32, i32, i32, p, i64, p, p, p, ctypes.POINTER(Options)]
    lib.topk_decode_blockskip.argtypes = [p, i64, i64, p, i32, i32, i32, p, i64, p, p, p, ctypes.POINTER(Options)]
    lib.topk_prefill.argtypes = [p, i64, i64, p, p, i32, p, p]
    lib.topk_prefill_ex.argtypes = [p, i64, i64, p, p, i32, p, p, ctypes.POINTER(Options)]
    lib.gvr_plan.argtypes = [i64, i64, i32, ctypes.POINTER(Options), i32] + [ctypes.POINTER(i32)] * 4
    sz = ctypes.c_size_t
    lib.topk_decode_ws.argtypes = [p, i64, i64, p, i32, i32, i32, p, p, p, sz, p, ctypes.POINTER(Options)]
    lib.topk_prefill_ws.argtypes = [p, i64, i64, p, p, i32, p, p, sz, p, ctypes.POINTER(Options)]
    lib.gvr_workspace_size.argtypes = [i32, ctypes.POINTER(sz)]
    lib.topk_decode_noalloc.argtypes = [p, i64, i64, p, i32, i32, i32, p, p, p]
    for f in (lib.topk_decode, lib.topk_decode_ex, lib.topk_decode_hinted, lib.topk_decode_blockskip,
              lib.topk_prefill, lib.topk_prefill_ex, lib.gvr_plan, lib.topk_decode_ws, lib.topk_prefill_ws,
              lib.gvr_workspace_size, lib.topk_decode_noalloc):
        f.restype = ctypes.c_int
    lib.gvr_status_string.argtypes = [ctypes.c_int]
    lib.gvr_status_string.restype = ctypes.c_char_p
    return lib


def load_library(path: str | None = None):
    """Load libgvrtopk.so; raises if it has not been built."""
    global _lib
    with _lock:
        if path is not None:
            return _declare(ctypes.CDLL(path))
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                                   "`python -m sparse_attention_indexer_exact_gb300._build` (no CPU fallback exists)")
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
        return _lib


def _check(status: int):
    if status != 0:
        lib = load_library()
        raise GvrError(status, lib.gvr_status_string(status).decode())


# ----------------------------------------------------------------------------- raw pointers
def topk_decode_raw(logits_ptr: int, row_stride: int, num_rows: int, kv_lens_ptr: int, next_n: int,
                    compress_ratio: int, k: int, indices_ptr: int, values_ptr: int | None, stream: int,
                    options: Options | None = None) -> None:
    """``topk_decode`` / ``topk_decode_ex`` on raw device addresses (enqueue only)."""
    lib = load_library()
    if options is None:
        st = lib.topk_decode(logits_ptr, row_stride, num_rows, kv_lens_ptr, next_n, compress_ratio, k,
                             indices_ptr, values_ptr, stream)
    else:
        st = lib.topk_decode_ex(logits_ptr, row_stride, num_rows, kv_lens_ptr, next_n, compress_ratio, k,
                                indices_ptr, values_ptr, stream, ctypes.byref(options))
    _check(st)


def topk_decode_hinted_raw(logits_ptr: int, row_stride: int, num_rows: int, kv_lens_ptr: int, next_n: int,
                           compress_ratio: int, k: int, pre_idx_ptr: int, pre_idx_stride: int, indices_ptr: int,
                           values_ptr: int | None, stream: int, options: Options | None = None) -> None:
    """``topk_decode_hinted`` on raw device addresses (enqueue only)."""
    lib = load_library()
    st = lib.topk_decode_hinted(logits_ptr, row_stride, num_rows, kv_lens_ptr, next_n, compress_ratio, k,
                                pre_idx_ptr, pre_idx_stride, indices_ptr, values_ptr, stream,
                                ctypes.byref(options) if options is not None else None)
    _check(st)


def topk_decode_blockskip_raw(logits_ptr: int, row_stride: int, num_rows: int, kv_lens_ptr: int, next_n: int,
                              compress_ratio: int, k: int, block_max_ptr: int, block_max_stride: int,
                              indices_ptr: int, values_ptr: int | None, stream: int,
                              options: Options | None = None) -> None:
    """``topk_decode_blockskip`` on raw device addresses (enqueue only)."""
    lib = load_library()
    st = lib.topk_decode_blockskip(logits_ptr, row_stride, num_rows, kv_lens_ptr, next_n, compress_ratio, k,
                                   block_max_ptr, block_max_stride, indices_ptr, values_ptr, stream,
                                   ctypes.byref(options) if options is not None else None)
    _check(st)


def topk_prefill_raw(logits_ptr: int, row_stride: int, num_rows: int, row_starts_ptr: int, row_ends_ptr: int,
                     k: int, indices_ptr: int, stream: int, options: Options | None = None) -> None:
    """``topk_prefill`` / ``topk_prefill_ex`` on raw device addresses (enqueue only)."""
    lib = load_library()
    if options is None:
        st = lib.topk_prefill(logits_ptr, row_stride, num_rows, row_starts_ptr, row_ends_ptr, k, indices_ptr,
                              stream)
    else:
        st = lib.topk_prefill_ex(logits_ptr, row_stride, num_rows, row_starts_ptr, row_ends_ptr, k, indices_ptr,
                                 stream, ctypes.byref(options))
    _check(st)


def topk_decode_ws_raw(logits_ptr: int, row_stride: int, num_rows: int, kv_lens_ptr: int, next_n: int,
                       compress_ratio: int, k: int, indices_ptr: int, values_ptr: int | None, workspace_ptr: int,
                       workspace_bytes: int, stream: int, options: Options | None = None) -> None:
    """``topk_decode_ws`` on raw device addresses (enqueue only)."""
    lib = load_library()
    st = lib.topk_decode_ws(logits_ptr, row_stride, num_rows, kv_lens_ptr, next_n, compress_ratio, k, indices_ptr,
                            values_ptr, workspace_ptr, workspace_bytes, stream,
                            ctypes.byref(options) if options is not None else None)
    _check(st)


def topk_prefill_ws_raw(logits_ptr: int, row_stride: int, num_rows: int, row_starts_ptr: int, row_ends_ptr: int,
                        k: int, indices_ptr: int, workspace_ptr: int, workspace_bytes: int, stream: int,
                        options: Options | None = None) -> None:
    """``topk_prefill_ws`` on raw device addresses (enqueue only)."""
    lib = load_library()
    st = lib.topk_prefill_ws(logits_ptr, row_stride, num_rows, row_starts_ptr, row_ends_ptr, k, indices_ptr,
                             workspace_ptr, workspace_bytes, stream,
                             ctypes.byref(options) if options is not None else None)
    _check(st)


def topk_decode_noalloc_raw(logits_ptr: int, row_stride: int, num_rows: int, kv_lens_ptr: int, next_n: int,
                            compress_ratio: int, k: int, indices_ptr: int, values_ptr: int | None,
                            stream: int) -> None:
    """``topk_decode_noalloc`` on raw device addresses: the library's own fixed scratch, no
    allocation and no workspace (at most 128 rows; calls that overlap on the GPU race)."""
    lib = load_library()
    _check(lib.topk_decode_noalloc(logits_ptr, row_stride, num_rows, kv_lens_ptr, next_n, compress_ratio, k,
                                   indices_ptr, values_ptr, stream))


def workspace_size(sm_count: int = 0) -> int:
    """Bytes of workspace the *_ws entry points need (current device, or a device of sm_count SMs)."""
    lib = load_library()
    out = ctypes.c_size_t(0)
    _check(lib.gvr_workspace_size(sm_count, ctypes.byref(out)))
    return int(out.value)


_workspaces: dict = {}


def workspace(device, stream_handle: int):
    """The zero-filled workspace this binding keeps per (device, stream): calls on one stream are
    ordered, so they may share it; calls on different streams get different ones.  It is
    allocated (torch.zeros) on the first call for that pair, so make that call before capturing
    a CUDA graph that replays it."""
    torch = _torch()
    key = (device.index, int(stream_handle))
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.zeros(workspace_size(), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def plan(row_stride: int, num_rows: int, k: int, options: Options | None = None, sm_count: int = 0) -> dict:
    """Launch geometry the library would choose (host only)."""
    lib = load_library()
    outs = [ctypes.c_int32(0) for _ in range(4)]
    st = lib.gvr_plan(row_stride, num_rows, k, ctypes.byref(options) if options is not None else None, sm_count,
                      *[ctypes.byref(o) for o in outs])
    _check(st)
    cs, stages, threads, smem = (o.value for o in outs)
    return {"cluster_size": cs, "ring_stages": stages, "threads": threads, "smem_bytes": smem}


# ----------------------------------------------------------------------------- torch tensors
def _torch():
    import torch
    return torch


def _stream_handle(stream, device) -> int:
    """The CUDA stream handle to launch on: ``stream`` if given, else the current stream of
    ``device`` (the tensors' device, not whichever device happens to be current)."""
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _same_device(device, **tensors):
    """Every given tensor must live on ``device``: the library launches on one device with
    pointers that must all belong to it."""
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, logits on {device}: all tensors must share one device")


def _rows_2d(logits):
    """(rows, row stride) of a 2-D fp32 CUDA tensor.  The row stride passed to the library is the
    row length: windows are clamped to it, so a narrowed view (stride(0) > shape[1]) is refused
    rather than read past its columns."""
    torch = _torch()
    if not isinstance(logits, torch.Tensor) or not logits.is_cuda:
        raise TypeError("logits must be a CUDA tensor")
    if logits.dtype != torch.float32:
        raise TypeError("logits must be float32")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit inner stride")
    if logits.shape[0] > 1 and logits.stride(0) != logits.shape[1]:
        raise ValueError("logits rows must be packed (stride(0) == shape[1]); pass .contiguous() for a "
                         "narrowed view")
    return logits.shape[0], logits.shape[1]


def _int32_vec(t, n, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.int32:
        raise TypeError(f"{name} must be a CUDA int32 tensor")
    if t.dim() != 1 or t.stride(0) != 1 or t.numel() < n:
        raise ValueError(f"{name} must be 1-D contiguous with at least {n} entries")


def _out(t, rows, k, dtype, device, name):
    torch = _torch()
    if t is None:
        return torch.empty((rows, k), dtype=dtype, device=device)
    if t.dtype != dtype or not t.is_cuda or t.shape != (rows, k) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor of shape ({rows}, {k})")
    return t


def topk_decode(logits, kv_lens, next_n: int, compress_ratio: int, k: int, indices=None, values=None, *,
                want_values: bool = False, stream=None, options: Options | None = None, pre_idx=None,
                block_max=None):
    """Decode top-K of each row of ``logits`` [rows, >=n]; returns (indices, values or None).

    ``logits.stride(0)`` is the row stride.  ``kv_lens`` is int32 [ceil(rows / next_n)].
    ``pre_idx`` (optional) is int32 [ceil(rows / next_n), >= k] with unit inner stride: each
    request's previous selection, used only as sample positions (``topk_decode_hinted``).
    ``block_max`` (optional) is fp32 [rows, >= ceil(row_stride / 32)] with unit inner stride: an
    upper bound of every 32-score block of each row's window (``topk_decode_blockskip``).
    """
    rows, stride = _rows_2d(logits)
    _int32_vec(kv_lens, (rows + next_n - 1) // max(next_n, 1), "kv_lens")
    _same_device(logits.device, kv_lens=kv_lens, indices=indices, values=values, pre_idx=pre_idx,
                 block_max=block_max)
    with _torch().cuda.device(logits.device):
        return _topk_decode_on_device(logits, rows, stride, kv_lens, next_n, compress_ratio, k, indices, values,
                                      want_values, stream, options, pre_idx, block_max)


def _topk_decode_on_device(logits, rows, stride, kv_lens, next_n, compress_ratio, k, indices, values, want_values,
                           stream, options, pre_idx, block_max):
    indices = _out(indices, rows, k, _torch().int32, logits.device, "indices")
    if values is None and want_values:
        values = _out(None, rows, k, _torch().float32, logits.device, "values")
    elif values is not None:
        values = _out(values, rows, k, _torch().float32, logits.device, "values")
    vptr = values.data_ptr() if values is not None else None
    if pre_idx is not None and block_max is not None:
        raise ValueError("pre_idx and block_max select different entry points; pass one of them")
    if block_max is not None:
        torch = _torch()
        if (block_max.dtype != torch.float32 or not block_max.is_cuda or block_max.dim() != 2
                or block_max.shape[0] != rows or block_max.shape[1] < (stride + 31) // 32 or block_max.stride(1) != 1):
            raise ValueError(f"block_max must be a CUDA fp32 tensor [{rows}, >= {(stride + 31) // 32}] "
                             "with unit inner stride")
        topk_decode_blockskip_raw(logits.data_ptr(), stride, rows, kv_lens.data_ptr(), next_n, compress_ratio, k,
                                  block_max.data_ptr(), block_max.stride(0), indices.data_ptr(), vptr,
                                  _stream_handle(stream, logits.device), options)
    elif pre_idx is not None:
        torch = _torch()
        reqs = (rows + next_n - 1) // max(next_n, 1)
        if (pre_idx.dtype != torch.int32 or not pre_idx.is_cuda or pre_idx.dim() != 2 or pre_idx.shape[0] != reqs
                or pre_idx.shape[1] < k or pre_idx.stride(1) != 1):
            raise ValueError(f"pre_idx must be a CUDA int32 tensor [{reqs}, >= {k}] with unit inner stride")
        topk_decode_hinted_raw(logits.data_ptr(), stride, rows, kv_lens.data_ptr(), next_n, compress_ratio, k,
                               pre_idx.data_ptr(), pre_idx.stride(0), indices.data_ptr(), vptr,
                               _stream_handle(stream, logits.device), options)
    else:
        h = _stream_handle(stream, logits.device)
        ws = workspace(logits.device, h)
        topk_decode_ws_raw(logits.data_ptr(), stride, rows, kv_lens.data_ptr(), next_n, compress_ratio, k,
                           indices.data_ptr(), vptr, ws.data_ptr(), ws.numel(), h, options)
    return indices, values


def topk_prefill(logits, row_starts, row_ends, k: int, indices=None, *, stream=None,
                 options: Options | None = None):
    """Prefill top-K over per-row windows [row_starts, row_ends); returns local indices [rows, k]."""
    rows, stride = _rows_2d(logits)
    _int32_vec(row_starts, rows, "row_starts")
    _int32_vec(row_ends, rows, "row_ends")
    _same_device(logits.device, row_starts=row_starts, row_ends=row_ends, indices=indices)
    with _torch().cuda.device(logits.device):
        indices = _out(indices, rows, k, _torch().int32, logits.device, "indices")
        h = _stream_handle(stream, logits.device)
        ws = workspace(logits.device, h)
        topk_prefill_ws_raw(logits.data_ptr(), stride, rows, row_starts.data_ptr(), row_ends.data_ptr(), k,
                            indices.data_ptr(), ws.data_ptr(), ws.numel(), h, options)
    return indices
