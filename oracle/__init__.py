"""CPU oracle for the exact per-row top-K -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or executes it, and this
package never imports the product path: the two share no code.

The arithmetic lives in ``gvr_oracle.c`` (plain C, full sort per row); this
module only builds it with gcc and marshals numpy arrays through ctypes.

Each function states the passage of the pages it follows:

* decode rows -- "Block-skip fast path for self-sampling GVR top-K decode"
  (TensorRT-LLM PR #18122), commit "run_varlen": n = (kv_len - next_n +
  row % next_n + 1) / compress_ratio, request = row // next_n, kv_len < next_n
  is an empty row ("engine/reference convention alignment" commit);
* prefill rows -- "Self-sampling GVR V2 prefill indexer top-K" (PR #18702),
  section "Kernel": top-K of logits[r, ks:ke] in the local frame with a -1 pad,
  identity when nv <= k;
* exactness -- PR #18122 "Contract": exact (tie-interchangeable) top-K,
  signed zeros normalized; NaN inside a window is outside the contract, and
  the oracle refuses it (``OracleNaNError``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gvr_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgvr_oracle.so")
_lock = threading.Lock()
_lib = None

OK, BAD_ARG, NAN_IN_WINDOW, NO_MEMORY = 0, 1, 2, 3


class OracleNaNError(ValueError):
    """A NaN inside a selection window: outside the method's contract."""


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile ``src`` with gcc into a shared library at ``out`` and return its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build() -> str:
    """Build ``libgvr_oracle.so`` beside its source if missing or stale."""
    with _lock:
        if (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            compile_oracle()
    return _LIB_PATH


def _declare(lib):
    i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.oracle_topk_decode.argtypes = [p, i64, i64, p, i32, i32, i32, p, p, p, ctypes.c_int, p]
    lib.oracle_topk_decode.restype = ctypes.c_int
    lib.oracle_topk_prefill.argtypes = [p, i64, i64, p, p, i32, p, p, ctypes.c_int, p]
    lib.oracle_topk_prefill.restype = ctypes.c_int
    lib.oracle_topk_window.argtypes = [p, i64, i32, p, p, p]
    lib.oracle_topk_window.restype = ctypes.c_int
    lib.oracle_decode_row_len.argtypes = [i64, p, i32, i32, i64]
    lib.oracle_decode_row_len.restype = i64
    lib.oracle_thread_count.argtypes = [ctypes.c_int]
    lib.oracle_thread_count.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first when ``path`` is None)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, nan_row):
    if rc == NAN_IN_WINDOW:
        raise OracleNaNError(f"NaN inside the selection window of row {nan_row.value}")
    if rc != OK:
        raise ValueError(f"oracle rejected its arguments (code {rc})")


def decode_row_len(row: int, kv_lens, next_n: int, compress_ratio: int, row_stride: int, lib=None) -> int:
    """Valid length n of decode row ``row`` (the MTP window formula)."""
    lib = lib or load()
    kv = np.ascontiguousarray(kv_lens, dtype=np.int32)
    return int(lib.oracle_decode_row_len(row, _ptr(kv), next_n, compress_ratio, row_stride))


def topk_decode(logits, kv_lens, next_n: int, compress_ratio: int, k: int, *, want_values=False,
                nthreads: int = 0, lib=None):
    """Exact decode top-K.  Returns (indices [rows,k] int32, values or None, tau [rows] f32)."""
    lib = lib or load()
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    kv = np.ascontiguousarray(kv_lens, dtype=np.int32)
    rows, stride = logits.shape
    if kv.size * next_n < rows:
        raise ValueError("kv_lens needs ceil(rows / next_n) entries")
    idx = np.empty((rows, k), np.int32)
    vals = np.empty((rows, k), np.float32) if want_values else None
    tau = np.empty(rows, np.float32)
    bad = ctypes.c_int64(-1)
    rc = lib.oracle_topk_decode(_ptr(logits), stride, rows, _ptr(kv), next_n, compress_ratio, k,
                                _ptr(idx), _ptr(vals), _ptr(tau), nthreads, ctypes.byref(bad))
    _check(rc, bad)
    return idx, vals, tau


def topk_prefill(logits, row_starts, row_ends, k: int, *, nthreads: int = 0, lib=None):
    """Exact prefill top-K over per-row windows.  Returns (indices [rows,k] int32, tau [rows])."""
    lib = lib or load()
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    ks = np.ascontiguousarray(row_starts, dtype=np.int32)
    ke = np.ascontiguousarray(row_ends, dtype=np.int32)
    rows, stride = logits.shape
    if ks.size != rows or ke.size != rows:
        raise ValueError("row_starts / row_ends need one entry per row")
    idx = np.empty((rows, k), np.int32)
    tau = np.empty(rows, np.float32)
    bad = ctypes.c_int64(-1)
    rc = lib.oracle_topk_prefill(_ptr(logits), stride, rows, _ptr(ks), _ptr(ke), k, _ptr(idx), _ptr(tau),
                                 nthreads, ctypes.byref(bad))
    _check(rc, bad)
    return idx, tau


def topk_window(w, k: int, lib=None):
    """Exact top-K of one window (any k >= 1).  Returns (indices [k], values [k], tau)."""
    lib = lib or load()
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(k, np.int32)
    vals = np.empty(k, np.float32)
    tau = ctypes.c_float(0.0)
    rc = lib.oracle_topk_window(_ptr(w), w.size, k, _ptr(out), _ptr(vals), ctypes.byref(tau))
    if rc == NAN_IN_WINDOW:
        raise OracleNaNError("NaN inside the selection window")
    if rc != OK:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out, vals, np.float32(tau.value)


def thread_count(nthreads: int = 0, lib=None) -> int:
    """Threads the oracle's row loop uses for a request of ``nthreads`` (0 = all)."""
    lib = lib or load()
    return int(lib.oracle_thread_count(nthreads))
