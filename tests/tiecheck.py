"""Tie-aware comparison of a top-K result against the oracle's.

Several results are correct when values tie at the K-th largest value tau, so
the comparison checks what is unique and that the rest is valid ("Block-skip
fast path for self-sampling GVR top-K decode", PR #18122, "Contract": exact,
tie-interchangeable top-K with signed zeros normalized and poisoned pads never
selected; "GVR K=2048 reg_clus ..." PR #20998, setup of the performance
tables: every replay checks index range, unique indices and the exact selected
value multiset; short rows compare by exact equality, long rows by value
multiset).

For a row with window w (length nv):
* nv <= k: the result must equal [0, 1, ..., nv-1, -1, ..., -1] exactly;
* nv > k: (i) k entries, all in [0, nv), no duplicates;
  (ii) the set of selected indices with w' > tau equals the oracle's;
  (iii) the sorted multiset of w' over the selection equals the oracle's,
  bit for bit; w' is w with -0 mapped to +0;
  (iv) optional values equal w at the selected indices (zero sign ignored).
(i)-(iii) together force the remaining entries to be ties at tau.
"""
from __future__ import annotations

import numpy as np


def normalize_zero(w: np.ndarray) -> np.ndarray:
    w = np.asarray(w, dtype=np.float32).copy()
    w[w == 0] = np.float32(0.0)
    return w


def _bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def check_row(w: np.ndarray, k: int, got: np.ndarray, ref: np.ndarray, *, got_values=None) -> str | None:
    """Return None when ``got`` is a correct top-K of window ``w``, else a reason."""
    w = np.asarray(w, dtype=np.float32)
    got = np.asarray(got, dtype=np.int64)
    ref = np.asarray(ref, dtype=np.int64)
    nv = w.size
    if got.shape != (k,):
        return f"shape {got.shape} != ({k},)"
    if nv <= k:
        want = np.where(np.arange(k) < nv, np.arange(k), -1)
        if not np.array_equal(got, want):
            bad = np.nonzero(got != want)[0][:5]
            return f"short row (nv={nv}) identity mismatch at {bad.tolist()}: got {got[bad].tolist()}"
        if got_values is not None:
            gv = np.asarray(got_values, dtype=np.float32)
            wv = np.where(np.arange(k) < nv, np.concatenate([w, np.zeros(k, np.float32)])[:k],
                          np.float32(-np.finfo(np.float32).max)).astype(np.float32)
            if not np.array_equal(_bits(normalize_zero(gv)), _bits(normalize_zero(wv))):
                return "short row values mismatch"
        return None
    if got.min() < 0 or got.max() >= nv:
        return f"index out of window: min {got.min()} max {got.max()} nv {nv}"
    if np.unique(got).size != k:
        return "duplicate indices"
    wn = normalize_zero(w)
    tau = wn[ref].min()
    gset = set(got[wn[got] > tau].tolist())
    rset = set(ref[wn[ref] > tau].tolist())
    if gset != rset:
        return f"winners above tau differ: missing {sorted(rset - gset)[:5]} extra {sorted(gset - rset)[:5]}"
    if not np.array_equal(np.sort(_bits(wn[got])), np.sort(_bits(wn[ref]))):
        return "selected value multiset differs"
    if got_values is not None:
        gv = normalize_zero(np.asarray(got_values, dtype=np.float32))
        if not np.array_equal(_bits(gv), _bits(wn[got])):
            return "values differ from the window at the selected indices"
    return None


def decode_windows(logits: np.ndarray, kv_lens, next_n: int, cr: int):
    """Yield (row, window) for decode rows using the length formula of the oracle's inputs."""
    rows, stride = logits.shape
    kv_lens = np.asarray(kv_lens)
    for r in range(rows):
        kv = int(kv_lens[r // next_n])
        n = 0 if kv < next_n else min((kv - next_n + r % next_n + 1) // cr, stride)
        yield r, logits[r, :n]


def prefill_windows(logits: np.ndarray, ks, ke):
    rows, stride = logits.shape
    for r in range(rows):
        a = max(int(ks[r]), 0)
        b = min(int(ke[r]), stride)
        yield r, logits[r, a:max(a, b)]


def compare_rows(windows, k: int, got: np.ndarray, ref: np.ndarray, got_values=None, max_report: int = 5):
    """Compare every row; return (n_inexact, reasons[:max_report])."""
    bad, reasons = 0, []
    for r, w in windows:
        why = check_row(w, k, got[r], ref[r], got_values=None if got_values is None else got_values[r])
        if why is not None:
            bad += 1
            if len(reasons) < max_report:
                reasons.append(f"row {r}: {why}")
    return bad, reasons
