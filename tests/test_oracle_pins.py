"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

The oracle must be trusted before any GPU result is compared with it, so it is
pinned here to things other than itself:

* golden files written by hand from the pages' rules (tests/golden/);
* brute force over every K-subset of tiny windows (a valid top-K set S has
  min over S >= max over the rest; the number of valid sets is C(t, K - g)
  with g values above tau and t values equal to it);
* the invariant count(> tau) < K <= count(>= tau) on every selected row;
* numpy's partition, an independent selection routine, on random rows;
* closed forms: all-equal, two-valued, -inf and +inf tie classes, signed
  zero, the short-row identity with its -1 / -FLT_MAX pad;
* translation invariance of prefill windows with a misaligned start.

Each pin is a function of the loaded oracle library so that
``test_pins_catch_planted_mistakes`` can run the same pins on deliberately
broken copies of the oracle (mistakes planted on the CPU) and show that every
plausible slip is caught by at least one pin.
"""
from __future__ import annotations

import itertools
import math
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FLT_MAX = np.float32(np.finfo(np.float32).max)


def _nz(w):
    w = np.asarray(w, np.float32).copy()
    w[w == 0] = 0.0
    return w


# ----------------------------------------------------------------------------- pins
def pin_golden_decode_row_len(lib):
    for line in open(os.path.join(GOLDEN, "decode_row_len.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        kv, next_n, cr, row, stride, n = (int(x) for x in line.split())
        kv_lens = np.full(row // next_n + 1, kv, np.int32)
        got = oracle.decode_row_len(row, kv_lens, next_n, cr, stride, lib=lib)
        assert got == n, f"kv={kv} next_n={next_n} cr={cr} row={row}: n={got}, expected {n}"
        # the batched entry must use the same rows: row r of a batch selects over its first n scores
        logits = np.arange(stride, dtype=np.float32)[None, :].repeat(row + 1, 0)
        idx, _, _ = oracle.topk_decode(logits[:, :stride], kv_lens, next_n, cr, 1, lib=lib)
        want = -1 if n == 0 else n - 1  # ascending scores: the largest valid one is the last
        assert idx[row, 0] == want, f"decode row {row}: top-1 {idx[row, 0]} expected {want}"


def _parse_golden_topk():
    for line in open(os.path.join(GOLDEN, "tiny_topk.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        vals, win, k, exp, tau = (p.strip() for p in line.split("|"))
        row = np.array([float(x) for x in vals.split()], np.float32)
        ks, ke = (int(x) for x in win.split())
        yield row, ks, ke, int(k), [int(x) for x in exp.split()], float(tau)


GOLDEN_POISON = 100.0  # larger than every golden score: selected whenever a window leaks onto it


def pin_golden_tiny_topk(lib):
    for row, ks, ke, k, exp, tau in _parse_golden_topk():
        stride = ((row.size + 3) // 4) * 4
        # The golden row sits between two poison rows on each side, with NaN padding after its
        # values: a window that ignores the row's bounds (a dropped clamp) reads poison or NaN in
        # the same allocation and its result changes, instead of reading outside the buffer.
        assert -2 * stride <= ks and ke <= 3 * stride, "golden windows stay within the poison rows"
        logits = np.full((5, stride), GOLDEN_POISON, np.float32)
        logits[2, :] = np.nan
        logits[2, :row.size] = row
        starts = np.array([0, 0, ks, 0, 0], np.int32)
        ends = np.array([0, 0, ke, 0, 0], np.int32)
        idx, t = oracle.topk_prefill(logits, starts, ends, k, lib=lib)
        assert idx[2].tolist() == exp, f"{row.tolist()} [{ks},{ke}) k={k}: {idx[2].tolist()} != {exp}"
        if math.isnan(tau):
            assert math.isnan(t[2])
        else:
            assert t[2] == np.float32(tau) and not (t[2] == 0 and np.signbit(t[2])), (t[2], tau)


def _tiny_rows(seed=7, count=160):
    g = np.random.default_rng(seed)
    alphabet = np.array([-np.inf, -2.0, -1.0, -0.0, 0.0, 1.0, 1.5, 2.0, np.inf], np.float32)
    for _ in range(count):
        nv = int(g.integers(1, 13))
        yield alphabet[g.integers(0, alphabet.size, nv)]


def pin_brute_force_tiny(lib):
    for w in _tiny_rows():
        nv = w.size
        wn = _nz(w)
        for k in range(1, nv + 1):
            idx, vals, tau = oracle.topk_window(w, k, lib=lib)
            if nv <= k:
                assert idx.tolist() == list(range(nv)) + [-1] * (k - nv)
                continue
            valid = []
            for s in itertools.combinations(range(nv), k):
                rest = [j for j in range(nv) if j not in s]
                if min(wn[list(s)]) >= max(wn[rest]):
                    valid.append(frozenset(s))
            sel = frozenset(idx.tolist())
            assert len(sel) == k and sel in valid, f"{w.tolist()} k={k}: {sorted(sel)} not a valid top-K"
            true_tau = max(min(wn[list(s)]) for s in valid)
            assert tau == true_tau, (tau, true_tau)
            g = int((wn > tau).sum())
            t = int((wn == tau).sum())
            assert len(valid) == math.comb(t, k - g)
            # the documented order: value descending, then window index ascending
            keyed = [(-float(wn[j]), int(j)) for j in idx]
            assert keyed == sorted(keyed), f"order {idx.tolist()} for {w.tolist()}"
            assert np.array_equal(vals.view(np.uint32), w[idx].view(np.uint32))


def pin_invariant_random(lib):
    g = np.random.default_rng(11)
    for trial in range(60):
        nv = int(g.integers(2, 3000))
        k = int(g.integers(1, nv))
        kind = trial % 3
        if kind == 0:
            w = g.standard_normal(nv).astype(np.float32)
        elif kind == 1:
            w = g.integers(-3, 4, nv).astype(np.float32)
        else:
            w = np.round(g.standard_normal(nv) * 4).astype(np.float32) / 4
            w[g.random(nv) < 0.2] = -np.inf
        wn = _nz(w)
        idx, _, tau = oracle.topk_window(w, k, lib=lib)
        assert (wn > tau).sum() < k <= (wn >= tau).sum(), (trial, tau)
        assert np.unique(idx).size == k and idx.min() >= 0 and idx.max() < nv
        assert wn[idx].min() == tau


def pin_partition_crosscheck(lib):
    g = np.random.default_rng(13)
    for trial in range(40):
        nv = int(g.integers(100, 20000))
        k = int(g.integers(1, min(nv, 2048)))
        w = (g.standard_normal(nv) * (1 + trial)).astype(np.float32)
        if trial % 4 == 0:
            w = np.round(w).astype(np.float32)
        idx, _, _ = oracle.topk_window(w, k, lib=lib)
        want = np.sort(-np.partition(-_nz(w).astype(np.float64), k - 1)[:k])
        assert np.array_equal(np.sort(_nz(w)[idx].astype(np.float64)), want)


def pin_closed_forms(lib):
    k = 512
    # all-equal row: tau = c and the first k indices (smallest-index ties)
    w = np.full(5000, 1.25, np.float32)
    idx, _, tau = oracle.topk_window(w, k, lib=lib)
    assert tau == np.float32(1.25) and idx.tolist() == list(range(k))
    # two-valued rows: tau = the high value when it has >= k members, else the low value
    g = np.random.default_rng(3)
    for hi_count in (k - 1, k, k + 1, 3000):
        w = np.full(6000, 1.0, np.float32)
        w[g.choice(6000, hi_count, replace=False)] = 2.0
        idx, _, tau = oracle.topk_window(w, k, lib=lib)
        assert tau == (2.0 if hi_count >= k else 1.0)
        assert int((w[idx] == 2.0).sum()) == min(hi_count, k)
    # more than nv - k entries at -inf: tau = -inf and every finite entry is selected
    w = g.standard_normal(4000).astype(np.float32)
    neg = g.choice(4000, 4000 - k + 50, replace=False)
    w[neg] = -np.inf
    idx, _, tau = oracle.topk_window(w, k, lib=lib)
    assert tau == -np.inf
    assert set(np.nonzero(np.isfinite(w))[0].tolist()) <= set(idx.tolist())
    # a +inf class of k-3 members is always selected; tau is the 3rd largest finite value
    w = g.standard_normal(4000).astype(np.float32)
    pos = g.choice(4000, k - 3, replace=False)
    w[pos] = np.inf
    idx, _, tau = oracle.topk_window(w, k, lib=lib)
    assert set(pos.tolist()) <= set(idx.tolist())
    assert tau == np.sort(w[np.isfinite(w)])[-3]
    # signed zero: -0 and +0 are one tie class, tau = +0
    w = -np.abs(g.standard_normal(3000)).astype(np.float32) - 1
    z = g.choice(3000, 40, replace=False)
    w[z[:20]] = -0.0
    w[z[20:]] = 0.0
    idx, _, tau = oracle.topk_window(w, 30, lib=lib)
    assert tau == 0 and not np.signbit(tau)
    assert set(idx.tolist()) <= set(z.tolist())


def pin_short_rows(lib):
    k = 512
    for nv in (0, 1, k - 1, k):
        stride = 1024
        logits = np.full((1, stride), np.inf, np.float32)
        logits[0, :nv] = np.arange(nv, dtype=np.float32)[::-1] - 7
        kv = np.array([nv], np.int32)
        idx, vals, tau = oracle.topk_decode(logits, kv, 1, 1, k, want_values=True, lib=lib)
        assert idx[0].tolist() == list(range(nv)) + [-1] * (k - nv), nv
        want = np.concatenate([logits[0, :nv], np.full(k - nv, -FLT_MAX, np.float32)])
        assert np.array_equal(vals[0].view(np.uint32), want.view(np.uint32)), nv
        assert math.isnan(tau[0])
    # nv = k + 1: a real selection happens, so exactly one valid index is left out
    nv = k + 1
    logits = np.zeros((1, 1024), np.float32)
    logits[0, :nv] = np.arange(nv, dtype=np.float32)
    idx, vals, _ = oracle.topk_decode(logits, np.array([nv], np.int32), 1, 1, k, want_values=True, lib=lib)
    assert sorted(idx[0].tolist()) == list(range(1, nv))
    assert np.array_equal(vals[0], logits[0, idx[0]])


def pin_prefill_translation(lib):
    g = np.random.default_rng(5)
    k = 64
    for s in range(4):
        for nv in (10, 64, 65, 300, 1001):
            stride = 2048
            w = np.round(g.standard_normal(nv) * 3).astype(np.float32)
            row = np.full(stride, np.nan, np.float32)
            ks = 4 * int(g.integers(0, 64)) + s
            row[ks:ks + nv] = w
            row[:ks] = np.inf
            idx, tau = oracle.topk_prefill(row[None, :], [ks], [ks + nv], k, lib=lib)
            aligned = np.full((1, stride), -np.inf, np.float32)
            aligned[0, :nv] = w
            ref, rtau = oracle.topk_prefill(aligned, [0], [nv], k, lib=lib)
            assert idx[0].tolist() == ref[0].tolist(), (s, nv)
            assert (math.isnan(tau[0]) and math.isnan(rtau[0])) or tau[0] == rtau[0]
            # and the decode form of the same aligned window agrees
            didx, _, _ = oracle.topk_decode(aligned, np.array([nv], np.int32), 1, 1, k, lib=lib)
            assert didx[0].tolist() == ref[0].tolist()
        # windows that end exactly at the row stride, or claim to end past it (clamped to the
        # stride), equal the same scores copied to an aligned window; the row sits between poison
        # rows, so a window that runs past the stride would read poison instead
        for nv, over in ((300, 0), (300, 7), (64, 1), (1001, 5)):
            stride = 2048
            w = np.round(g.standard_normal(nv) * 3).astype(np.float32)
            rows = np.full((3, stride), GOLDEN_POISON, np.float32)
            ks = stride - nv
            rows[1, :ks] = np.inf
            rows[1, ks:] = w
            idx, tau = oracle.topk_prefill(rows, [0, ks, 0], [0, stride + over, 0], k, lib=lib)
            aligned = np.full((1, stride), -np.inf, np.float32)
            aligned[0, :nv] = w
            ref, rtau = oracle.topk_prefill(aligned, [0], [nv], k, lib=lib)
            assert idx[1].tolist() == ref[0].tolist(), (s, nv, over)
            assert (math.isnan(tau[1]) and math.isnan(rtau[0])) or tau[1] == rtau[0]


ALL_PINS = [pin_golden_decode_row_len, pin_golden_tiny_topk, pin_brute_force_tiny, pin_invariant_random,
            pin_partition_crosscheck, pin_closed_forms, pin_short_rows, pin_prefill_translation]


# ----------------------------------------------------------------------------- tests
@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_refuses_nan_in_window(oracle_lib):
    w = np.array([1, 2, np.nan, 4, 5], np.float32)
    with pytest.raises(oracle.OracleNaNError):
        oracle.topk_window(w, 2, lib=oracle_lib)
    # NaN outside the window is never looked at
    logits = np.array([[1, 2, 3, 4, 5, np.nan, np.nan, np.nan]], np.float32)
    idx, _, _ = oracle.topk_decode(logits, np.array([5], np.int32), 1, 1, 2, lib=oracle_lib)
    assert sorted(idx[0].tolist()) == [3, 4]


def test_oracle_threads_agree(oracle_lib):
    g = np.random.default_rng(17)
    logits = np.round(g.standard_normal((37, 4096)) * 2).astype(np.float32)
    kv = g.integers(0, 9000, 19).astype(np.int32)
    a, va, ta = oracle.topk_decode(logits, kv, 2, 2, 256, want_values=True, nthreads=1, lib=oracle_lib)
    b, vb, tb = oracle.topk_decode(logits, kv, 2, 2, 256, want_values=True, nthreads=4, lib=oracle_lib)
    assert np.array_equal(a, b) and np.array_equal(va, vb) and np.array_equal(ta, tb, equal_nan=True)


# Each mutant is one plausible slip in the oracle's source; the pins must catch every one.
MUTANTS = {
    "ascending_values": ("if (a->v > b->v) return -1;\n  if (a->v < b->v) return 1;",
                         "if (a->v < b->v) return -1;\n  if (a->v > b->v) return 1;"),
    "ties_by_largest_index": ("if (a->j < b->j) return -1;\n  if (a->j > b->j) return 1;",
                              "if (a->j > b->j) return -1;\n  if (a->j < b->j) return 1;"),
    "mtp_drops_plus_one": ("int64_t num = kv - next_n + (r % next_n) + 1;",
                           "int64_t num = kv - next_n + (r % next_n);"),
    "mtp_request_by_row": ("int64_t kv = kv_lens[r / next_n];", "int64_t kv = kv_lens[r % next_n];"),
    "mtp_no_empty_rule": ("if (kv < next_n) return 0;", "if (kv < 1) return 0;"),
    "no_stride_clamp": ("if (n > row_stride) n = row_stride;", ""),
    "short_rows_strict": ("if (nv <= k) {", "if (nv < k) {"),
    "pad_zero": ("out[i] = i < nv ? (int32_t)i : -1;", "out[i] = i < nv ? (int32_t)i : 0;"),
    "values_pad_zero": ("vals[i] = i < nv ? w[i] : -FLT_MAX;", "vals[i] = i < nv ? w[i] : 0.0f;"),
    "prefill_global_frame": ("logits + r * row_stride + a, nv", "logits + r * row_stride, nv"),
    "tau_off_by_one": ("*tau = scratch[k - 1].v;", "*tau = scratch[k].v;"),
    "values_from_sorted_slot": ("vals[i] = w[scratch[i].j];", "vals[i] = w[i];"),
    "no_ks_clamp": ("if (ks < 0) ks = 0;", ""),
    "no_ke_clamp": ("if (ke > row_stride) ke = row_stride;", ""),
}


def _pins_fail(lib):
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception:  # noqa: BLE001 - any failure counts as caught
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gvr_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutant pattern for {name} not found"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "mutant.c")
        open(path, "w").write(src.replace(old, new))
        so = oracle.compile_oracle(path, os.path.join(d, "libmutant.so"))
        # The pins run in a child process: a mutant that drops a bound may write past its own
        # scratch buffer, and a crash of the child counts as a caught mistake.
        code = ("import sys; sys.path[:0] = sys.argv[2:4]; import oracle, test_oracle_pins as t; "
                "print('FAILED=' + ','.join(t._pins_fail(oracle.load(sys.argv[1]))))")
        here = os.path.dirname(os.path.abspath(__file__))
        r = subprocess.run([sys.executable, "-c", code, so, os.path.dirname(here), here],
                           capture_output=True, text=True, timeout=900)
        out = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED=")]
        failed = ["(child process crashed)"] if r.returncode != 0 or not out else \
            [x for x in out[-1][len("FAILED="):].split(",") if x]
    assert failed, f"planted mistake {name} passed every pin"
