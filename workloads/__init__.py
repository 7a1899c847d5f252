"""Seeded synthetic inputs for the exact per-row top-K (shared by tests and bench).

This module only synthesises inputs: it holds none of the selection method's
arithmetic, and it imports neither the CUDA path nor the oracle.  Every array
is numpy on the host; callers move them to the device themselves.

The pages measure on captured model rows (GLM-5.3-Flash MRCR rows, DeepSeek
V3.2/V4 decode captures, a 144-case stress set) that are not available; these
seeded generators stand in for them with the shapes, strides, length mixes and
value distributions described for each workload.

Randomness: ``numpy.random.Generator(numpy.random.Philox(seed))``; workload c
uses seed 1000 + c, variants 1000 + 10 c + v; row r draws from
``Philox(seed).jumped(r + 1)`` and shared draws (lengths, positions) from
``Philox(seed).jumped(0)``.

Poison outside a window cycles by column: decode pads through
(+inf, NaN, 3e38); prefill pads through (+inf, NaN, 3e38, -inf).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DECODE_POISON = np.array([np.inf, np.nan, 3e38], dtype=np.float32)
PREFILL_POISON = np.array([np.inf, np.nan, 3e38, -np.inf], dtype=np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed).jumped(stream))


def roundup(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclass
class DecodeCase:
    """Decode batch: logits [rows, row_stride], kv_lens per request."""
    name: str
    logits: np.ndarray
    kv_lens: np.ndarray
    next_n: int
    compress_ratio: int
    k: int
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.logits.shape[0]

    @property
    def row_stride(self) -> int:
        return self.logits.shape[1]

    def row_lengths(self) -> np.ndarray:
        """Per-row valid length, for sizing only (bytes moved, poisoning)."""
        r = np.arange(self.rows)
        kv = self.kv_lens[r // self.next_n].astype(np.int64)
        num = kv - self.next_n + (r % self.next_n) + 1
        n = np.where(kv < self.next_n, 0, num // self.compress_ratio)
        return np.minimum(n, self.row_stride)


@dataclass
class PrefillCase:
    """Prefill tile: logits [rows, row_stride], per-row window [row_starts, row_ends)."""
    name: str
    logits: np.ndarray
    row_starts: np.ndarray
    row_ends: np.ndarray
    k: int
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.logits.shape[0]

    @property
    def row_stride(self) -> int:
        return self.logits.shape[1]

    def window_lengths(self) -> np.ndarray:
        ks = np.maximum(self.row_starts.astype(np.int64), 0)
        ke = np.minimum(self.row_ends.astype(np.int64), self.row_stride)
        return np.maximum(ke - ks, 0)


def _poison_decode(logits: np.ndarray, n: np.ndarray) -> None:
    cols = np.arange(logits.shape[1])
    pad_vals = DECODE_POISON[cols % DECODE_POISON.size]
    for r in range(logits.shape[0]):
        logits[r, n[r]:] = pad_vals[n[r]:]


def _poison_prefill(logits: np.ndarray, ks: np.ndarray, ke: np.ndarray) -> None:
    cols = np.arange(logits.shape[1])
    pad_vals = PREFILL_POISON[cols % PREFILL_POISON.size]
    for r in range(logits.shape[0]):
        a, b = max(int(ks[r]), 0), min(int(ke[r]), logits.shape[1])
        logits[r, :a] = pad_vals[:a]
        if b < logits.shape[1]:
            logits[r, max(b, a):] = pad_vals[max(b, a):]


def _decode_lengths(kv_lens, next_n, cr, rows, stride):
    r = np.arange(rows)
    kv = kv_lens[r // next_n].astype(np.int64)
    num = kv - next_n + (r % next_n) + 1
    return np.minimum(np.where(kv < next_n, 0, num // cr), stride)


# --------------------------------------------------------------------------- workload 1
def single_decode_row(seed: int = 1001, n: int = 8192, k: int = 512) -> DecodeCase:
    """One decode row: n valid scores ~ N(0,1), stride n, K=512, next_n = cr = 1."""
    rng = _rng(seed, 1)
    logits = rng.standard_normal((1, n), dtype=np.float32)
    return DecodeCase("single_decode_row", logits, np.array([n], np.int32), 1, 1, k,
                      {"workload": f"decode rows=1 n={n} stride={n} K={k}"})


# --------------------------------------------------------------------------- workload 2
def decode_batch(seed: int = 1002, requests: int = 64, next_n: int = 2, cr: int = 4, k: int = 1024,
                 stride: int = 131072, kv_lo: int = 16384, kv_hi: int = 524288,
                 boundary: bool = True, empty_request: bool = False) -> DecodeCase:
    """Decode batch: 64 requests x next_n=2 rows, kv_lens ~ U{16K..524K}, cr=4, K=1024.

    Scores of row r are z_j + u_r * j / n_r with z ~ N(0,1) and u_r ~ U(0,2):
    standard normal plus a position-linear bias.  Requests 61/62/63 get
    kv_len 4093/4097/4101 (n = K-1, K, K+1 at cr=4); with ``empty_request``
    request 60 gets kv_len = 1 (empty rows).  Pad columns j >= n are poisoned.
    """
    g0 = _rng(seed, 0)
    kv = g0.integers(kv_lo, kv_hi, size=requests, endpoint=True).astype(np.int32)
    if boundary and requests >= 64:
        kv[61], kv[62], kv[63] = 4 * (k - 1) + 1, 4 * k + 1, 4 * (k + 1) + 1
    if empty_request and requests >= 61:
        kv[60] = 1
    rows = requests * next_n
    n = _decode_lengths(kv, next_n, cr, rows, stride)
    logits = np.empty((rows, stride), np.float32)
    for r in range(rows):
        g = _rng(seed, r + 1)
        u = g.uniform(0.0, 2.0)
        nr = int(n[r])
        z = g.standard_normal(nr, dtype=np.float32).astype(np.float64)
        if nr:
            logits[r, :nr] = (z + u * np.arange(nr) / nr).astype(np.float32)
    _poison_decode(logits, n)
    return DecodeCase("decode_batch", logits, kv, next_n, cr, k,
                      {"workload": f"decode requests={requests} next_n={next_n} rows={rows} cr={cr} K={k} "
                                   f"stride={stride} kv_lens~U[{kv_lo},{kv_hi}]"})


def peaky_decode_batch(seed: int = 1006, requests: int = 64, next_n: int = 2, cr: int = 4, k: int = 1024,
                       stride: int = 131072, kv_lo: int = 16384, kv_hi: int = 524288,
                       hot_frac: float = 0.015) -> DecodeCase:
    """The decode batch's geometry with block-concentrated scores, a stand-in for captured
    attention rows (the block-skip pass targets them): a low N(0,1) - 4 background, the first
    and last 128 positions (sink and recent tokens) and a random hot_frac of the 32-score
    blocks raised by +5.  Pad columns j >= n are poisoned.
    """
    g0 = _rng(seed, 0)
    kv = g0.integers(kv_lo, kv_hi, size=requests, endpoint=True).astype(np.int32)
    rows = requests * next_n
    n = _decode_lengths(kv, next_n, cr, rows, stride)
    logits = np.empty((rows, stride), np.float32)
    for r in range(rows):
        g = _rng(seed, r + 1)
        nr = int(n[r])
        if not nr:
            continue
        x = g.standard_normal(nr, dtype=np.float32) - 4.0
        nb = (nr + 31) // 32
        hot = g.random(nb) < hot_frac
        boost = np.repeat(hot, 32)[:nr].astype(np.float32) * 5.0
        boost[:128] = 5.0
        boost[-128:] = 5.0
        logits[r, :nr] = x + boost
    _poison_decode(logits, n)
    return DecodeCase("peaky_decode_batch", logits, kv, next_n, cr, k,
                      {"workload": f"peaky decode requests={requests} next_n={next_n} rows={rows} cr={cr} K={k} "
                                   f"stride={stride} hot blocks {hot_frac}"})


# --------------------------------------------------------------------------- workload 3
def prefill_tile(seed: int = 1003, rows: int = 4096, k: int = 2048,
                 lengths=(512, 1536, 4096, 8192)) -> PrefillCase:
    """Prefill q-tile: 4 packed requests, causal windows, ks % 4 covering {0,1,2,3}.

    Request q starts at column off_q with a gap of q poisoned columns before
    it, so off = (0, 513, 2051, 6150) for the default lengths.  Tile row i is
    query position floor(i * total / rows) of the ungapped packed sequence
    (floor(3.5 i) for the default 4096 rows of 14336 tokens); its window is
    [off_q, off_q + pos + 1).  Rows 4090..4095 are overridden to positions
    2046, 2047, 2048 of requests 2 and 3 (nv = K-1, K, K+1).  Stride is the
    width plus >=256 floats of slack rounded to 256 floats (1024 B).
    """
    lengths = list(lengths)
    # a gap of q poisoned columns before request q: off_q = sum(L_<q) + (1 + ... + q)
    offs = [sum(lengths[:q]) + q * (q + 1) // 2 for q in range(len(lengths))]
    width = offs[-1] + lengths[-1]
    stride = roundup(width + 256, 256)
    ends = np.cumsum(lengths)
    total = int(ends[-1])
    ks = np.empty(rows, np.int32)
    ke = np.empty(rows, np.int32)
    for i in range(rows):
        p = min(i * total // rows, total - 1)  # floor(3.5 i) for 4096 rows of 14336 tokens
        q = int(np.searchsorted(ends, p, side="right"))
        pos = p - (int(ends[q - 1]) if q else 0)
        ks[i], ke[i] = offs[q], offs[q] + pos + 1
    if rows >= 4096 and len(lengths) >= 4:
        for t, (q, pos) in enumerate([(2, k - 2), (2, k - 1), (2, k), (3, k - 2), (3, k - 1), (3, k)]):
            i = rows - 6 + t
            ks[i], ke[i] = offs[q], offs[q] + pos + 1
    logits = np.empty((rows, stride), np.float32)
    for r in range(rows):
        g = _rng(seed, r + 1)
        nv = int(ke[r] - ks[r])
        logits[r, ks[r]:ke[r]] = g.standard_normal(nv, dtype=np.float32)
    _poison_prefill(logits, ks, ke)
    return PrefillCase("prefill_tile", logits, ks, ke, k,
                       {"workload": f"prefill rows={rows} K={k} requests={tuple(lengths)} stride={stride}",
                        "offsets": offs})


# --------------------------------------------------------------------------- workload 4
ADVERSARIAL_VARIANTS = ("base", "all_equal", "two_valued", "neg_inf_10pct", "neg_inf_tau",
                        "signed_zero_tau", "pos_inf_class")


def adversarial_row(variant: str = "base", seed: int = 1004, kv_len: int = 459852, cr: int = 4,
                    stride: int = 131072, k: int = 512) -> DecodeCase:
    """Adversarial single decode row: n = 114963 of stride 131072, K=512, cr=4.

    base: positions [0, n/5) ~ 20 N(0,1) + 50, the rest ~ 40 N(0,1) + 60,
    600 distinct positions in [n/5, n) replaced by U(150, 250) -- a prefix
    sample underestimates tau.  Variants (seed 1040 + v): all_equal (1.0),
    two_valued (50/50 of 1.0 / 2.0), neg_inf_10pct (10% of positions -inf),
    neg_inf_tau (more than n - K positions -inf, so tau = -inf),
    signed_zero_tau (a -0/+0 mix straddling tau), pos_inf_class (K-3 +inf).
    """
    if variant not in ADVERSARIAL_VARIANTS:
        raise ValueError(variant)
    v = ADVERSARIAL_VARIANTS.index(variant)
    seed = seed if v == 0 else 1040 + v
    n = min((kv_len - 1 + 0 + 1) // cr, stride)
    g0 = _rng(seed, 0)
    g = _rng(seed, 1)
    head = n // 5
    row = np.empty(n, np.float32)
    row[:head] = (20.0 * g.standard_normal(head) + 50.0).astype(np.float32)
    row[head:] = (40.0 * g.standard_normal(n - head) + 60.0).astype(np.float32)
    spikes = g0.choice(np.arange(head, n), size=600, replace=False)
    row[spikes] = g.uniform(150.0, 250.0, size=600).astype(np.float32)
    if variant == "all_equal":
        row[:] = 1.0
    elif variant == "two_valued":
        row[:] = np.where(g.random(n) < 0.5, 1.0, 2.0).astype(np.float32)
    elif variant == "neg_inf_10pct":
        pos = g0.choice(n, size=n // 10, replace=False)
        row[pos] = -np.inf
    elif variant == "neg_inf_tau":
        pos = g0.choice(n, size=n - k + 100, replace=False)
        row[pos] = -np.inf
    elif variant == "signed_zero_tau":
        # K/2 positive values, then a block of zeros (half -0) that must hold tau.
        row[:] = -(np.abs(g.standard_normal(n)) + 1.0).astype(np.float32)
        pos = g0.choice(n, size=k // 2 + 2 * k, replace=False)
        row[pos[: k // 2]] = (np.abs(g.standard_normal(k // 2)) + 1.0).astype(np.float32)
        zeros = pos[k // 2:]
        row[zeros] = np.where(np.arange(zeros.size) % 2 == 0, np.float32(-0.0), np.float32(0.0))
    elif variant == "pos_inf_class":
        pos = g0.choice(n, size=k - 3, replace=False)
        row[pos] = np.inf
    logits = np.empty((1, stride), np.float32)
    logits[0, :n] = row
    _poison_decode(logits, np.array([n]))
    return DecodeCase(f"adversarial_{variant}", logits, np.array([kv_len], np.int32), 1, cr, k,
                      {"workload": f"adversarial {variant} n={n} stride={stride} K={k} cr={cr}"})


# --------------------------------------------------------------------------- workload 5
SWEEP_BS = (1, 4, 16, 64, 256)
SWEEP_N = (16384, 32768, 65536, 131072)
SWEEP_K = (512, 1024, 2048)


def _heavy_tail_rows(seed: int, rows: int, n: int, stride: int) -> np.ndarray:
    logits = np.empty((rows, stride), np.float32)
    for r in range(rows):
        g = _rng(seed, r + 1)
        x = g.standard_normal(n, dtype=np.float32)
        spikes = g.choice(n, size=max(1, n // 100), replace=False)
        pareto = (1.0 - g.random(spikes.size)) ** (-1.0 / 1.5)
        x[spikes] = (x[spikes] + pareto).astype(np.float32)
        logits[r, :n] = x
    return logits


def sweep_decode(bs: int, n: int, k: int, seed: int | None = None) -> DecodeCase:
    """Throughput sweep, decode mode: next_n = cr = 1, kv_len = N, stride = N rounded to 64.

    Scores ~ N(0,1) with 1% of positions raised by a Pareto(alpha=1.5, x_m=1) spike.
    """
    seed = seed if seed is not None else 1005
    stride = roundup(n, 64)
    logits = _heavy_tail_rows(seed, bs, n, stride)
    _poison_decode(logits, np.full(bs, n))
    return DecodeCase(f"sweep_decode_bs{bs}_n{n}_k{k}", logits, np.full(bs, n, np.int32), 1, 1, k,
                      {"workload": f"sweep decode BS={bs} N={n} K={k} stride={stride}"})


def sweep_prefill(bs: int, n: int, k: int, seed: int | None = None) -> PrefillCase:
    """Throughput sweep, prefill mode: window [r % 4, N) per row (all four lead offsets)."""
    seed = seed if seed is not None else 1005
    stride = roundup(n, 64)
    logits = _heavy_tail_rows(seed, bs, n, stride)
    ks = (np.arange(bs) % 4).astype(np.int32)
    ke = np.full(bs, n, np.int32)
    _poison_prefill(logits, ks, ke)
    return PrefillCase(f"sweep_prefill_bs{bs}_n{n}_k{k}", logits, ks, ke, k,
                       {"workload": f"sweep prefill BS={bs} N={n} K={k} stride={stride}"})
