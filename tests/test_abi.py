"""Host-side checks of the C ABI (no GPU needed).

The library must build for sm_103a, load, export every function that
include/gvr_topk.h declares, reject bad arguments with the documented status
codes before touching the device, and choose launch geometries whose register
capacity covers the row envelope.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gvr_topk.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_exact_gb300 import _build
    _build.build_library()
    import sparse_attention_indexer_exact_gb300 as gvr
    return gvr.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    for want in ("topk_decode", "topk_prefill", "topk_decode_ex", "topk_prefill_ex", "gvr_status_string",
                 "gvr_plan"):
        assert want in names, names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libgvrtopk.so does not export {name}"


def test_status_strings(lib):
    for code in range(7):
        s = lib.gvr_status_string(code)
        assert s and len(s) > 1
    assert lib.gvr_status_string(0) == b"ok"
    assert lib.gvr_status_string(99) == b"unknown status"


# Fake, never-dereferenced device addresses: validation must reject before any device work.
ALIGNED = 0x10000
K = 512


def test_decode_argument_errors(lib):
    f = lib.topk_decode
    ok = (ALIGNED, 1024, 4, ALIGNED, 1, 1, K, ALIGNED, None, None)

    def call(**kw):
        args = list(ok)
        names = ["logits", "row_stride", "num_rows", "kv_lens", "next_n", "cr", "k", "indices", "values", "stream"]
        for key, v in kw.items():
            args[names.index(key)] = v
        return f(*args)

    assert call(logits=None) == 1
    assert call(kv_lens=None) == 1
    assert call(indices=None) == 1
    assert call(logits=ALIGNED + 4) == 2
    assert call(indices=ALIGNED + 2) == 2
    assert call(values=ALIGNED + 1) == 2
    assert call(row_stride=1026) == 3
    assert call(row_stride=0) == 3
    assert call(row_stride=1 << 31) == 3
    for bad_k in (0, 1, 256, 511, 513, 4096):
        assert call(k=bad_k) == 4
    assert call(num_rows=-1) == 5
    assert call(next_n=0) == 5
    assert call(cr=0) == 5
    assert call(num_rows=0, logits=None, indices=None, kv_lens=None) == 0  # empty batch: no-op


def test_hinted_argument_errors(lib):
    f = lib.topk_decode_hinted
    ok = [ALIGNED, 1024, 4, ALIGNED, 1, 1, K, ALIGNED, K, ALIGNED, None, None, None]
    names = ["logits", "row_stride", "num_rows", "kv_lens", "next_n", "cr", "k", "pre_idx", "pre_stride",
             "indices", "values", "stream", "options"]

    def call(**kw):
        args = list(ok)
        for key, v in kw.items():
            args[names.index(key)] = v
        return f(*args)

    assert call(pre_idx=None) == 1
    assert call(pre_idx=ALIGNED + 2) == 2
    assert call(pre_stride=K - 1) == 5
    assert call(logits=None) == 1
    assert call(logits=ALIGNED + 4) == 2
    assert call(k=300) == 4
    assert call(next_n=0) == 5
    assert call(num_rows=0, logits=None, indices=None, kv_lens=None, pre_idx=None) == 0


def test_blockskip_argument_errors(lib):
    f = lib.topk_decode_blockskip
    ok = [ALIGNED, 1024, 4, ALIGNED, 1, 1, K, ALIGNED, 32, ALIGNED, None, None, None]
    names = ["logits", "row_stride", "num_rows", "kv_lens", "next_n", "cr", "k", "bmax", "bmax_stride",
             "indices", "values", "stream", "options"]

    def call(**kw):
        args = list(ok)
        for key, v in kw.items():
            args[names.index(key)] = v
        return f(*args)

    assert call(bmax=None) == 1
    assert call(bmax=ALIGNED + 1) == 2
    assert call(bmax_stride=31) == 5
    assert call(row_stride=1028, bmax_stride=32) == 5  # ceil(1028 / 32) = 33 blocks
    assert call(row_stride=1028, bmax_stride=33) != 5
    assert call(logits=None) == 1
    assert call(k=300) == 4
    assert call(num_rows=0, logits=None, indices=None, kv_lens=None, bmax=None) == 0


def test_prefill_argument_errors(lib):
    f = lib.topk_prefill
    assert f(None, 1024, 4, ALIGNED, ALIGNED, K, ALIGNED, None) == 1
    assert f(ALIGNED, 1024, 4, None, ALIGNED, K, ALIGNED, None) == 1
    assert f(ALIGNED, 1024, 4, ALIGNED, None, K, ALIGNED, None) == 1
    assert f(ALIGNED + 8, 1024, 4, ALIGNED, ALIGNED, K, ALIGNED, None) == 2
    assert f(ALIGNED, 1022, 4, ALIGNED, ALIGNED, K, ALIGNED, None) == 3
    assert f(ALIGNED, 1024, 4, ALIGNED, ALIGNED, 1000, ALIGNED, None) == 4
    assert f(ALIGNED, 1024, -3, ALIGNED, ALIGNED, K, ALIGNED, None) == 5
    assert f(None, 1024, 0, None, None, K, None, None) == 0


def test_option_errors(lib):
    import sparse_attention_indexer_exact_gb300 as gvr
    # the balanced kernel's flags (512, 1024) belong to the *_ws entry points only; the short-row
    # and cluster kernels cannot both be forced; 16384 is no flag
    for bad in (dict(cluster_size=3), dict(cluster_size=32), dict(ring_stages=2), dict(ring_stages=17), dict(reserved=1),
                dict(flags=512), dict(flags=1024), dict(flags=256 | 4096), dict(flags=16384)):
        o = gvr.Options(**bad)
        st = lib.topk_decode_ex(ALIGNED, 1024, 4, ALIGNED, 1, 1, K, ALIGNED, None, None, ctypes.byref(o))
        assert st == 5, bad


@pytest.mark.parametrize("stride", [4, 64, 1024, 8192, 14848, 65536, 131072, 131076, 262144, 1 << 20])
@pytest.mark.parametrize("rows", [1, 4, 64, 128, 4096])
@pytest.mark.parametrize("k", [512, 2048])
def test_plan_geometry(lib, stride, rows, k):
    import sparse_attention_indexer_exact_gb300 as gvr
    d = gvr.plan(stride, rows, k, sm_count=152)
    if stride <= 16384 and rows <= 4 * 2 * 152:  # the short-row kernel: four waves of two CTAs per SM
        assert (d["cluster_size"], d["ring_stages"], d["threads"]) == (1, 0, 1024), d
        assert 16 * (stride // 4 + 1) < d["smem_bytes"] <= (228 * 1024 - 2 * 1024) // 2, d
    else:
        assert d["threads"] == 128, d
    p = gvr.plan(stride, rows, k, gvr.Options(flags=256), sm_count=152)  # the cluster kernel's geometry
    cs = p["cluster_size"]
    assert cs in (1, 2, 4, 8, 16)
    share_vec = -(-(stride // 4) // cs)
    if stride // 4 >= 8 * 8192:
        assert cs >= 8  # long rows always spread over a full cluster (shares of at most 8192 float4)
    if rows * 8 * 2 <= 7 * 152 and stride // 4 >= 8 * 256:
        assert cs >= 8  # few rows: spread each row wide
    if rows * 16 * 2 <= 7 * 152 and stride // 4 >= 16 * 256:
        assert cs == 16  # very few long rows: sixteen CTAs each
    assert share_vec <= max(8192, -(-(stride // 4) // 16))  # balanced shares
    assert p["threads"] == 128 and 3 <= p["ring_stages"] <= 16
    per_sm = min(7, (228 * 1024) // (p["smem_bytes"] + 1024))
    per_sm_min = min(7, (228 * 1024) // (gvr.plan(stride, rows, k, gvr.Options(ring_stages=3), sm_count=152)
                                       ["smem_bytes"] + 1024))
    if p["ring_stages"] > 3:
        # a deeper ring only when it keeps the shallowest ring's occupancy, or while every
        # cluster stays resident at once, and never deeper than the share
        assert per_sm >= per_sm_min or rows * cs <= 152 * per_sm
        assert p["ring_stages"] <= -(-share_vec // 256)


def test_plan_short_kernel_policy(lib):
    """Plain calls go to the short-row kernel while the stride fits it and the rows fit four
    waves of its CTAs; flags other than its own (and forced rescue) keep the cluster kernel."""
    import sparse_attention_indexer_exact_gb300 as gvr
    short = lambda stride, rows, o=None: gvr.plan(stride, rows, 1024, o, sm_count=152)["threads"] == 1024
    assert short(16384, 1216) and not short(16384, 1217) and not short(16388, 1)
    assert short(4, 1) and short(8192, 64)
    assert short(16384, 4096, gvr.Options(flags=4096)) and short(16384, 4096, gvr.Options(flags=4096 | 1))
    assert short(8192, 1, gvr.Options(flags=4096 | 2048)) and short(8192, 1, gvr.Options(flags=4096 | 2048 | 1))
    for flags in (4096 | 16, 4096 | 32, 4096 | 128, 4096 | 2):  # its flag with another: the cluster kernel
        assert not short(8192, 1, gvr.Options(flags=flags)), flags
    for flags in (1, 2, 4, 8, 16, 32, 64, 128, 256, 2048):
        assert not short(8192, 1, gvr.Options(flags=flags)), flags
    assert not short(8192, 1, gvr.Options(cluster_size=2)) and not short(8192, 1, gvr.Options(ring_stages=4))
    assert short(8192, 1, gvr.Options(row_stats=0))


def test_plan_respects_overrides(lib):
    import sparse_attention_indexer_exact_gb300 as gvr
    o = gvr.Options(cluster_size=2, ring_stages=5)
    p = gvr.plan(131072, 1, 1024, o, sm_count=152)
    assert p["cluster_size"] == 2 and p["ring_stages"] == 5


def test_product_path_has_no_oracle_dependency():
    """The CUDA path and its binding never import or link the oracle (and vice versa)."""
    pkg = os.path.join(ROOT, "sparse_attention_indexer_exact_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in text.lower(), f"{fn} mentions the oracle"
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith((".py", ".c")):
            text = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "sparse_attention_indexer_exact_gb300" not in text and "gvr_topk.h" not in text


def test_binding_refuses_tensors_on_different_devices():
    # The binding launches on logits' device with every pointer it is given; a tensor on another
    # device must be refused on the host before anything is enqueued.
    import types

    import torch

    import sparse_attention_indexer_exact_gb300 as gvr
    d0, d1 = torch.device("cuda", 0), torch.device("cuda", 1)
    on = lambda d: types.SimpleNamespace(device=d)  # noqa: E731 - only .device is looked at
    gvr._same_device(d0, kv_lens=on(d0), indices=on(d0), values=None)
    for name in ("kv_lens", "indices", "values", "pre_idx", "block_max", "row_starts", "row_ends"):
        with pytest.raises(ValueError, match=name):
            gvr._same_device(d0, **{name: on(d1)})


def test_workspace_size_for_a_device_shape(lib):
    # The balanced kernel's workspace: per-row counters, then per chunk (6 CTAs per SM) a count
    # and 4096 published (score, index) pairs.  Sized without touching a device.
    size = ctypes.c_size_t(0)
    assert lib.gvr_workspace_size(152, ctypes.byref(size)) == 0
    grid = 152 * 6
    assert size.value == 512 * 4 + grid * 4 + grid * 4096 * 8
    assert lib.gvr_workspace_size(152, None) == 1
