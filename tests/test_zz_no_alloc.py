"""dkv_compact_noalloc: compaction for callers that cannot allocate device memory.

Some callers cannot hand dkv_compact a workspace: an engine whose GPU memory is
all reserved up front by its own pool allocator, or a caller with no device
allocator at all.  dkv_compact_noalloc takes its scratch from a fixed-size array
inside the library instead.  These tests check, through the C ABI, that it gives
exactly what dkv_compact gives with a caller workspace, on two calls in a row
on the same pools (the second call continues after the first), and that a batch
too large for the built-in scratch is refused up front.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.gpu_helpers import fetch, make_compactor, to_device

pytestmark = pytest.mark.gpu


def _same(a: dict, b: dict):
    for key in ("classes", "fwd", "unit_hdr", "free_list", "cursors", "rev_unit", "rev_idx", "page_cls"):
        assert np.array_equal(a[key], b[key]), key
    live = np.nonzero(a["page_cls"])[0]
    assert live.size > 0
    assert np.array_equal(a["pages"][live], b["pages"][live])


@pytest.mark.parametrize("shape", [dict(), dict(L=3, Hq=28, Hkv=4, lens=[1000, 333, 0, 2049], P=32)])
def test_noalloc_matches_workspace_call_twice(shape):
    w = W.small("noalloc", **shape)
    F = 2 * w.pool_pages
    with_ws = make_compactor(w, F=F)
    no_ws = make_compactor(w, F=F)
    for seed in (21, 22):
        inp = to_device(W.make_inputs(w, seed=seed))
        with_ws.compact(inp, w.alpha_h, w.alpha_l)
        assert libdkv.dkv_get_status(with_ws.pool) == libdkv.DKV_OK
        libdkv.dkv_compact_noalloc(no_ws.batch(inp), w.alpha_h, w.alpha_l, no_ws.pool, no_ws.tables)
        assert libdkv.dkv_get_status(no_ws.pool) == libdkv.DKV_OK
        torch.cuda.synchronize()
        _same(fetch(with_ws), fetch(no_ws))


def test_noalloc_rejects_batches_over_the_scratch_limit():
    w = W.get("longcot")  # needs about 97 MiB of scratch, above the 16 MiB built in
    b = libdkv.dkv_batch(w.L, w.R, w.Hq, w.Hkv, 128, max(w.lens), w.T, 0, 256, 256, 256, 256, 256, 256)
    assert libdkv.dkv_workspace_size(b) > 16 << 20
    pool = libdkv.dkv_pool(64, 16, 0, 256, 256, 256, 256, 256, 256, 256)
    tab = libdkv.dkv_tables(256, 1100, 0, 256)
    par = libdkv.dkv_params(1.0, 0.2, -1, 0, None)
    rc = libdkv.load().dkv_compact_noalloc(ctypes.byref(b), ctypes.byref(par), ctypes.byref(pool),
                                          ctypes.byref(tab), None)
    assert rc == libdkv.DKV_E_INVAL
