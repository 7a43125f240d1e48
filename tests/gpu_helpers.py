"""GPU-side test helpers: run libdkv through its C ABI and fetch its state."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W


def to_device(inp: dict, device="cuda") -> dict:
    out = dict(inp)
    for k in ("k", "v", "sig_sum", "sig_cnt", "lens"):
        out[k] = inp[k].to(device).contiguous()
    return out


def make_compactor(w: W.Workload, L: int | None = None, F: int | None = None) -> libdkv.Compactor:
    L = w.L if L is None else L
    return libdkv.Compactor(L, w.R, w.Hq, w.Hkv, w.T, max(w.lens + [0]), w.P,
                            w.pool_pages if F is None else F, scheme=w.scheme)


def fetch(comp: libdkv.Compactor, pages=True) -> dict:
    torch.cuda.synchronize()
    p = comp.pool
    st = {
        "classes": comp.classes.cpu().numpy(),
        "fwd": comp.tables.fwd.cpu().numpy(),
        "unit_hdr": comp.tables.unit_hdr.cpu().numpy(),
        "free_list": p.free_list.cpu().numpy(),
        "cursors": p.cursors.cpu().numpy().view(np.uint64),
        "rev_unit": p.rev_unit.cpu().numpy(),
        "rev_idx": p.rev_idx.cpu().numpy(),
        "page_cls": p.page_cls.cpu().numpy(),
    }
    if pages:
        st["pages"] = p.pages.cpu().numpy()
    return st


def oracle_state(pool: oracle.Pool, tab: oracle.Tables) -> dict:
    return {
        "classes": tab.classes, "fwd": tab.fwd, "unit_hdr": tab.unit_hdr, "free_list": pool.free_list,
        "cursors": pool.cursors, "rev_unit": pool.rev_unit, "rev_idx": pool.rev_idx,
        "page_cls": pool.page_cls, "pages": pool.pages,
    }


def assert_same_state(gpu: dict, ora: dict, page_ids=None, what=""):
    """Bit-exact comparison of classes, tables, cursors and live pages."""
    for key in ("classes", "fwd", "unit_hdr", "free_list", "cursors", "rev_unit", "rev_idx", "page_cls"):
        a, b = gpu[key], ora[key]
        if not np.array_equal(a.reshape(-1), b.reshape(-1)):
            bad = np.nonzero(a.reshape(-1) != b.reshape(-1))[0]
            raise AssertionError(f"{what}{key}: {bad.size} mismatches, first at {bad[:5]}: "
                                 f"gpu {a.reshape(-1)[bad[:5]]} oracle {b.reshape(-1)[bad[:5]]}")
    if "pages" in gpu and "pages" in ora:
        live = np.nonzero(ora["page_cls"] != 0)[0] if page_ids is None else np.asarray(page_ids)
        ga, ob = gpu["pages"][live], ora["pages"][live]
        if not np.array_equal(ga, ob):
            bad_pages = live[np.nonzero((ga != ob).any(axis=1))[0]]
            pid = bad_pages[0]
            off = np.nonzero(gpu["pages"][pid] != ora["pages"][pid])[0]
            raise AssertionError(f"{what}pages: {bad_pages.size} of {live.size} live pages differ; page {pid} "
                                 f"first bytes at {off[:8]}")
