"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (one dkv_compact over the whole batch).

Compared with the CPU oracle, bit-exact: the class of every token row, every
unit's header and forward row, the reverse table and class of every page, the
cursors, and every byte of the pages of sampled units (two layers; the oracle
quantises only those).  The oracle runs one layer at a time on the same pool
(global unit ids via unit_base), so it needs host copies of the significance
sums of every layer but of K and V only for the sampled layers.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _host(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().numpy()


def _bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _run_full(name: str):
    w = W.get(name)
    dev = torch.device("cuda", 0)
    inp = W.make_inputs(w, device=dev)
    comp = libdkv.Compactor(w.L, w.R, w.Hq, w.Hkv, w.T, max(w.lens), w.P, w.pool_pages, device=dev)
    comp.compact(inp, w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    torch.cuda.synchronize()

    Ul = w.R * w.Hkv
    sample_layers = [0, w.L - 1]
    sample_req = sorted({0, w.R // 2, w.R - 1})
    pool = oracle.Pool(w.pool_pages, w.P)
    cls_o = np.empty(w.rows, dtype=np.uint8)
    fwd_o = np.empty((w.U, w.pmax), dtype=np.int32)
    hdr_o = np.empty((w.U, 4), dtype=np.int32)
    cnt = _host(inp["sig_cnt"])
    lens = _host(inp["lens"])
    dummy = np.zeros((1, 1, w.Hkv, 128), dtype=np.uint16)
    for l in range(w.L):
        sampled = l in sample_layers
        layer = {"L": 1, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T, "unit_base": l * Ul,
                 "sig_sum": _host(inp["sig_sum"][l:l + 1]), "sig_cnt": cnt, "lens": lens,
                 "k": _bf16_host(inp["k"][l:l + 1]) if sampled else dummy,
                 "v": _bf16_host(inp["v"][l:l + 1]) if sampled else dummy}
        mask = np.zeros(Ul, dtype=np.uint8)
        if sampled:
            for r in sample_req:
                mask[r * w.Hkv:(r + 1) * w.Hkv] = 1
        tab = oracle.Tables(Ul, w.pmax, w.T * w.Hkv)
        assert oracle.compact(layer, w.alpha_h, w.alpha_l, pool, tab, mask) == oracle.OK
        cls_o[l * w.T * w.Hkv:(l + 1) * w.T * w.Hkv] = tab.classes
        fwd_o[l * Ul:(l + 1) * Ul] = tab.fwd
        hdr_o[l * Ul:(l + 1) * Ul] = tab.unit_hdr

    assert np.array_equal(_host(comp.classes[:w.rows]), cls_o)
    assert np.array_equal(_host(comp.tables.unit_hdr), hdr_o)
    assert np.array_equal(_host(comp.tables.fwd), fwd_o)
    for key in ("free_list", "rev_unit", "rev_idx", "page_cls"):
        assert np.array_equal(_host(getattr(comp.pool, key)), getattr(pool, key)), key
    assert np.array_equal(_host(comp.pool.cursors).view(np.uint64), pool.cursors)

    # every byte of the sampled units' pages
    ids = []
    for l in sample_layers:
        for r in sample_req:
            for h in range(w.Hkv):
                row = fwd_o[l * Ul + r * w.Hkv + h]
                ids.extend(int(x) for x in row[row >= 0])
    ids = np.array(sorted(ids), dtype=np.int64)
    assert ids.size > 0
    got = _host(comp.pool.pages[torch.from_numpy(ids).to(dev)])
    assert np.array_equal(got, pool.pages[ids])
    # dequantisation of a few of them, bit-exact with the oracle's
    some = ids[:: max(1, ids.size // 16)]
    k, v, pos = libdkv.dkv_dequant_pages(comp.pool, torch.from_numpy(some).to(torch.int32))
    k, v, pos = _host(k), _host(v), _host(pos)
    for i, pid in enumerate(some):
        ko, vo, po = oracle.dequant_page(pool, int(pid))
        assert np.array_equal(k[i].view(np.uint32), ko.view(np.uint32))
        assert np.array_equal(v[i].view(np.uint32), vo.view(np.uint32))
        assert np.array_equal(pos[i], po)
    frac = np.bincount(cls_o, minlength=3) / cls_o.size
    return frac


def test_full_llama_prefill():
    frac = _run_full("llama")
    # class mix of the log-normal(2) generator: about 11% pruned, 39% K4V2, 50% K8V4
    assert abs(frac[2] - 0.499) < 0.01 and abs(frac[1] - 0.390) < 0.01


def test_full_qwen_ragged():
    frac = _run_full("qwen")
    assert frac[0] > 0.3  # heavy hitters x50 at sigma 2.5: many tokens pruned


def test_full_long_cot():
    _run_full("longcot")
