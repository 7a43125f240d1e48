"""GPU parity: libdkv (through its C ABI) against the CPU oracle.

Bit-exact on token classes, page ids, forward / reverse tables, page classes,
cursors and every byte of every live page; dequantised values bit-exact
against the oracle's dequantisation and within the quantiser's error bound of
the bf16 input.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.gpu_helpers import assert_same_state, fetch, make_compactor, oracle_state, to_device
from tests.edge_rows import dequant_bound
from tests.oracle_helpers import bf16_to_f32, f16, run_oracle

pytestmark = pytest.mark.gpu


def _run_both(w, inp_t, alpha_h=None, alpha_l=None, F=None, head0=None):
    ah = w.alpha_h if alpha_h is None else alpha_h
    al = w.alpha_l if alpha_l is None else alpha_l
    n = W.to_numpy(inp_t)
    comp = make_compactor(w, L=int(inp_t["L"]), F=F)
    pool = oracle.Pool(comp.pool.F, w.P)
    if head0 is not None:
        comp.pool.cursors.copy_(torch.tensor([head0, head0 + comp.pool.F], dtype=torch.int64))
        pool.cursors[:] = [head0, head0 + comp.pool.F]
    comp.compact(to_device(inp_t), ah, al)
    st_gpu = libdkv.dkv_get_status(comp.pool)
    st_ora, pool, tab = run_oracle(w, n, ah, al, pool=pool)
    return comp, st_gpu, st_ora, pool, tab


def test_tiny_bit_exact():
    w = W.get("tiny")
    inp = W.make_inputs(w)
    comp, sg, so, pool, tab = _run_both(w, inp)
    assert sg == so == oracle.OK
    assert_same_state(fetch(comp), oracle_state(pool, tab))


ALPHAS = [(1.0, 0.2), (2.0, 0.6), (0.0, 0.0), (1e30, 0.0), (1e30, 1e30), (0.5, 0.5)]


@pytest.mark.parametrize("alphas", ALPHAS, ids=[f"{a}-{b}" for a, b in ALPHAS])
@pytest.mark.parametrize("seed", [1, 2])
def test_small_ragged_bit_exact(alphas, seed):
    w = W.small("ragged")
    inp = W.make_inputs(w, seed=seed)
    comp, sg, so, pool, tab = _run_both(w, inp, *alphas)
    assert sg == so == oracle.OK
    assert_same_state(fetch(comp), oracle_state(pool, tab))


@pytest.mark.parametrize("shape", [
    dict(L=1, Hq=4, Hkv=4, lens=[1], P=2),
    dict(L=3, Hq=12, Hkv=3, lens=[128, 256, 129, 127], P=16),
    dict(L=1, Hq=28, Hkv=4, lens=[1000, 2049, 64], P=32, sigma=2.5, heavy_frac=0.05),
    dict(L=2, Hq=64, Hkv=8, lens=[700, 300], P=16, decay=512.0, recent=64),
    dict(L=1, Hq=7, Hkv=1, lens=[513, 5], P=6),
])
def test_shapes_bit_exact(shape):
    w = W.small("shape", **shape)
    inp = W.make_inputs(w, seed=5)
    comp, sg, so, pool, tab = _run_both(w, inp)
    assert sg == so == oracle.OK
    assert_same_state(fetch(comp), oracle_state(pool, tab))


def test_wraparound_and_successive_calls():
    """Head starts near the end of the ring; a second call continues after the first."""
    w = W.small("wrap")
    inp1, inp2 = W.make_inputs(w, seed=11), W.make_inputs(w, seed=12)
    F = 2 * w.pool_pages
    comp = make_compactor(w, F=F)
    pool = oracle.Pool(F, w.P)
    head0 = F - 37
    comp.pool.cursors.copy_(torch.tensor([head0, head0 + F], dtype=torch.int64))
    pool.cursors[:] = [head0, head0 + F]
    for inp in (inp1, inp2):
        comp.compact(to_device(inp), w.alpha_h, w.alpha_l)
        assert libdkv.dkv_get_status(comp.pool) == oracle.OK
        st, pool, tab = run_oracle(w, W.to_numpy(inp), pool=pool)
        assert st == oracle.OK
        assert_same_state(fetch(comp), oracle_state(pool, tab))
    assert int(pool.cursors[0]) // F >= 1  # the head wrapped


def test_layer_split_on_gpu():
    w = W.small("split", L=3)
    inp = W.make_inputs(w, seed=3)
    full = make_compactor(w)
    full.compact(to_device(inp), w.alpha_h, w.alpha_l)
    a = fetch(full)
    per = make_compactor(w, L=1)
    Ul = w.R * w.Hkv
    for l in range(w.L):
        il = dict(inp, L=1, k=inp["k"][l:l + 1], v=inp["v"][l:l + 1], sig_sum=inp["sig_sum"][l:l + 1])
        per.compact(to_device(il), w.alpha_h, w.alpha_l, unit_base=l * Ul)
        b = fetch(per)
        assert np.array_equal(b["fwd"], a["fwd"][l * Ul:(l + 1) * Ul])
        assert np.array_equal(b["unit_hdr"], a["unit_hdr"][l * Ul:(l + 1) * Ul])
        assert np.array_equal(b["classes"], a["classes"].reshape(w.L, -1)[l])
    for key in ("cursors", "rev_unit", "rev_idx", "page_cls", "free_list"):
        assert np.array_equal(a[key], b[key])
    live = np.nonzero(a["page_cls"])[0]
    assert np.array_equal(a["pages"][live], b["pages"][live])


def _snapshot(comp):
    st = fetch(comp)
    st.pop("classes")
    return st


def test_out_of_memory_is_all_or_nothing():
    w = W.small("nomem")
    inp = W.make_inputs(w, seed=4)
    st, pool, tab = run_oracle(w, W.to_numpy(inp))
    need = int(pool.cursors[0])
    comp = make_compactor(w, F=need - 1)
    before = _snapshot(comp)
    comp.compact(to_device(inp), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_E_NOMEM
    after = _snapshot(comp)
    for k in before:
        if k == "pages":
            continue  # free pages may be scribbled; none is live
        assert np.array_equal(before[k], after[k]), k
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK  # read clears


def test_range_error_is_all_or_nothing():
    w = W.small("range")
    inp = W.make_inputs(w, seed=6)
    st, pool, tab = run_oracle(w, W.to_numpy(inp))
    cls = tab.classes.reshape(w.L, w.T, w.Hkv)
    l, t, h = [int(x[-1]) for x in np.nonzero(cls == 2)]
    bad = dict(inp, k=inp["k"].clone())
    bad["k"][l, t, h, 77] = float("inf")
    comp = make_compactor(w)
    before = _snapshot(comp)
    comp.compact(to_device(bad), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_E_RANGE
    after = _snapshot(comp)
    for k in before:
        if k != "pages":
            assert np.array_equal(before[k], after[k]), k
    assert oracle.compact(W.to_numpy(bad), w.alpha_h, w.alpha_l, oracle.Pool(w.pool_pages, w.P),
                          oracle.Tables(w.U, w.pmax, w.rows)) == oracle.E_RANGE


def test_bad_lengths_report_lens():
    w = W.small("lens")
    inp = W.make_inputs(w, seed=7)
    comp = make_compactor(w)
    bad = dict(inp, lens=inp["lens"].clone())
    bad["lens"][0] += 1
    comp.compact(to_device(bad), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_E_LENS
    comp.compact(to_device(inp), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK


def test_scan_timeout_path_is_bounded_and_recoverable():
    """spin_limit = 0 makes every partition after the first give up at once:
    the call reports DKV_E_TIMEOUT, changes nothing, and the next call works."""
    w = W.small("timeout", L=2, lens=[5] * 40, Hq=4, Hkv=2)   # U = 160 > one partition
    inp = W.make_inputs(w, seed=8)
    comp = make_compactor(w)
    before = _snapshot(comp)
    comp.compact(to_device(inp), w.alpha_h, w.alpha_l, spin_limit=0)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_E_TIMEOUT
    after = _snapshot(comp)
    for k in before:
        if k != "pages":
            assert np.array_equal(before[k], after[k]), k
    comp.compact(to_device(inp), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    st, pool, tab = run_oracle(w, W.to_numpy(inp))
    assert_same_state(fetch(comp), oracle_state(pool, tab))


def test_empty_batch():
    w = W.small("empty", lens=[0, 0, 0])
    inp = W.make_inputs(w)
    # give the empty tensors a valid address
    inp = dict(inp, k=torch.zeros((w.L, 1, w.Hkv, 128), dtype=torch.bfloat16),
               v=torch.zeros((w.L, 1, w.Hkv, 128), dtype=torch.bfloat16),
               sig_sum=torch.zeros((w.L, 1, w.Hq)), sig_cnt=torch.zeros(1, dtype=torch.int32))
    comp = make_compactor(w, F=8)
    comp.compact(to_device(inp), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    st = fetch(comp)
    assert np.all(st["fwd"] == -1) and np.all(st["unit_hdr"] == 0) and int(st["cursors"][0]) == 0


def test_dequant_matches_oracle_and_bound():
    w = W.small("dequant", L=1, lens=[300, 129])
    inp = W.make_inputs(w, seed=9)
    comp, sg, so, pool, tab = _run_both(w, inp)
    assert sg == so == oracle.OK
    live = np.nonzero(pool.page_cls)[0]
    k, v, pos = libdkv.dkv_dequant_pages(comp.pool, torch.tensor(live, dtype=torch.int32))
    k, v, pos = k.cpu().numpy(), v.cpu().numpy(), pos.cpu().numpy()
    n = W.to_numpy(inp)
    for i, pid in enumerate(live):
        ko, vo, po = oracle.dequant_page(pool, int(pid))
        assert np.array_equal(k[i].view(np.uint32), ko.view(np.uint32))
        assert np.array_equal(v[i].view(np.uint32), vo.view(np.uint32))
        assert np.array_equal(pos[i], po)
        # bound against the bf16 input, per element, with the slot's own scale
        u = int(pool.rev_unit[pid])
        h, r = u % w.Hkv, (u // w.Hkv) % w.R
        start = sum(w.lens[:r])
        high = pool.page_cls[pid] == 2
        meta = pool.pages[pid][192 * w.P:208 * w.P].view(np.uint16).reshape(2 * w.P, 4)
        for s in np.nonzero(po >= 0)[0]:
            t = start + po[s]
            ms = f16(meta[s]).astype(np.float64)
            for x_bits, xq, sc, nb in ((n["k"][0, t, h], k[i][s], ms[0], 8 if high else 4),
                                       (n["v"][0, t, h], v[i][s], ms[2], 4 if high else 2)):
                x = bf16_to_f32(x_bits).astype(np.float64)
                assert np.all(np.abs(x - xq.astype(np.float64)) <= dequant_bound(sc, nb)), (pid, s)
    k1, v1, p1 = libdkv.dkv_dequant_page(comp.pool, int(live[0]))
    assert torch.equal(k1.cpu(), torch.from_numpy(k[0]))
