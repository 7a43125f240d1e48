"""GPU parity of the precision schemes K8V2/K4V1 and K4V8/K2V4 beside
K8V4/K4V2 (DiffKV review, free-parameter list: the precision-level scheme was
chosen by comparing K8V4, K4V8, K8V2, K4V2, K2V4 and K4V1), through the C ABI,
byte for byte against the oracle: prefill compaction on a ragged batch and on
the quantiser's edge rows (ties, clamps, subnormal scales and minima, signed
zeros, +-65280), generation steps with demotions through k_demote and the
in-place requantiser, and page dequantisation."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests import edge_rows as E
from tests.decode_helpers import HostDecode, check_state
from tests.gpu_helpers import assert_same_state, fetch, make_compactor, oracle_state, to_device
from tests.oracle_helpers import run_oracle
from tests.test_decode_gpu import _run, check_slot_index, compare, gpu_decoder, gpu_state
from tests.test_quantizer_edges_gpu import _check_bound, _edge_update

pytestmark = pytest.mark.gpu

SCHEMES = [0, 1, 2]


@pytest.mark.parametrize("scheme", SCHEMES)
@pytest.mark.parametrize("alphas", [(1.0, 0.2), (0.0, 0.0), (1e30, 0.0)], ids=["mixed", "all_high", "all_low"])
def test_ragged_prefill_bit_exact(scheme, alphas):
    w = W.small("sch", lens=[300, 7, 517, 0, 129], scheme=scheme)
    inp = W.make_inputs(w, seed=2)
    comp = make_compactor(w)
    assert comp.pool.pages.shape[1] == oracle.page_bytes(w.P, scheme)
    comp.compact(to_device(inp), *alphas)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    st, pool, tab = run_oracle(w, W.to_numpy(inp), *alphas)
    assert st == oracle.OK
    assert_same_state(fetch(comp), oracle_state(pool, tab))
    live = np.nonzero(pool.page_cls)[0][:64]
    k, v, pos = libdkv.dkv_dequant_pages(comp.pool, torch.tensor(live, dtype=torch.int32))
    for i, pid in enumerate(live):
        ko, vo, po = oracle.dequant_page(pool, int(pid))
        assert np.array_equal(k[i].cpu().numpy().view(np.uint32), ko.view(np.uint32))
        assert np.array_equal(v[i].cpu().numpy().view(np.uint32), vo.view(np.uint32))
        assert np.array_equal(pos[i].cpu().numpy(), po)


@pytest.mark.parametrize("scheme", [1, 2])
@pytest.mark.parametrize("shape", [dict(lens=[150, 37, 200], Hq=4, Hkv=2, L=2, P=16),
                                   dict(lens=[129, 1, 64], Hq=8, Hkv=1, L=1, P=2)])
def test_edge_rows_prefill_bit_exact(scheme, shape):
    w, inp, aim = E.edge_batch(shape["lens"], shape["Hq"], shape["Hkv"], seed=23, L=shape["L"], P=shape["P"])
    w.scheme = scheme
    comp = make_compactor(w)
    comp.compact(to_device(inp), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    n = W.to_numpy(inp)
    st, pool, tab = run_oracle(w, n)
    assert st == oracle.OK and np.array_equal(tab.classes, aim.reshape(-1))
    assert_same_state(fetch(comp), oracle_state(pool, tab))
    starts = np.concatenate([[0], np.cumsum(w.lens)])

    def where(pid, pos):
        u = int(pool.rev_unit[pid])
        h, r, l = u % w.Hkv, (u // w.Hkv) % w.R, u // (w.Hkv * w.R)
        return l, starts[r] + pos, h

    assert _check_bound(pool.pages, pool.page_cls, w.P, n["k"], n["v"], where, comp.pool, scheme) == int((aim > 0).sum())


@pytest.mark.parametrize("scheme", [1, 2])
def test_decode_steps_bit_exact(scheme):
    """Ordinary churn over several steps, with the free-list head wrapping."""
    w = W.small("sch_dec", lens=[300, 7, 517, 0, 129], scheme=scheme)
    used = int(HostDecode(w, cap=560, inp=W.make_inputs(w, 77)).pool.cursors[0])
    _run(w, cap=560, steps=10, p_prune=0.05, p_demote=0.08, F=used + 6, slot_check_every=5)


@pytest.mark.parametrize("scheme", [1, 2])
def test_decode_heavy_churn_bit_exact(scheme):
    w = W.small("sch_churn", lens=[700, 9, 520, 1, 333], L=2, Hq=8, Hkv=2, scheme=scheme)
    _run(w, cap=720, steps=4, p_prune=0.25, p_demote=0.35, slot_check_every=1)


@pytest.mark.parametrize("scheme", [1, 2])
def test_edge_rows_requantise_bit_exact(scheme):
    """Edge rows prefilled, then a few staged demotions, then every remaining
    high token demoted at once (past the job buffer: in-place requantiser),
    then prunes; new tokens are edge rows."""
    w, inp, aim = E.edge_batch([150, 37, 200], 4, 2, seed=35, L=1, P=16)
    w.scheme = scheme
    cap = 208
    hd = HostDecode(w, cap, inp=inp)
    dec = gpu_decoder(hd, inp)
    compare(gpu_state(dec), hd, "after prefill + index:")
    rng = np.random.default_rng(6)
    for step in range(3):
        held = (np.arange(cap)[None, :] < hd.ctx_lens[:, None]).reshape(1, -1, 1)
        hi = (hd.classes == 2) & held
        lo = (hd.classes == 1) & held
        demote = np.zeros_like(hi)
        prune = np.zeros_like(hi)
        if step == 0:
            demote.reshape(-1)[rng.permutation(np.flatnonzero(hi))[:40]] = True
        elif step == 1:
            demote = hi.copy()
        else:
            prune.reshape(-1)[rng.permutation(np.flatnonzero(lo))[:60]] = True
        upd = _edge_update(hd, step, demote, prune)
        d = {"k_new": upd["k_new"].cuda(), "v_new": upd["v_new"].cuda(), "sig_sum": hd.ctx["sig_sum"].cuda(),
             "sig_cnt": hd.ctx["sig_cnt"].cuda(), "ctx_lens": hd.ctx["ctx_lens"].cuda(),
             "new_lens": upd["new_lens"].cuda()}
        dec.step(d, w.alpha_h, w.alpha_l)
        st = libdkv.dkv_get_status(dec.pool)
        assert hd.step(upd) == oracle.OK
        assert st == libdkv.DKV_OK, libdkv.status_string(st)
        g = gpu_state(dec)
        compare(g, hd, f"step {step}:")
        check_slot_index(g, hd)
    check_state(w, cap, hd.pool, hd.tab.fwd, hd.tab.unit_hdr, hd.classes, hd.ctx_lens)
