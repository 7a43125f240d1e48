"""GPU parity of every quantiser on hand-built edge rows (tests/edge_rows.py),
through the C ABI, byte for byte against the CPU oracle:

  - k_pack (prefill compaction) at both classes: exact-grid rows whose every
    element is a tie at 8, 4 and 2 bits, rows one bf16 ulp off the ties,
    constant rows (scale 0), spans that underflow binary16, subnormal scales
    whose top codes clamp, subnormal minima that binary16 rounds, rows
    reaching +-65280 and rows whose extremes are -0 and +0;
  - the generation step's three requantisers on the same rows: k_demote
    (staged demotions), the in-place requantiser of k_apply (a step that
    demotes more tokens than the job buffer holds) and the new-token
    quantiser of k_apply;
and every dequantised value within the error bound derived from the fp32
arithmetic (tests/edge_rows.dequant_bound, with the slot's own scale)."""
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
from tests.oracle_helpers import Layout, bf16_to_f32, f16, run_oracle
from tests.test_decode_gpu import check_slot_index, compare, gpu_decoder, gpu_state

pytestmark = pytest.mark.gpu


def _check_bound(pages: np.ndarray, page_cls: np.ndarray, P: int, k_in: np.ndarray, v_in: np.ndarray,
                 where, comp_pool, scheme: int = 0):
    """Dequantise every live page on the GPU and hold each element to the
    bound with the slot's own scale.  where(page, pos) -> (layer, token row,
    head) of the input row."""
    lay = Layout(P, scheme)
    live = np.nonzero(page_cls)[0]
    k, v, pos = libdkv.dkv_dequant_pages(comp_pool, torch.tensor(live, dtype=torch.int32))
    k, v, pos = k.cpu().numpy(), v.cpu().numpy(), pos.cpu().numpy()
    checked = 0
    for i, pid in enumerate(live):
        high = page_cls[pid] == 2
        meta = pages[pid][lay.meta:lay.pos].view(np.uint16).reshape(2 * P, 4)
        for s in np.nonzero(pos[i] >= 0)[0]:
            l, t, h = where(int(pid), int(pos[i][s]))
            ms = f16(meta[s]).astype(np.float64)
            for x_bits, xq, sc, nb in ((k_in[l, t, h], k[i][s], ms[0], lay.kbits(high)),
                                       (v_in[l, t, h], v[i][s], ms[2], lay.vbits(high))):
                x = bf16_to_f32(x_bits).astype(np.float64)
                bound = E.dequant_bound(sc, nb, x.max() - x.min())
                assert np.all(np.abs(x - xq.astype(np.float64)) <= bound), (pid, s)
            checked += 1
    return checked


@pytest.mark.parametrize("shape", [
    dict(lens=[150, 37, 200], Hq=4, Hkv=2, L=2, P=16),
    dict(lens=[129, 1, 64], Hq=8, Hkv=1, L=1, P=2),
    dict(lens=[300], Hq=7, Hkv=7, L=1, P=32),
])
def test_edge_rows_prefill_bit_exact(shape):
    w, inp, aim = E.edge_batch(shape["lens"], shape["Hq"], shape["Hkv"], seed=21, L=shape["L"], P=shape["P"])
    comp = make_compactor(w)
    comp.compact(to_device(inp), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    n = W.to_numpy(inp)
    st, pool, tab = run_oracle(w, n)
    assert st == oracle.OK
    assert np.array_equal(tab.classes, aim.reshape(-1))  # the rows landed in the intended classes
    assert_same_state(fetch(comp), oracle_state(pool, tab))
    starts = np.concatenate([[0], np.cumsum(w.lens)])

    def where(pid, pos):
        u = int(pool.rev_unit[pid])
        h, r, l = u % w.Hkv, (u // w.Hkv) % w.R, u // (w.Hkv * w.R)
        return l, starts[r] + pos, h

    assert _check_bound(pool.pages, pool.page_cls, w.P, n["k"], n["v"], where, comp.pool) == int((aim > 0).sum())


def _edge_update(hd: HostDecode, step: int, demote: np.ndarray, prune: np.ndarray):
    """This step's significance update on hd.ctx (in place) and its new
    tokens.  Held rows marked in `demote` move to the middle tier, rows in
    `prune` to zero, the rest keep their average; every count grows by one.
    The new token of each (request, KV head) gets a score of 4/N, 0.5/N or
    0.02/N and K / V from the edge rows."""
    w, cap = hd.w, hd.cap
    G = w.Hq // w.Hkv
    rng = np.random.default_rng(1000 + step)
    clen = hd.ctx["ctx_lens"].to(torch.int64)
    N = (clen + 1).to(torch.float32)
    sig = hd.ctx["sig_sum"].view(w.L, w.R, cap, w.Hkv, G)
    cnt = hd.ctx["sig_cnt"].view(w.R, cap)
    cntf = cnt.to(torch.float32)[None, :, :, None, None]
    mid = (torch.tensor(W.ALPHA_MID, dtype=torch.float32) / N)[None, :, None, None, None]
    dm = torch.from_numpy(demote.reshape(w.L, w.R, cap, w.Hkv))[..., None]
    pm = torch.from_numpy(prune.reshape(w.L, w.R, cap, w.Hkv))[..., None]
    held = (torch.arange(cap)[None, :] < clen[:, None])[None, :, :, None, None]
    upd = torch.where(pm, torch.zeros_like(sig), torch.where(dm, mid * cntf, sig + sig / cntf))
    sig.copy_(torch.where(held, upd, sig))
    cnt[held[0, :, :, 0, 0]] += 1
    room = clen < cap
    level = torch.from_numpy(rng.choice([4.0, 0.5, 0.02], size=(w.L, w.R, w.Hkv)).astype(np.float32))
    for r in range(w.R):
        if room[r]:
            p = int(clen[r])
            sig[:, r, p] = (level[:, r] / N[r])[:, :, None].expand(w.L, w.Hkv, G)
            cnt[r, p] = 1
    k_new, v_new = E.new_token_rows(w.L, w.R, w.Hkv, seed=2000 + step)
    return {"k_new": k_new, "v_new": v_new, "new_lens": room.to(torch.int32)}


def test_edge_rows_requantise_bit_exact():
    """Prefill edge rows, then three generation steps: a few demotions (all
    staged for k_demote), then every remaining K8V4 token demoted at once
    (more than the job buffer holds: the rest requantise in place in
    k_apply), then prunes.  New tokens are edge rows of both classes."""
    w, inp, aim = E.edge_batch([150, 37, 200], 4, 2, seed=33, L=1, P=16)
    cap = 208
    hd = HostDecode(w, cap, inp=inp)
    dec = gpu_decoder(hd, inp)
    g = gpu_state(dec)
    compare(g, hd, "after prefill + index:")
    njobs = (w.L * w.R * cap * w.Hkv) // 16 + 64   # the job buffer of this shape (one held row in 16, + 64)
    rng = np.random.default_rng(5)
    for step in range(3):
        held = (np.arange(cap)[None, :] < hd.ctx_lens[:, None]).reshape(1, -1, 1)
        hi = (hd.classes == 2) & held
        lo = (hd.classes == 1) & held
        demote = np.zeros_like(hi)
        prune = np.zeros_like(hi)
        if step == 0:
            pick = rng.permutation(np.flatnonzero(hi))[:40]
            demote.reshape(-1)[pick] = True
        elif step == 1:
            demote = hi.copy()
            assert demote.sum() > njobs + 64, "too few demotions to overflow the job buffer"
        else:
            pick = rng.permutation(np.flatnonzero(lo))[:60]
            prune.reshape(-1)[pick] = True
        upd = _edge_update(hd, step, demote, prune)
        d = {"k_new": upd["k_new"].cuda(), "v_new": upd["v_new"].cuda(), "sig_sum": hd.ctx["sig_sum"].cuda(),
             "sig_cnt": hd.ctx["sig_cnt"].cuda(), "ctx_lens": hd.ctx["ctx_lens"].cuda(),
             "new_lens": upd["new_lens"].cuda()}
        dec.step(d, w.alpha_h, w.alpha_l)
        st = libdkv.dkv_get_status(dec.pool)
        before = hd.classes.copy()
        assert hd.step(upd) == oracle.OK
        assert st == libdkv.DKV_OK, libdkv.status_string(st)
        if step < 2:
            assert int(((before == 2) & (hd.classes == 1) & held).sum()) == int(demote.sum())
        g = gpu_state(dec)
        compare(g, hd, f"step {step}:")
        check_slot_index(g, hd)
    check_state(w, cap, hd.pool, hd.tab.fwd, hd.tab.unit_hdr, hd.classes, hd.ctx_lens)
