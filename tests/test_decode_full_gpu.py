"""GPU parity of the generation step at the full decode workload: 32 layers,
256 requests holding 2048..8192 tokens, 100 steps, the free ring wrapping.

The library runs the whole workload in one pool.  The CPU oracle replays
sampled units (2 layers x 3 requests x 8 KV heads) in a pool of their own,
fed with the same bytes: the prefill inputs of those requests and, every
step, their significance rows, counts and new tokens copied from the device.
Page ids differ between the two pools, so the comparison is per unit: the
header, every byte of every slot of both lists in list order, and the
classes, bit-exact.  Every unit of the library's state is checked against
the invariants the oracle's pins establish: headers match the classes,
page counts are ceil(n / capacity), forward and reverse tables agree, owned
pages and the free ring partition the pool, and the slot index points at
each held token's slot."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import decode_setup as DS
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.decode_helpers import HostDecode, list_slots

pytestmark = pytest.mark.gpu

SAMPLE_LAYERS = (0, 31)
SAMPLE_REQS = (0, 128, 255)
SEED = W.SEED_BASE + 5


def _token_rows(w: W.Workload, reqs) -> torch.Tensor:
    starts = np.concatenate([[0], np.cumsum(w.lens)[:-1]])
    return torch.cat([torch.arange(int(starts[r]), int(starts[r]) + w.lens[r]) for r in reqs])


def _replicas(w: W.Workload, cap: int, dev) -> dict:
    """One oracle state per sampled layer, prefilled with the same bytes the
    library's prefill of that layer read."""
    ws = dataclasses.replace(w, L=1, lens=[w.lens[r] for r in SAMPLE_REQS])
    rows = _token_rows(w, SAMPLE_REQS).to(dev)
    out = {}
    for l in SAMPLE_LAYERS:
        inp = {"L": 1, "R": ws.R, "Hq": w.Hq, "Hkv": w.Hkv, "T": ws.T,
               "k": W.make_kv_layer(w, SEED, l, 0, dev)[rows][None].cpu(),
               "v": W.make_kv_layer(w, SEED, l, 1, dev)[rows][None].cpu(),
               "sig_sum": W.make_sig_layer(w, SEED, l, dev)[rows][None].cpu(),
               "sig_cnt": W.sig_cnt_prefill(ws), "lens": torch.tensor(ws.lens, dtype=torch.int32)}
        out[l] = HostDecode(ws, cap, F=ws.pool_pages, inp=inp)
    return out


def _feed(hd: HostDecode, l: int, ctx: dict, upd: dict, cap: int):
    """The sampled requests' rows of this step's device inputs, for the oracle."""
    R, Hq = ctx["R"], ctx["Hq"]
    idx = torch.tensor(SAMPLE_REQS, device=ctx["sig_sum"].device)
    hd.ctx["sig_sum"][0].view(len(SAMPLE_REQS), cap, Hq).copy_(ctx["sig_sum"][l].view(R, cap, Hq)[idx].cpu())
    hd.ctx["sig_cnt"].view(len(SAMPLE_REQS), cap).copy_(ctx["sig_cnt"].view(R, cap)[idx].cpu())
    assert torch.equal(hd.ctx["ctx_lens"], ctx["ctx_lens"][idx].cpu())
    return {"k_new": upd["k_new"][l:l + 1, idx].cpu(), "v_new": upd["v_new"][l:l + 1, idx].cpu(),
            "new_lens": upd["new_lens"][idx].cpu()}


def _compare(dec: libdkv.Decoder, reps: dict, w: W.Workload, cap: int, step: int):
    hdr = dec.tables.unit_hdr
    for l, hd in reps.items():
        for j, r in enumerate(SAMPLE_REQS):
            for h in range(w.Hkv):
                u = (l * w.R + r) * w.Hkv + h
                uo = j * w.Hkv + h
                gh = hdr[u].cpu().numpy()
                assert np.array_equal(gh, hd.tab.unit_hdr[uo]), (step, l, r, h, gh, hd.tab.unit_hdr[uo])
                nt = int(gh[2] + gh[3])
                ids = dec.tables.fwd[u, :nt].long()
                gp = dec.pool.pages[ids].cpu().numpy()
                local = np.arange(nt, dtype=np.int32)
                got = list_slots(gp, local, gh, w.P)
                want = list_slots(hd.pool.pages, hd.tab.fwd[uo], hd.tab.unit_hdr[uo], w.P)
                assert got == want, (step, l, r, h)
                n = int(hd.ctx_lens[j])
                gc = dec.classes.view(w.L, w.R, cap, w.Hkv)[l, r, :n, h].cpu().numpy()
                oc = hd.classes[0, j * cap:j * cap + n, h]
                assert np.array_equal(gc, oc), (step, l, r, h)


def _invariants(dec: libdkv.Decoder, w: W.Workload, cap: int, ctx_lens: torch.Tensor):
    """Every unit of the library's state, on the device."""
    P, F, U, pmax = w.P, dec.pool.F, w.U, dec.pmax
    hdr = dec.tables.unit_hdr.long()
    fwd = dec.tables.fwd.long()
    assert torch.equal(hdr[:, 2], (hdr[:, 0] + P - 1) // P)
    assert torch.equal(hdr[:, 3], (hdr[:, 1] + 2 * P - 1) // (2 * P))
    tot = hdr[:, 2] + hdr[:, 3]
    k = torch.arange(pmax, device=fwd.device)[None, :]
    live = k < tot[:, None]
    assert bool((fwd[~live] == -1).all())
    ids = fwd[live]
    assert bool(((ids >= 0) & (ids < F)).all())
    units = torch.arange(U, device=fwd.device)[:, None].expand(U, pmax)[live]
    assert torch.equal(dec.pool.rev_unit.long()[ids], units)
    assert torch.equal(dec.pool.rev_idx.long()[ids], k.expand(U, pmax)[live])
    want_cls = torch.where(k.expand(U, pmax) < hdr[:, 2:3], 2, 1)[live]
    assert torch.equal(dec.pool.page_cls.long()[ids], want_cls)
    cur = dec.pool.cursors.cpu().numpy().view(np.uint64)
    head, tail = int(cur[0]), int(cur[1])
    ring = dec.pool.free_list.long()[torch.arange(head, tail, device=fwd.device) % F]
    seen = torch.bincount(torch.cat([ids, ring]), minlength=F)
    assert bool((seen == 1).all()), "owned pages and the free ring must partition the pool"
    # headers against the classes of held positions; the slot index per layer
    cls = dec.classes.view(w.L, w.R, cap, w.Hkv)
    held = torch.arange(cap, device=fwd.device)[None, :] < ctx_lens.long()[:, None]  # [R, cap]
    so = dec.slot_of.view(w.L, w.R, cap, w.Hkv)
    pb = 216 * P
    flat = dec.pool.pages.view(-1)
    for l in range(w.L):
        c = cls[l]
        n_hi = ((c == 2) & held[:, :, None]).sum(1).reshape(-1)
        n_lo = ((c == 1) & held[:, :, None]).sum(1).reshape(-1)
        hl = hdr[l * w.R * w.Hkv:(l + 1) * w.R * w.Hkv]
        assert torch.equal(n_hi, hl[:, 0]) and torch.equal(n_lo, hl[:, 1]), l
        m = (c > 0) & held[:, :, None]
        r_i, i_i, h_i = torch.nonzero(m, as_tuple=True)
        s = so[l][m].long()
        cc = c[m].long()
        u = (l * w.R + r_i) * w.Hkv + h_i
        per = torch.where(cc == 2, P, 2 * P)
        kidx = torch.where(cc == 2, 0, hdr[u, 2]) + s // per
        assert bool((s >= 0).all())
        pid = fwd[u, kidx]
        off = pid * pb + 208 * P + 4 * (s % per)
        pos = (flat[off].long() | (flat[off + 1].long() << 8) | (flat[off + 2].long() << 16)
               | (flat[off + 3].long() << 24))
        assert torch.equal(pos, i_i), l
        assert bool((so[l][(c == 0) & held[:, :, None]] == -1).all()), l


def test_decode_workload_full_size():
    w = W.get("decode")
    steps = int(w.extra["steps"])
    dev = torch.device("cuda", 0)
    dec, ctx, cap, used = DS.decode_setup(w, dev, SEED, steps + 1)
    F = dec.pool.F
    head0 = int(dec.pool.cursors[0])
    reps = _replicas(w, cap, dev)
    _compare(dec, reps, w, cap, -1)
    for s in range(steps):
        upd = W.decode_update_inputs(w, ctx, s, device=dev)
        d = {"k_new": upd["k_new"], "v_new": upd["v_new"], "sig_sum": ctx["sig_sum"], "sig_cnt": ctx["sig_cnt"],
             "ctx_lens": ctx["ctx_lens"], "new_lens": upd["new_lens"]}
        dec.step(d, w.alpha_h, w.alpha_l)
        for l, hd in reps.items():
            assert hd.step(_feed(hd, l, ctx, upd, cap)) == oracle.OK
        st = libdkv.dkv_get_status(dec.pool)
        assert st == libdkv.DKV_OK, libdkv.status_string(st)
        ctx["ctx_lens"] += upd["new_lens"]
        if s % 10 == 9:
            _compare(dec, reps, w, cap, s)
    _invariants(dec, w, cap, ctx["ctx_lens"])
    assert int(dec.pool.cursors[0]) // F > head0 // F, "the free ring's head did not wrap"
