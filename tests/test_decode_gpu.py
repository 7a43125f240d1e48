"""GPU parity of the generation step (dkv_decode_step, dkv_decode_index)
against the CPU oracle, bit-exact after every step: classes, unit headers,
forward rows, reverse tables, page classes, the free ring and its cursors,
and every byte of every owned page; plus the slot index the library keeps
(every held token's slot holds its position).

Inputs are drawn on the host (seeded), copied to the device, and fed to both
sides; the oracle never sees a value the GPU produced."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.decode_helpers import HostDecode, check_state
from tests.oracle_helpers import Layout

pytestmark = pytest.mark.gpu


def _dev(t):
    return t.to("cuda").contiguous()


def gpu_decoder(hd: HostDecode, inp_cpu: dict) -> libdkv.Decoder:
    """Device copy of the oracle's prefill: per-layer dkv_compact on the same
    inputs, then dkv_decode_index."""
    w = hd.w
    dec = libdkv.Decoder(w.L, w.R, w.Hq, w.Hkv, hd.cap, w.P, hd.pool.F, window=hd.window, mode=hd.mode,
                         scheme=w.scheme)
    for l in range(w.L):
        layer = {"L": 1, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T,
                 "k": _dev(inp_cpu["k"][l:l + 1]), "v": _dev(inp_cpu["v"][l:l + 1]),
                 "sig_sum": _dev(inp_cpu["sig_sum"][l:l + 1]), "sig_cnt": _dev(inp_cpu["sig_cnt"]),
                 "lens": _dev(inp_cpu["lens"])}
        dec.prefill_layer(layer, l, max(w.lens + [0]), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_OK
    dec.index(_dev(hd.ctx["ctx_lens"]))
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_OK
    return dec


def gpu_state(dec: libdkv.Decoder) -> dict:
    torch.cuda.synchronize()
    p = dec.pool
    return {"classes": dec.classes.cpu().numpy(), "slot_of": dec.slot_of.cpu().numpy(),
            "fwd": dec.tables.fwd.cpu().numpy(), "unit_hdr": dec.tables.unit_hdr.cpu().numpy(),
            "free_list": p.free_list.cpu().numpy(), "cursors": p.cursors.cpu().numpy().view(np.uint64),
            "rev_unit": p.rev_unit.cpu().numpy(), "rev_idx": p.rev_idx.cpu().numpy(),
            "page_cls": p.page_cls.cpu().numpy(), "pages": p.pages.cpu().numpy()}


def compare(g: dict, hd: HostDecode, what: str):
    o = hd.snapshot()
    for key in ("classes", "fwd", "unit_hdr", "cursors", "rev_unit", "rev_idx", "page_cls"):
        a, b = g[key].reshape(-1), o[key].reshape(-1)
        if not np.array_equal(a, b):
            bad = np.nonzero(a != b)[0]
            raise AssertionError(f"{what} {key}: {bad.size} mismatches at {bad[:5]}: gpu {a[bad[:5]]} "
                                 f"oracle {b[bad[:5]]}")
    # the free ring [head, tail)
    F = hd.pool.F
    head, tail = int(o["cursors"][0]), int(o["cursors"][1])
    ring = np.arange(head, tail) % F
    assert np.array_equal(g["free_list"][ring], o["free_list"][ring]), f"{what} free ring"
    live = np.nonzero(o["page_cls"] != 0)[0]
    if not np.array_equal(g["pages"][live], o["pages"][live]):
        bad = [int(i) for i in live if not np.array_equal(g["pages"][i], o["pages"][i])]
        raise AssertionError(f"{what} pages differ: {len(bad)} of {live.size}, first {bad[:5]}")


def check_slot_index(g: dict, hd: HostDecode):
    """slot_of of every held token points at the slot holding its position;
    -1 for pruned positions."""
    w, cap, P = hd.w, hd.cap, hd.w.P
    lay = Layout(P, w.scheme)
    cls = g["classes"].reshape(w.L, w.R * cap, w.Hkv)
    so = g["slot_of"].reshape(w.L, w.R * cap, w.Hkv)
    pages = g["pages"]
    for l in range(w.L):
        for r in range(w.R):
            c = int(hd.ctx_lens[r])
            for h in range(w.Hkv):
                u = (l * w.R + r) * w.Hkv + h
                n_hi, n_lo, p_hi, p_lo = (int(x) for x in g["unit_hdr"][u])
                fw = g["fwd"][u]
                for i in range(c):
                    k = int(cls[l, r * cap + i, h])
                    s = int(so[l, r * cap + i, h])
                    if k == 0:
                        assert s == -1, (u, i)
                        continue
                    per = P if k == 2 else 2 * P
                    pid = fw[(0 if k == 2 else p_hi) + s // per]
                    o = lay.pos + 4 * (s % per)
                    pos = pages[pid][o:o + 4].view(np.int32)[0]
                    assert pos == i, (u, i, s, pos)


def _run(w: W.Workload, cap: int, steps: int, p_prune: float, p_demote: float, F: int | None = None,
         slot_check_every: int = 5, window: int = 0, mode: int = 0):
    inp = W.make_inputs(w, 77)
    hd = HostDecode(w, cap, F=F, inp=inp, window=window, mode=mode)
    dec = gpu_decoder(hd, inp)
    g = gpu_state(dec)
    compare(g, hd, "after prefill + index:")
    check_slot_index(g, hd)
    heads = [int(hd.pool.cursors[0])]
    hd.held_changes = 0  # class changes of tokens held before their step
    for s in range(steps):
        held = (np.arange(cap)[None, :] < hd.ctx_lens[:, None]).reshape(-1)
        before = hd.classes.copy()
        upd = W.decode_update_inputs(w, hd.ctx, s, p_prune=p_prune, p_demote=p_demote)
        d = {"k_new": _dev(upd["k_new"]), "v_new": _dev(upd["v_new"]), "sig_sum": _dev(hd.ctx["sig_sum"]),
             "sig_cnt": _dev(hd.ctx["sig_cnt"]), "ctx_lens": _dev(hd.ctx["ctx_lens"]),
             "new_lens": _dev(upd["new_lens"])}
        dec.step(d, w.alpha_h, w.alpha_l)
        st = libdkv.dkv_get_status(dec.pool)
        assert hd.step(upd) == oracle.OK
        assert st == libdkv.DKV_OK, libdkv.status_string(st)
        hd.held_changes += int(((before != hd.classes) & held[None, :, None]).sum())
        g = gpu_state(dec)
        compare(g, hd, f"step {s}:")
        if s % slot_check_every == slot_check_every - 1 or s == steps - 1:
            check_slot_index(g, hd)
        heads.append(int(hd.pool.cursors[0]))
    check_state(w, cap, hd.pool, hd.tab.fwd, hd.tab.unit_hdr, hd.classes, hd.ctx_lens)
    return hd, dec, heads


def test_decode_small_ragged_with_wrap():
    w = W.small("dec", lens=[300, 7, 517, 0, 129])
    used = int(HostDecode(w, cap=560, inp=W.make_inputs(w, 77)).pool.cursors[0])  # pages the prefill takes
    # six spare pages: the head wraps within 24 steps and never runs dry
    hd, dec, heads = _run(w, cap=560, steps=24, p_prune=0.03, p_demote=0.03, F=used + 6)
    F = hd.pool.F
    assert heads[-1] // F > heads[0] // F, "free-list head did not wrap"


@pytest.mark.parametrize("shape", [
    dict(Hq=28, Hkv=4, P=32, lens=[1000, 33, 700], alpha_h=1.5, alpha_l=0.3, sigma=2.5),  # G = 7, scalar loads
    dict(Hq=16, Hkv=2, P=16, lens=[2100, 64], L=1),                                     # G = 8, two float4
    dict(Hq=4, Hkv=4, P=2, lens=[90, 91, 1], L=1),                                       # G = 1, tiny pages
    dict(Hq=4, Hkv=1, P=16, lens=[700, 130], L=1),                                       # G = 4, one row a thread
    dict(Hq=12, Hkv=3, P=16, lens=[400, 257, 1], L=1),                                   # G = 4, Hkv not 2^k
    dict(Hq=32, Hkv=8, P=16, lens=[600, 70, 333], L=2),                                  # G = 4, head pairs
])
def test_decode_shapes(shape):
    w = W.small("dec_shape", **shape)
    cap = -(-(max(w.lens) + 20) // 16) * 16
    _run(w, cap=cap, steps=12, p_prune=0.02, p_demote=0.04, slot_check_every=6)


def test_decode_low_churn_many_steps():
    """The decode workload's update rates (0.5% pruned, 0.5% demoted per
    step) over 40 steps on a small batch."""
    w = W.small("dec_slow", lens=[2048, 3000, 2500], L=1, Hq=8, Hkv=2)
    _run(w, cap=3072, steps=40, p_prune=0.005, p_demote=0.005, slot_check_every=20)


def _snap(dec):
    return gpu_state(dec)


def test_decode_errors_change_nothing():
    w = W.small("dec_err", lens=[300, 7, 517, 0, 129])
    inp = W.make_inputs(w, 77)
    hd = HostDecode(w, 560, inp=inp)
    dec = gpu_decoder(hd, inp)
    upd = W.decode_update_inputs(w, hd.ctx, 0, p_prune=0.05, p_demote=0.05)

    def d_of(**over):
        d = {"k_new": _dev(upd["k_new"]), "v_new": _dev(upd["v_new"]), "sig_sum": _dev(hd.ctx["sig_sum"]),
             "sig_cnt": _dev(hd.ctx["sig_cnt"]), "ctx_lens": _dev(hd.ctx["ctx_lens"]),
             "new_lens": _dev(upd["new_lens"])}
        d.update(over)
        return d

    before = _snap(dec)

    def same():
        after = _snap(dec)
        for k in before:
            assert np.array_equal(before[k], after[k]), k

    # RANGE: an infinite value in a kept new token
    kbad = upd["k_new"].clone()
    kbad[1, 2, 1, 7] = float("inf")
    sig = hd.ctx["sig_sum"].clone()
    n2 = int(hd.ctx["ctx_lens"][2])
    sig[1, 2 * 560 + n2] = 1.0
    dec.step(d_of(k_new=_dev(kbad), sig_sum=_dev(sig)), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_E_RANGE
    same()
    # LENS: a request past its capacity
    lens = hd.ctx["ctx_lens"].clone()
    lens[1] = 560
    dec.step(d_of(ctx_lens=_dev(lens)), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_E_LENS
    same()
    # NOMEM: no free pages left (head moved up to tail on the device)
    cur = dec.pool.cursors.clone()
    dec.pool.cursors[0] = dec.pool.cursors[1]
    before = _snap(dec)
    dec.step(d_of(), w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_E_NOMEM
    same()
    dec.pool.cursors.copy_(cur)
    # TIMEOUT: a look-back that may not wait (more than one scan partition)
    w2 = W.small("dec_to", lens=[40] * 70, L=2, Hq=8, Hkv=2)
    inp2 = W.make_inputs(w2, 3)
    hd2 = HostDecode(w2, 48, inp=inp2)
    dec2 = gpu_decoder(hd2, inp2)
    assert w2.U > 256
    upd2 = W.decode_update_inputs(w2, hd2.ctx, 0)
    d2 = {"k_new": _dev(upd2["k_new"]), "v_new": _dev(upd2["v_new"]), "sig_sum": _dev(hd2.ctx["sig_sum"]),
          "sig_cnt": _dev(hd2.ctx["sig_cnt"]), "ctx_lens": _dev(hd2.ctx["ctx_lens"]),
          "new_lens": _dev(upd2["new_lens"])}
    before2 = _snap(dec2)
    dec2.step(d2, w2.alpha_h, w2.alpha_l, spin_limit=0)
    assert libdkv.dkv_get_status(dec2.pool) == libdkv.DKV_E_TIMEOUT
    after2 = _snap(dec2)
    for k in before2:
        assert np.array_equal(before2[k], after2[k]), k
    # and the same step then succeeds and matches the oracle
    dec2.step(d2, w2.alpha_h, w2.alpha_l)
    assert libdkv.dkv_get_status(dec2.pool) == libdkv.DKV_OK
    assert hd2.step(upd2) == oracle.OK
    compare(gpu_state(dec2), hd2, "after timeout retry:")


def test_identity_step_on_device():
    """new_lens = 0 and unchanged scores: nothing changes on the device."""
    w = W.small("dec_id", lens=[300, 7, 517, 0, 129])
    inp = W.make_inputs(w, 77)
    hd = HostDecode(w, 560, inp=inp)
    dec = gpu_decoder(hd, inp)
    before = _snap(dec)
    z = torch.zeros((w.L, w.R, w.Hkv, 128), dtype=torch.bfloat16, device="cuda")
    d = {"k_new": z, "v_new": z, "sig_sum": _dev(hd.ctx["sig_sum"]), "sig_cnt": _dev(hd.ctx["sig_cnt"]),
         "ctx_lens": _dev(hd.ctx["ctx_lens"]), "new_lens": torch.zeros(w.R, dtype=torch.int32, device="cuda")}
    dec.step(d, w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_OK
    after = _snap(dec)
    for k in before:
        assert np.array_equal(before[k], after[k]), k


@pytest.mark.parametrize("p_prune,p_demote", [(0.25, 0.35), (0.6, 0.3)])
def test_decode_heavy_churn(p_prune, p_demote):
    """Most of a unit's tokens change class in one step: the per-unit mark
    lists overflow into the in-place path, demotions run to several batches
    of 32, and lists shrink by many pages at once."""
    w = W.small("dec_churn", lens=[700, 9, 520, 1, 333], L=2, Hq=8, Hkv=2)
    _run(w, cap=720, steps=6, p_prune=p_prune, p_demote=p_demote, slot_check_every=1)


def test_decode_zero_low_threshold():
    """alpha_l = 0: nothing is pruned by score and the threshold test takes the
    IEEE division for every row."""
    w = W.small("dec_a0", lens=[300, 77, 5], L=1, Hq=8, Hkv=2, alpha_h=0.7, alpha_l=0.0)
    _run(w, cap=320, steps=5, p_prune=0.05, p_demote=0.1, slot_check_every=5)


@pytest.mark.parametrize("window,mode", [(0, 1), (3, 0), (3, 1), (64, 0), (64, 1), (600, 0), (600, 1)])
def test_decode_recent_window_and_candidate(window, mode):
    """Recent window W and the single-candidate policy (mode 1): same bytes as
    the oracle after every step.  Heavy churn so that candidates do change;
    request lengths below, at and above W; W = 600 covers every request, so
    in either mode nothing held changes class (in mode 1 no candidate leaves
    the window)."""
    w = W.small("decw", lens=[300, 7, 517, 0, 129, 64, 3])
    hd, dec, _ = _run(w, cap=560, steps=10, p_prune=0.3, p_demote=0.3, window=window, mode=mode)
    if window == 600 or (window == 0 and mode == 1):
        assert hd.held_changes == 0  # every token in the window; or only new tokens classified
    else:
        assert hd.held_changes > 0, "no held token changed class: the case tests nothing"
