"""Pins for the oracle's generation (decode) step, CPU only.

Each test ties the decode step to something other than itself: the prefill
compaction it must reduce to (itself pinned in test_oracle_pins), the
identity of a step that changes nothing, the byte-for-byte preservation of
tokens a step does not touch, the textbook quantiser on exactly representable
rows, error bounds, and the pool / table invariants.

Source: DiffKV (arXiv 2412.03131), Pith review page: "Core claim" (K8V4 /
K4V2 / pruned; unified pages; circular free page list; bidirectional page
table), Referee Report, major comment 2 (Algorithm 1 classifies tokens as they
age in the generation phase; demotion and pruning are irreversible).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.decode_helpers import HostDecode, check_state, decode_pmax, list_slots, slot_codes
from tests.oracle_helpers import bf16_to_f32, f16


def _small(**kw):
    base = dict(lens=[300, 7, 517, 0, 129])
    base.update(kw)
    return W.small("dec", **base)


def _state(hd: HostDecode):
    return check_state(hd.w, hd.cap, hd.pool, hd.tab.fwd, hd.tab.unit_hdr, hd.classes, hd.ctx_lens)


def test_step_without_changes_is_identity():
    """No new tokens and unchanged scores: classify(s, N) with the prefill's N
    gives the prefill's classes back, so nothing moves.  Then a new token with
    zero attention (pruned) and scores re-averaged over N + 1: thresholds only
    fall, classes never rise, so again every byte stays."""
    w = _small()
    hd = HostDecode(w, cap=560)
    snap = hd.snapshot()
    L, R, Hkv = w.L, w.R, w.Hkv
    zero_kv = torch.zeros((L, R, Hkv, 128), dtype=torch.bfloat16)
    st = hd.step({"k_new": zero_kv, "v_new": zero_kv, "new_lens": torch.zeros(R, dtype=torch.int32)})
    assert st == oracle.OK
    after = hd.snapshot()
    for k in snap:
        assert np.array_equal(snap[k], after[k]), k
    # a pruned new token: sig 0 at the new position, counts + 1 elsewhere with
    # the same average
    ctx = hd.ctx
    lens = ctx["ctx_lens"].to(torch.int64)
    for r in range(R):
        c = int(lens[r])
        sl = slice(r * hd.cap, r * hd.cap + c)
        cnt = ctx["sig_cnt"][sl].to(torch.float32)
        ctx["sig_sum"][:, sl] = ctx["sig_sum"][:, sl] + ctx["sig_sum"][:, sl] / cnt[None, :, None]
        ctx["sig_cnt"][sl] += 1
        ctx["sig_sum"][:, r * hd.cap + c] = 0.0
        ctx["sig_cnt"][r * hd.cap + c] = 1
    st = hd.step({"k_new": zero_kv, "v_new": zero_kv, "new_lens": torch.ones(R, dtype=torch.int32)})
    assert st == oracle.OK
    after = hd.snapshot()
    for k in snap:
        assert np.array_equal(snap[k], after[k]), k


def _stable_inputs(w1: W.Workload, seed: int):
    """Inputs of w1 whose scores are 5/N, 0.5/N or 0.01/N per (layer, token,
    KV head) with N = the request length minus one: far enough from the
    thresholds that the classes at N and N + 1 agree."""
    inp = W.make_inputs(w1, seed)
    g = torch.Generator().manual_seed(seed)
    G = w1.Hq // w1.Hkv
    pick = torch.randint(0, 3, (w1.L, w1.T, w1.Hkv), generator=g)
    level = torch.tensor([5.0, 0.5, 0.01], dtype=torch.float64)[pick]
    lens = torch.tensor(w1.lens, dtype=torch.int64)
    req, pos = W._positions(w1, "cpu")
    n0 = (lens[req] - 1).clamp(min=1).to(torch.float64)
    score = (level / n0[None, :, None]).repeat_interleave(G, dim=2)
    return inp, score


def test_append_reduces_to_prefill():
    """Prefill of N tokens then one decode step that appends token N (classes
    stable) equals a prefill of N + 1 tokens: the same unit headers and the
    same bytes in every slot of every list page (pages compared by list index,
    since page ids differ).  Covers page-boundary crossings in both lists."""
    seed = 123
    lens1 = [33, 1, 64, 17, 65, 32]
    w1 = _small(lens=lens1, L=2)
    inp1, score = _stable_inputs(w1, seed)
    cnt1 = W.sig_cnt_prefill(w1)
    inp1["sig_sum"] = (score * cnt1.to(torch.float64)[None, :, None]).to(torch.float32)
    # the N-token prefix of every request
    keep = torch.ones(w1.T, dtype=torch.bool)
    ends = torch.cumsum(torch.tensor(lens1), 0) - 1
    keep[ends] = False
    w0 = _small(lens=[n - 1 for n in lens1], L=2)
    cnt0 = W.sig_cnt_prefill(w0)
    inp0 = {"L": 2, "R": w0.R, "Hq": w0.Hq, "Hkv": w0.Hkv, "T": w0.T, "k": inp1["k"][:, keep],
            "v": inp1["v"][:, keep], "sig_cnt": cnt0, "lens": torch.tensor(w0.lens, dtype=torch.int32),
            "sig_sum": (score[:, keep] * cnt0.to(torch.float64)[None, :, None]).to(torch.float32)}
    cap = 80
    hd = HostDecode(w0, cap, F=4096, inp=inp0)
    # the decode step: context counts + 1, scores unchanged; new token = row N
    req, pos = W._positions(w1, "cpu")
    ctx = hd.ctx
    dst1 = req * cap + pos
    ctx["sig_sum"][:, dst1] = inp1["sig_sum"]
    ctx["sig_cnt"][dst1] = cnt1
    k_new = inp1["k"][:, ends].contiguous()
    v_new = inp1["v"][:, ends].contiguous()
    st = hd.step({"k_new": k_new, "v_new": v_new, "new_lens": torch.ones(w0.R, dtype=torch.int32)})
    assert st == oracle.OK
    pool1 = oracle.Pool(4096, w1.P)
    tab1 = oracle.Tables(w1.U, decode_pmax(cap, w1.P), w1.rows)
    assert oracle.compact(W.to_numpy(inp1), w1.alpha_h, w1.alpha_l, pool1, tab1) == oracle.OK
    assert np.array_equal(hd.tab.unit_hdr, tab1.unit_hdr)
    for u in range(w1.U):
        a = list_slots(hd.pool.pages, hd.tab.fwd[u], hd.tab.unit_hdr[u], w1.P)
        b = list_slots(pool1.pages, tab1.fwd[u], tab1.unit_hdr[u], w1.P)
        assert a == b, u
    cls1 = tab1.classes.reshape(w1.L, w1.T, w1.Hkv)
    assert np.array_equal(hd.classes[:, dst1.numpy()], cls1)
    _state(hd)


def _churn(hd: HostDecode, steps: int, p_prune: float, p_demote: float, track_prefill: dict):
    """Run steps, checking the invariants and that tokens keep their bytes."""
    w = hd.w
    for _ in range(steps):
        before = hd.classes.copy()
        assert hd.step(p_prune=p_prune, p_demote=p_demote) == oracle.OK
        cls = hd.classes
        # classes never rise and only change where the scores say so
        live = np.zeros_like(cls, dtype=bool)
        for r in range(w.R):
            live[:, r * hd.cap:r * hd.cap + int(hd.ctx_lens[r]) - 1] = True
        assert np.all(cls[live] <= before[live])
        where = _state(hd)
        for (u, p), (li, raw, _) in where.items():
            if (u, p) in track_prefill and track_prefill[(u, p)][0] == li:
                assert track_prefill[(u, p)][1] == raw, (u, p)
    return where


def test_untouched_tokens_keep_their_bytes_and_pool_wraps():
    """Twenty steps with 3% pruning and 3% demotion per step on a pool small
    enough that the free-list head wraps: after every step the invariants
    hold, a token still in its prefill class keeps its prefill bytes exactly
    (moves copy bytes), and no class ever rises."""
    w = _small()
    used = int(HostDecode(w, cap=560).pool.cursors[0])  # pages the prefill takes
    F = used + 12
    hd = HostDecode(w, cap=560, F=F)
    where0 = _state(hd)
    head0 = int(hd.pool.cursors[0])
    where = _churn(hd, 20, 0.03, 0.03, where0)
    assert int(hd.pool.cursors[0]) // F > head0 // F, "free-list head did not wrap"
    assert any(li == 1 and (u, p) in where0 and where0[(u, p)][0] == 0 for (u, p), (li, _, _) in where.items()), \
        "no demoted token survived"


def test_hole_fill_keeps_low_slots_in_place():
    """Reading of the hole-fill: a surviving token whose slot is below the
    number of survivors stays where it was; only tokens from the tail move,
    and tokens appended this step come after every survivor."""
    w = _small()
    hd = HostDecode(w, cap=560)
    for _ in range(5):
        prev = {}
        for u in range(w.U):
            for li, slots in enumerate(list_slots(hd.pool.pages, hd.tab.fwd[u], hd.tab.unit_hdr[u], w.P)):
                for si, s in enumerate(slots):
                    if s[3] >= 0:
                        prev[(u, li, s[3])] = si
        assert hd.step(p_prune=0.05, p_demote=0.05) == oracle.OK
        for u in range(w.U):
            hdr = hd.tab.unit_hdr[u]
            for li, slots in enumerate(list_slots(hd.pool.pages, hd.tab.fwd[u], hdr, w.P)):
                n = int(hdr[li])
                # survivors of the old list; the appended tokens come after them
                keep = sum(1 for s in slots[:n] if (u, li, s[3]) in prev)
                for si, s in enumerate(slots[:n]):
                    old = prev.get((u, li, s[3]))
                    if old is not None:
                        assert si < keep
                        if old < keep:
                            assert old == si, (u, li, s[3])


def test_demoted_codes_on_exact_grid_equal_the_textbook_quantiser():
    """Rows whose K8V4 codes dequantise exactly (K integers 0..255, V integers
    0..15): after demotion the K4V2 codes must equal the 4-bit / 2-bit
    quantisation of the original bf16 rows, and the demoted tokens must sit in
    the K4V2 list after its survivors in ascending position order."""
    w = _small(lens=[70, 40], L=1, Hq=4, Hkv=2, n_outlier=0)
    inp = W.make_inputs(w, 5)
    g = torch.Generator().manual_seed(9)
    kk = torch.stack([torch.randperm(256, generator=g)[:128] for _ in range(w.T * w.Hkv)]).to(torch.float32)
    vv = torch.randint(0, 16, (w.T * w.Hkv, 128), generator=g).to(torch.float32)
    vv[:, 0], vv[:, 1] = 0.0, 15.0
    kk[:, 0], kk[:, 1] = 0.0, 255.0
    inp["k"] = kk.view(1, w.T, w.Hkv, 128).to(torch.bfloat16)
    inp["v"] = vv.view(1, w.T, w.Hkv, 128).to(torch.bfloat16)
    # everything K8V4 at prefill
    inp["sig_sum"] = (inp["sig_cnt"].to(torch.float32) * 10.0 / 70)[None, :, None].expand(1, w.T, w.Hq).contiguous()
    hd = HostDecode(w, cap=96, inp=inp)
    assert np.all(hd.tab.unit_hdr[:, 1] == 0)
    upd = W.decode_update_inputs(w, hd.ctx, 0, p_prune=0.0, p_demote=0.2)
    assert hd.step(upd) == oracle.OK
    kb = inp["k"].view(torch.int16).numpy().view(np.uint16)
    vb = inp["v"].view(torch.int16).numpy().view(np.uint16)
    seen = 0
    for u in range(w.U):
        r, h = u // w.Hkv, u % w.Hkv
        tok0 = sum(w.lens[:r])
        hdr = hd.tab.unit_hdr[u]
        low = list_slots(hd.pool.pages, hd.tab.fwd[u], hdr, w.P)[1][:int(hdr[1])]
        positions = [s[3] for s in low]
        assert positions == sorted(positions)  # all demoted this step: ascending position
        for s in low:
            kq, vq, meta = slot_codes(s[:3], high=False)
            st, k4, ks, kz = oracle.quant_row(kb[0, tok0 + s[3], h], 4)
            st2, v2, vs, vz = oracle.quant_row(vb[0, tok0 + s[3], h], 2)
            assert st == st2 == oracle.OK
            assert np.array_equal(kq, k4) and np.array_equal(vq, v2)
            assert list(meta) == [ks, kz, vs, vz]
            seen += 1
    assert seen > 5


def test_demoted_values_within_the_requantisation_bound():
    """Random rows: a demoted token's K4V2 dequantised values are within
    0.5 * s + |mn - z| + max(0, (mx - mn) - n * s) (+ fp32 rounding) of its
    K8V4 dequantised values, the bound of a min/max quantiser whose zero and
    scale were rounded to fp16."""
    w = _small(lens=[200, 90], L=1)
    hd = HostDecode(w, cap=256)
    high_before = {}
    for u in range(w.U):
        hdr = hd.tab.unit_hdr[u]
        for s in list_slots(hd.pool.pages, hd.tab.fwd[u], hdr, w.P)[0][:int(hdr[0])]:
            high_before[(u, s[3])] = s[:3]
    assert hd.step(p_prune=0.0, p_demote=0.3) == oracle.OK
    checked = 0
    for u in range(w.U):
        hdr = hd.tab.unit_hdr[u]
        for s in list_slots(hd.pool.pages, hd.tab.fwd[u], hdr, w.P)[1][:int(hdr[1])]:
            if (u, s[3]) not in high_before:
                continue
            k8, v8, m8 = slot_codes(high_before[(u, s[3])], high=True)
            k4, v2, m4 = slot_codes(s[:3], high=False)
            for q8, sc8, zc8, q4, sc4, zc4, n in ((k8, m8[0], m8[1], k4, m4[0], m4[1], 15),
                                                  (v8, m8[2], m8[3], v2, m4[2], m4[3], 3)):
                x = q8.astype(np.float64) * f16(sc8) + f16(zc8)
                y = q4.astype(np.float64) * f16(sc4) + f16(zc4)
                s4, z4 = float(f16(sc4)), float(f16(zc4))
                mn, mx = x.min(), x.max()
                bound = 0.5 * s4 + abs(mn - z4) + max(0.0, (mx - mn) - n * s4) + 1e-6 * (1 + abs(x).max())
                assert np.all(np.abs(x - y) <= bound), (u, s[3])
            checked += 1
    assert checked > 20


def test_nomem_and_range_are_all_or_nothing():
    w = _small()
    hd = HostDecode(w, cap=560)
    # exhaust the ring: head = tail
    hd.pool.cursors[0] = hd.pool.cursors[1]
    snap = hd.snapshot()
    st = hd.step(p_prune=0.0, p_demote=0.0)
    assert st == oracle.E_NOMEM
    after = hd.snapshot()
    for k in snap:
        assert np.array_equal(snap[k], after[k]), k
    hd2 = HostDecode(w, cap=560)
    snap = hd2.snapshot()
    upd = W.decode_update_inputs(w, hd2.ctx, 0)
    upd["k_new"][0, 2, 1, 5] = float("inf")
    n_new = hd2.ctx["ctx_lens"][2].item()
    hd2.ctx["sig_sum"][0, 2 * 560 + n_new] = 1.0  # the new token is kept
    assert hd2.step(upd) == oracle.E_RANGE
    after = hd2.snapshot()
    for k in snap:
        assert np.array_equal(snap[k], after[k]), k


def test_length_errors():
    w = _small()
    hd = HostDecode(w, cap=517)  # request 2 already fills its capacity
    upd = W.decode_update_inputs(w, hd.ctx, 0)
    assert int(upd["new_lens"][2]) == 0
    upd["new_lens"][2] = 1       # one more token than it can hold
    assert hd.step(upd) == oracle.E_LENS


# ------------------------------------------------------------ recent window --

def _held_classes(hd: HostDecode):
    out = {}
    for r in range(hd.w.R):
        c = int(hd.ctx_lens[r])
        out[r] = hd.classes[:, r * hd.cap:r * hd.cap + c].copy()
    return out


def test_window_covering_everything_only_appends():
    """Mode 0 with a window longer than every request: no held token is
    re-scored, each new token enters as K8V4, and every held token keeps its
    slot bytes; the appended token's codes are the textbook 8-bit / 4-bit
    quantisation of its row."""
    w = _small()
    hd = HostDecode(w, cap=560, window=10_000, mode=0)
    before = _state(hd)
    held = _held_classes(hd)
    upd = W.decode_update_inputs(w, hd.ctx, 0, p_prune=0.2, p_demote=0.2)
    ctx0 = hd.ctx_lens.copy()
    assert hd.step(upd) == oracle.OK
    after = _state(hd)
    for r in range(w.R):
        assert np.array_equal(hd.classes[:, r * 560:r * 560 + int(ctx0[r])], held[r])
    for key, val in before.items():
        assert after[key] == val, key  # same list, same slot, same bytes
    kb = upd["k_new"].view(torch.int16).numpy().view(np.uint16)
    vb = upd["v_new"].view(torch.int16).numpy().view(np.uint16)
    for u in range(w.U):
        l, r, h = u // (w.R * w.Hkv), (u // w.Hkv) % w.R, u % w.Hkv
        if int(upd["new_lens"][r]) == 0:
            continue
        li, raw, _ = after[(u, int(ctx0[r]))]
        assert li == 0  # K8V4
        kq, vq, meta = slot_codes(raw, high=True)
        _, k8, ks, kz = oracle.quant_row(kb[l, r, h], 8)
        _, v4, vs, vz = oracle.quant_row(vb[l, r, h], 4)
        assert np.array_equal(kq, k8) and np.array_equal(vq, v4) and list(meta) == [ks, kz, vs, vz]


@pytest.mark.parametrize("window", [0, 3, 40])
def test_candidate_mode_reclassifies_only_the_leaving_token(window):
    """Mode 1: per request only position ctx - W (the token the new one pushes
    out of the window) may change class, never upward; with W = 0 that is the
    new token itself, classified as in prefill."""
    w = _small()
    hd = HostDecode(w, cap=600, window=window, mode=1)
    for s in range(4):
        held = _held_classes(hd)
        ctx0 = hd.ctx_lens.copy()
        upd = W.decode_update_inputs(w, hd.ctx, s, p_prune=0.2, p_demote=0.2)
        assert hd.step(upd) == oracle.OK
        for r in range(w.R):
            c = int(ctx0[r])
            now = hd.classes[:, r * 600:r * 600 + c]
            diff = np.nonzero((now != held[r]).any(axis=(0, 2)))[0]
            assert all(i == c - window for i in diff) if window >= 1 else diff.size == 0, (s, r, diff)
            assert np.all(now <= held[r])
            if int(upd["new_lens"][r]) and window >= 1:
                assert np.all(hd.classes[:, r * 600 + c] == 2)
        _state(hd)


def test_window_invariants_over_steps_both_modes():
    w = _small()
    for mode in (0, 1):
        hd = HostDecode(w, cap=600, window=16, mode=mode)
        for s in range(6):
            assert hd.step(p_prune=0.05, p_demote=0.05) == oracle.OK
            _state(hd)
