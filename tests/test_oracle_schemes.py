"""Pins for the oracle's precision schemes (reading F; CPU only).

The DiffKV review's free-parameter list says the precision-level scheme
K8V4-K4V2 was chosen by comparing K8V4, K4V8, K8V2, K4V2, K2V4 and K4V1
(its Section 7.2).  Read as a pair of a high class and a half-width low class
they give three schemes: K8V4/K4V2 (0), K8V2/K4V1 (1) and K4V8/K2V4 (2).
Each is pinned here against something other than the oracle itself:
  - exact grids at every width the schemes use (8, 4, 2 and 1 bits) give codes
    equal to the grid index and an exact dequantisation;
  - with alpha_h = alpha_l = 0 every token is high class and each stored row
    equals the textbook per-token quantiser at the scheme's widths, at the
    offsets the documented page layout gives;
  - the classes, page ids, tables and cursors do not depend on the scheme
    (a low token takes exactly half a high token's code bytes, so the page
    demand is the same);
  - the 1-bit quantiser: a two-level row is exact and the midpoint is a tie
    that rounds to the even code 0;
  - the payload fraction of a scheme is ((kh + vh) n_hi + (kh + vh)/2 n_lo)
    / (32 N) of fp16, the review's 27.4% = (12 h + 6 l)/32 form for scheme 0;
  - demotion on exact grids equals the textbook quantiser at the low widths
    of the original rows, in every scheme.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import workloads as W
from oracle.host_decode import HostDecode
from tests.decode_helpers import list_slots, slot_codes
from tests.edge_rows import bf16_bits_exact
from tests.oracle_helpers import SCHEME_BITS, Layout, bf16_to_f32, f16, page_slots, run_oracle, unit_rows

SCHEMES = [0, 1, 2]


def _textbook(x_bits, nbits):
    """Per-token asymmetric uniform quantisation (KIVI-style) in numpy
    float32 / float16 arithmetic, ties to even."""
    x = bf16_to_f32(x_bits)
    n = np.float32((1 << nbits) - 1)
    mn, mx = x.min() + np.float32(0.0), x.max() + np.float32(0.0)
    s16 = np.float16(np.float32(mx - mn) / n)
    if mx > mn and s16 == 0:
        s16 = np.float16(2.0 ** -24)
    z16 = np.float16(mn)
    s, z = np.float32(s16), np.float32(z16)
    q = np.zeros(128, dtype=np.uint8) if s == 0 else np.clip(np.rint((x - z) / s), 0, n).astype(np.uint8)
    return q, np.array([s16, z16], dtype=np.float16).view(np.uint16)


@pytest.mark.parametrize("bits", [8, 4, 2, 1])
def test_exact_grid_at_every_width(bits):
    n = (1 << bits) - 1
    rng = np.random.default_rng(bits)
    grids = 0
    for z, s in ((-1.0, 2.0 ** -5), (0.5, 2.0 ** -3), (-96.0, 8.0)):
        cand = np.arange(n + 1)
        vals = (np.float64(z) + cand * s).astype(np.float32)
        cand = cand[(vals.view(np.uint32) & 0xFFFF) == 0]   # grid points bf16 holds exactly
        if cand[0] != 0 or cand[-1] != n:
            continue
        grids += 1
        k = rng.choice(cand, size=128)
        k[0], k[1] = 0, n
        x = (np.float64(z) + k * s).astype(np.float32)
        st, q, s16, z16 = oracle.quant_row(bf16_bits_exact(x), bits)
        assert st == oracle.OK
        assert np.array_equal(q, k) and f16([s16])[0] == np.float32(s) and f16([z16])[0] == np.float32(z)
    assert grids >= 2


def test_one_bit_two_levels_and_midpoint_tie():
    x = np.full(128, -0.5, dtype=np.float32)
    x[::3] = 1.5
    x[5] = 0.5                       # exactly half way: t = 1/2, ties to the even code 0
    x[7] = np.float32(0.50390625)    # one bf16 ulp above the midpoint: code 1
    st, q, s16, z16 = oracle.quant_row(bf16_bits_exact(x), 1)
    assert st == oracle.OK and f16([s16])[0] == 2.0 and f16([z16])[0] == -0.5
    want = (x > 0.5).astype(np.uint8)
    assert np.array_equal(q, want)


@pytest.mark.parametrize("scheme", SCHEMES)
def test_all_high_reduces_to_the_textbook_quantiser(scheme):
    w = W.small("sch_tb", L=1, lens=[70, 33], P=8, scheme=scheme)
    n = W.to_numpy(W.make_inputs(w, seed=3))
    st, pool, tab = run_oracle(w, n, alpha_h=0.0, alpha_l=0.0)
    assert st == oracle.OK and np.all(tab.classes == 2)
    kh, vh = SCHEME_BITS[scheme]
    assert pool.pages.shape[1] == (16 * (kh + vh) + 24) * w.P
    for u in range(w.U):
        l, r, h, start, N = unit_rows(w, 1, u)
        seen = 0
        for k in range(tab.pmax):
            pid = tab.fwd[u, k]
            if pid < 0:
                break
            for slot, (kc, vc, meta, pos) in enumerate(page_slots(pool.pages[pid], w.P, 2, scheme)):
                if pos < 0:
                    continue
                assert pos == k * w.P + slot
                qk, mk = _textbook(n["k"][0, start + pos, h], kh)
                qv, mv = _textbook(n["v"][0, start + pos, h], vh)
                assert np.array_equal(kc, qk) and np.array_equal(vc, qv)
                assert np.array_equal(meta, np.concatenate([mk, mv]))
                seen += 1
        assert seen == N


@pytest.mark.parametrize("scheme", [1, 2])
def test_tables_do_not_depend_on_the_scheme(scheme):
    w0 = W.small("sch_inv", lens=[300, 7, 517, 0, 129])
    w1 = W.small("sch_inv", lens=[300, 7, 517, 0, 129], scheme=scheme)
    n = W.to_numpy(W.make_inputs(w0, seed=4))
    st0, p0, t0 = run_oracle(w0, n)
    st1, p1, t1 = run_oracle(w1, n)
    assert st0 == st1 == oracle.OK
    for a, b in ((t0.classes, t1.classes), (t0.fwd, t1.fwd), (t0.unit_hdr, t1.unit_hdr), (p0.cursors, p1.cursors),
                 (p0.rev_unit, p1.rev_unit), (p0.rev_idx, p1.rev_idx), (p0.page_cls, p1.page_cls)):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("scheme", SCHEMES)
def test_low_class_rows_at_half_width(scheme):
    """alpha_h = inf, alpha_l = 0: every token is low class, stored at
    (kh/2, vh/2) bits, 2P to a page."""
    w = W.small("sch_lo", L=1, lens=[50], P=4, scheme=scheme)
    n = W.to_numpy(W.make_inputs(w, seed=6))
    st, pool, tab = run_oracle(w, n, alpha_h=1e30, alpha_l=0.0)
    assert st == oracle.OK and np.all(tab.classes == 1)
    kh, vh = SCHEME_BITS[scheme]
    for u in range(w.U):
        l, r, h, start, N = unit_rows(w, 1, u)
        for k in range(tab.pmax):
            pid = tab.fwd[u, k]
            if pid < 0:
                break
            for slot, (kc, vc, meta, pos) in enumerate(page_slots(pool.pages[pid], w.P, 1, scheme)):
                if pos < 0:
                    continue
                assert pos == k * 2 * w.P + slot
                qk, mk = _textbook(n["k"][0, start + pos, h], kh // 2)
                qv, mv = _textbook(n["v"][0, start + pos, h], vh // 2)
                assert np.array_equal(kc, qk) and np.array_equal(vc, qv)


@pytest.mark.parametrize("scheme", SCHEMES)
def test_payload_fraction_closed_form(scheme):
    """Code bytes of the stored tokens over the fp16 bytes of all tokens:
    ((kh + vh) n_hi + (kh + vh)/2 n_lo) / (32 N), counted from the pages."""
    w = W.small("sch_frac", L=1, lens=[400, 200], scheme=scheme)
    n = W.to_numpy(W.make_inputs(w, seed=8))
    st, pool, tab = run_oracle(w, n)
    assert st == oracle.OK
    kh, vh = SCHEME_BITS[scheme]
    lay = Layout(w.P, scheme)
    code_bytes = 0
    for pid in np.nonzero(pool.page_cls)[0]:
        high = pool.page_cls[pid] == 2
        for (kc, vc, meta, pos) in page_slots(pool.pages[pid], w.P, pool.page_cls[pid], scheme):
            if pos >= 0:
                code_bytes += 16 * (lay.kbits(high) + lay.vbits(high))
    n_hi, n_lo = int((tab.classes == 2).sum()), int((tab.classes == 1).sum())
    N = w.T * w.Hkv
    assert code_bytes / (2 * 2 * 128 * N) == pytest.approx(((kh + vh) * n_hi + (kh + vh) / 2 * n_lo) / (32 * N))


@pytest.mark.parametrize("scheme", SCHEMES)
def test_demotion_on_exact_grids_equals_the_textbook_quantiser(scheme):
    """Rows whose high-class codes dequantise exactly (integers from 0 to the
    high width's top code): after demotion the low-class codes equal the
    textbook quantisation of the original rows at the low widths."""
    kh, vh = SCHEME_BITS[scheme]
    w = W.small("sch_dem", lens=[70, 40], L=1, Hq=4, Hkv=2, n_outlier=0, scheme=scheme)
    inp = W.make_inputs(w, 5)
    g = torch.Generator().manual_seed(9)
    rows = w.T * w.Hkv
    kk = torch.randint(0, 1 << kh, (rows, 128), generator=g).to(torch.float32)
    vv = torch.randint(0, 1 << vh, (rows, 128), generator=g).to(torch.float32)
    kk[:, 0], kk[:, 1] = 0.0, float((1 << kh) - 1)
    vv[:, 0], vv[:, 1] = 0.0, float((1 << vh) - 1)
    inp["k"] = kk.view(1, w.T, w.Hkv, 128).to(torch.bfloat16)
    inp["v"] = vv.view(1, w.T, w.Hkv, 128).to(torch.bfloat16)
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
        for s in list_slots(hd.pool.pages, hd.tab.fwd[u], hdr, w.P, scheme)[1][:int(hdr[1])]:
            kq, vq, meta = slot_codes(s[:3], high=False, scheme=scheme)
            qk, mk = _textbook(kb[0, tok0 + s[3], h], kh // 2)
            qv, mv = _textbook(vb[0, tok0 + s[3], h], vh // 2)
            assert np.array_equal(kq, qk) and np.array_equal(vq, qv)
            assert list(meta) == list(np.concatenate([mk, mv]))
            seen += 1
    assert seen > 5


def test_one_bit_scale_overflow_is_lowered_to_the_largest_binary16():
    """Reading Q1 step 3: at 1 bit a span above 65519 would round the scale
    to infinity; it becomes 65504 (0x7bff), so x = min + k 65504 dequantise
    exactly and the top element clamps to code 1."""
    x = np.full(128, -65280.0, dtype=np.float32)
    x[1::4] = np.float32(-65280.0 + 65504.0)   # 224: min + one scale step, exact in bf16
    x[2] = 65280.0                             # span 130560: t = 1.993, clamped to code 1
    st, q, s16, z16 = oracle.quant_row(bf16_bits_exact(x), 1)
    assert st == oracle.OK and s16 == 0x7BFF and f16([z16])[0] == -65280.0
    assert np.array_equal(q, (x > -65280.0).astype(np.uint8))
    for bits in (2, 4, 8):  # wider codes never overflow: 130560 / 3 < 65504
        st, q, s16, z16 = oracle.quant_row(bf16_bits_exact(x), bits)
        assert st == oracle.OK and np.isfinite(f16([s16])[0])
