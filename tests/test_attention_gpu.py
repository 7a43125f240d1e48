"""GPU parity of decode attention over the unified pages
(dkv_decode_attention) against the oracle's double-precision attention.

Each state comes from a prefill plus generation steps with churn, run on the
GPU and the oracle alike (bit-identical, as the decode tests establish), so
both attend over the same bytes.  Outputs and the probabilities added to the
significance sums are compared per channel / token against the bound derived
from the fp32 arithmetic (tests/attention_helpers.py); positions that were
not attended must keep their significance bits."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.attention_helpers import U, attention_bounds, unit_tokens
from tests.decode_helpers import HostDecode
from tests.oracle_helpers import bf16_to_f32
from tests.test_decode_gpu import _dev, gpu_decoder

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _state(w, cap, steps, seed=77, p=0.05):
    inp = W.make_inputs(w, seed)
    hd = HostDecode(w, cap, inp=inp)
    dec = gpu_decoder(hd, inp)
    for s in range(steps):
        upd = W.decode_update_inputs(w, hd.ctx, s, p_prune=p, p_demote=p)
        d = {"k_new": _dev(upd["k_new"]), "v_new": _dev(upd["v_new"]), "sig_sum": _dev(hd.ctx["sig_sum"]),
             "sig_cnt": _dev(hd.ctx["sig_cnt"]), "ctx_lens": _dev(hd.ctx["ctx_lens"]),
             "new_lens": _dev(upd["new_lens"])}
        dec.step(d, w.alpha_h, w.alpha_l)
        assert hd.step(upd) == oracle.OK
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_OK
    torch.cuda.synchronize()
    assert np.array_equal(dec.tables.unit_hdr.cpu().numpy(), hd.tab.unit_hdr)
    return hd, dec


def _check(hd, dec, layer0, n_layers, with_new, scale=0.08838834764831845, seed=3):
    """One attention call on both sides; returns the largest error / bound."""
    w, cap = hd.w, hd.cap
    q = W.decode_queries(w, n_layers, seed)
    upd = W.decode_update_inputs(w, {k: (v.clone() if torch.is_tensor(v) else v) for k, v in hd.ctx.items()},
                                 99, seed=seed) if with_new else None
    kn = upd["k_new"][layer0:layer0 + n_layers].contiguous() if with_new else None
    vn = upd["v_new"][layer0:layer0 + n_layers].contiguous() if with_new else None
    nl = upd["new_lens"] if with_new else None
    ctx = hd.ctx["ctx_lens"]
    sig0 = hd.ctx["sig_sum"].clone()
    sig = _dev(sig0)
    out = torch.empty((n_layers, w.R, w.Hq, 128), dtype=torch.float32, device="cuda")
    dec.attend(_dev(q), _dev(ctx), out, scale, layer0=layer0, k_new=None if kn is None else _dev(kn),
               v_new=None if vn is None else _dev(vn), new_lens=None if nl is None else _dev(nl), sig_sum=sig)
    st = libdkv.dkv_get_status(dec.pool)
    assert st == libdkv.DKV_OK, libdkv.status_string(st)
    a = {"L": w.L, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "cap": cap, "layer0": layer0, "n_layers": n_layers,
         "q": _bits(q), "k_new": None if kn is None else _bits(kn), "v_new": None if vn is None else _bits(vn),
         "new_lens": None if nl is None else nl.numpy().astype(np.int32), "ctx_lens": ctx.numpy(), "scale": scale}
    rc, o_ref, p_ref = oracle.decode_attention(a, hd.pool, hd.tab)
    assert rc == oracle.OK
    o_gpu = out.cpu().numpy().astype(np.float64)
    s_gpu = sig.cpu().numpy().astype(np.float64)
    s_old = sig0.numpy().astype(np.float64)
    G = w.Hq // w.Hkv
    qf = bf16_to_f32(_bits(q)).astype(np.float64)
    worst = 0.0
    touched = np.zeros(s_old.shape, bool)
    for li in range(n_layers):
        l = layer0 + li
        for r in range(w.R):
            has_new = with_new and int(nl[r]) == 1
            for h in range(w.Hkv):
                u = (l * w.R + r) * w.Hkv + h
                toks = unit_tokens(hd.pool.pages, hd.tab.fwd[u], hd.tab.unit_hdr[u], w.P, w.scheme)
                pos = list(toks[6])
                if has_new:
                    pos.append(int(ctx[r]))
                newkv = None
                if has_new:
                    newkv = (bf16_to_f32(_bits(kn[li, r, h])).astype(np.float64),
                             bf16_to_f32(_bits(vn[li, r, h])).astype(np.float64))
                rows = r * cap + np.array(pos, dtype=np.int64)
                for g in range(G):
                    qh = h * G + g
                    p = p_ref[li, rows, qh] if pos else np.zeros(0)
                    ob, pb = attention_bounds(qf[li, r, qh], scale, toks, newkv, p)
                    err = np.abs(o_gpu[li, r, qh] - o_ref[li, r, qh])
                    assert np.all(err <= ob + 1e-30), (l, r, qh, float(err.max()), float(ob.max()))
                    if pos:
                        worst = max(worst, float((err / np.maximum(ob, 1e-300)).max()))
                        got = s_gpu[l, rows, qh]
                        want = p
                        base = s_old[l, rows, qh].copy()
                        if has_new:
                            base[-1] = 0.0  # the new token's row is set, not added to
                        serr = np.abs(got - (base + want))
                        sb = pb + U * np.abs(base + want)
                        assert np.all(serr <= sb + 1e-30), (l, r, qh, float(serr.max()))
                        touched[l, rows, qh] = True
    # rows nobody attended keep their bits
    assert np.array_equal(s_gpu[~touched].astype(np.float32).view(np.uint32),
                          s_old[~touched].astype(np.float32).view(np.uint32))
    return worst


@pytest.mark.parametrize("with_new", [False, True])
def test_attention_small_ragged(with_new):
    w = W.small("att", lens=[300, 7, 517, 0, 129])
    hd, dec = _state(w, cap=560, steps=4)
    _check(hd, dec, 0, w.L, with_new)


@pytest.mark.parametrize("shape", [
    dict(Hq=28, Hkv=4, P=32, lens=[1000, 33, 700], alpha_h=1.5, alpha_l=0.3, sigma=2.5),  # G = 7
    dict(Hq=16, Hkv=2, P=16, lens=[2100, 64], L=1),                                     # G = 8
    dict(Hq=4, Hkv=4, P=2, lens=[90, 91, 1], L=1),                                       # G = 1, tiny pages
    dict(Hq=8, Hkv=2, P=16, lens=[5000, 300, 2], L=1),                                   # G = 4
    dict(Hq=16, Hkv=2, P=16, lens=[5000, 64], L=1),                                      # G = 8, 2-block clusters
    dict(Hq=16, Hkv=2, P=16, lens=[15000, 700], L=1),                                    # G = 8, 8-block clusters
])
def test_attention_shapes(shape):
    w = W.small("atts", **shape)
    cap = (max(w.lens) + 16 + 15) // 16 * 16
    hd, dec = _state(w, cap=cap, steps=3)
    _check(hd, dec, 0, w.L, True)


@pytest.mark.parametrize("scheme", [1, 2], ids=["k8v2-k4v1", "k4v8-k2v4"])
@pytest.mark.parametrize("shape", [
    dict(lens=[300, 7, 517, 0, 129]),                            # G = 3, 2 layers
    dict(Hq=8, Hkv=2, P=16, lens=[2100, 300, 2], L=1),           # G = 4
    dict(Hq=16, Hkv=2, P=16, lens=[1500, 64], L=1),              # G = 8
    dict(Hq=4, Hkv=4, P=2, lens=[90, 91, 1], L=1),               # G = 1, tiny pages
], ids=["g3", "g4", "g8", "g1-p2"])
def test_attention_other_schemes(scheme, shape):
    """The bit-width schemes beside K8V4/K4V2: pages of K8V2/K4V1 (1-bit low
    values) and K4V8/K2V4 (2-bit low keys, 8-bit high values), after
    generation steps with churn, with the new token."""
    w = W.small("attsc", scheme=scheme, **shape)
    cap = (max(w.lens) + 16 + 15) // 16 * 16
    hd, dec = _state(w, cap=cap, steps=3)
    _check(hd, dec, 0, w.L, True)


def test_attention_one_layer_of_several():
    w = W.small("att1", lens=[300, 7, 517, 0, 129], L=3)
    hd, dec = _state(w, cap=560, steps=2)
    _check(hd, dec, 1, 1, True)


def test_attention_new_token_past_capacity_is_a_length_error():
    """A new token at ctx = cap cannot have a significance row: LENS, and the
    call attends without it."""
    w = W.small("attc", lens=[32, 5], L=1, Hq=4, Hkv=2)
    hd, dec = _state(w, cap=32, steps=0)
    q = W.decode_queries(w, 1, 1)
    kn = W.decode_queries(W.small("x", lens=[32, 5], L=1, Hq=2, Hkv=2), 1, 2)
    out = torch.empty((1, w.R, w.Hq, 128), dtype=torch.float32, device="cuda")
    dec.attend(_dev(q), _dev(hd.ctx["ctx_lens"]), out, 0.088, k_new=_dev(kn), v_new=_dev(kn),
               new_lens=_dev(torch.tensor([1, 1], dtype=torch.int32)))
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_E_LENS
    out2 = torch.empty_like(out)
    dec.attend(_dev(q), _dev(hd.ctx["ctx_lens"]), out2, 0.088, k_new=_dev(kn), v_new=_dev(kn),
               new_lens=_dev(torch.tensor([0, 1], dtype=torch.int32)))
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_OK
    assert torch.equal(out[0, 0], out2[0, 0])  # request 0 attended its held tokens only


def test_attention_leaves_out_what_contradicts_the_tables():
    """A unit header whose page counts do not match its token counts, or a
    forward entry outside the pool, is reported (DKV_E_INTERNAL) and left out:
    the kernel reads no page through it, and every other unit's output keeps
    its bits (the kernel's reductions run in a fixed order)."""
    w = W.small("attx", lens=[300, 7, 517, 0, 129], L=1)
    hd, dec = _state(w, cap=560, steps=1)
    q = _dev(W.decode_queries(w, 1, 4))
    ctx = _dev(hd.ctx["ctx_lens"])

    def run():
        out = torch.zeros((1, w.R, w.Hq, 128), dtype=torch.float32, device="cuda")
        dec.attend(q, ctx, out, 0.088)
        return out, libdkv.dkv_get_status(dec.pool)

    ref, st = run()
    assert st == libdkv.DKV_OK
    G = w.Hq // w.Hkv
    u_bad = 2 * w.Hkv + 1  # request 2, KV head 1
    keep = torch.ones(w.R * w.Hkv, dtype=torch.bool)
    keep[u_bad] = False
    keep = keep.view(w.R, w.Hkv).repeat_interleave(G, dim=1).cuda()  # [R, Hq]

    saved = dec.tables.unit_hdr[u_bad].clone()
    dec.tables.unit_hdr[u_bad, 2] += 1  # one more K8V4 page than its tokens need
    out, st = run()
    dec.tables.unit_hdr[u_bad] = saved
    assert st == libdkv.DKV_E_INTERNAL
    assert torch.equal(out[0][keep], ref[0][keep])
    assert not out[0, 2, G:2 * G].any()  # the rejected unit attends to nothing

    saved = dec.tables.fwd[u_bad, 0].clone()
    dec.tables.fwd[u_bad, 0] = dec.pool.F + 5  # a page id outside the pool
    out, st = run()
    dec.tables.fwd[u_bad, 0] = saved
    assert st == libdkv.DKV_E_INTERNAL
    assert torch.equal(out[0][keep], ref[0][keep])
    assert torch.isfinite(out).all()
    out, st = run()
    assert st == libdkv.DKV_OK and torch.equal(out, ref)
