"""GPU parity of decode attention at the full decode workload: 32 layers, 256
requests holding 2048..8192 tokens, every layer attended in one call with
the new tokens and the significance update, in the launch configuration the
benchmark times.

The oracle replays sampled units (layers 0 and 31, requests 0, 128 and 255,
all 8 KV heads) on a pool of their own built from the device's page bytes:
the same codes, metadata and positions, the units' forward rows renumbered.
Outputs and the probabilities added to the significance sums are held to the
bound derived from the fp32 arithmetic (tests/attention_helpers.py)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import decode_setup as DS
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.attention_helpers import U, attention_bounds, unit_tokens
from tests.oracle_helpers import bf16_to_f32

pytestmark = pytest.mark.gpu

SAMPLES = [(0, 0), (0, 128), (0, 255), (31, 0), (31, 128), (31, 255)]  # (layer, request)
SCALE = 0.08838834764831845


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def test_attention_decode_workload_full_size():
    w = W.get("decode")
    dev = torch.device("cuda", 0)
    dec, ctx, cap, _ = DS.decode_setup(w, dev, W.SEED_BASE + 7, 2)
    q = W.decode_queries(w, w.L, W.SEED_BASE + 3, device=dev)
    upd = W.decode_update_inputs(w, {k: (v.clone() if torch.is_tensor(v) else v) for k, v in ctx.items()}, 0,
                                 device=dev)
    sig0 = {(l, r): ctx["sig_sum"][l].view(w.R, cap, w.Hq)[r].cpu().numpy().astype(np.float64)
            for l, r in SAMPLES}
    out = torch.empty((w.L, w.R, w.Hq, 128), dtype=torch.float32, device=dev)
    dec.attend(q, ctx["ctx_lens"], out, SCALE, k_new=upd["k_new"], v_new=upd["v_new"], new_lens=upd["new_lens"],
               sig_sum=ctx["sig_sum"])
    st = libdkv.dkv_get_status(dec.pool)
    assert st == libdkv.DKV_OK, libdkv.status_string(st)

    # the sampled units' pages, renumbered into an oracle pool of their own
    Hkv, P = w.Hkv, w.P
    hdr = dec.tables.unit_hdr.cpu().numpy()
    fwd = dec.tables.fwd
    Rs = len(SAMPLES)
    units = [((l * w.R + r) * Hkv + h) for l, r in SAMPLES for h in range(Hkv)]
    npages = [int(hdr[u][2] + hdr[u][3]) for u in units]
    pool = oracle.Pool(sum(npages), P)
    tab = oracle.Tables(Rs * Hkv, dec.pmax, 1)
    base = 0
    for i, u in enumerate(units):
        ids = fwd[u, :npages[i]].long()
        pool.pages[base:base + npages[i]] = dec.pool.pages[ids].cpu().numpy()
        tab.fwd[i, :] = -1
        tab.fwd[i, :npages[i]] = np.arange(base, base + npages[i], dtype=np.int32)
        tab.unit_hdr[i] = hdr[u]
        base += npages[i]
    qs = torch.stack([q[l, r] for l, r in SAMPLES])[None]
    kn = torch.stack([upd["k_new"][l, r] for l, r in SAMPLES])[None]
    vn = torch.stack([upd["v_new"][l, r] for l, r in SAMPLES])[None]
    rq = [r for _, r in SAMPLES]
    nl = upd["new_lens"].cpu().numpy()[rq].astype(np.int32)
    cl = ctx["ctx_lens"].cpu().numpy()[rq].astype(np.int32)
    a = {"L": 1, "R": Rs, "Hq": w.Hq, "Hkv": Hkv, "cap": cap, "layer0": 0, "n_layers": 1, "q": _bits(qs),
         "k_new": _bits(kn), "v_new": _bits(vn), "new_lens": nl, "ctx_lens": cl, "scale": SCALE}
    rc, o_ref, p_ref = oracle.decode_attention(a, pool, tab)
    assert rc == oracle.OK
    G = w.Hq // Hkv
    qf = bf16_to_f32(_bits(qs[0])).astype(np.float64)
    knf = bf16_to_f32(_bits(kn[0])).astype(np.float64)
    vnf = bf16_to_f32(_bits(vn[0])).astype(np.float64)
    for j, (l, r) in enumerate(SAMPLES):
        o_gpu = out[l, r].cpu().numpy().astype(np.float64)
        s_gpu = ctx["sig_sum"][l].view(w.R, cap, w.Hq)[r].cpu().numpy().astype(np.float64)
        for h in range(Hkv):
            i = j * Hkv + h
            toks = unit_tokens(pool.pages, tab.fwd[i], tab.unit_hdr[i], P)
            pos = list(toks[6]) + ([int(cl[j])] if nl[j] else [])
            newkv = (knf[j, h], vnf[j, h]) if nl[j] else None
            for g in range(G):
                qh = h * G + g
                p = p_ref[0, j * cap + np.array(pos, dtype=np.int64), qh]
                ob, pb = attention_bounds(qf[j, qh], SCALE, toks, newkv, p)
                err = np.abs(o_gpu[qh] - o_ref[0, j, qh])
                assert np.all(err <= ob), (l, r, qh, float(err.max()), float(ob.max()))
                base_s = sig0[(l, r)][pos, qh].copy()
                if nl[j]:
                    base_s[-1] = 0.0
                serr = np.abs(s_gpu[pos, qh] - (base_s + p))
                assert np.all(serr <= pb + U * np.abs(base_s + p)), (l, r, qh, float(serr.max()))
