"""GPU parity of prefill attention with significance accumulation
(dkv_prefill_attention) against the oracle's double-precision result: the
outputs and significance sums inside the bound derived from the fp32
arithmetic (tests/attention_helpers.py), the counts exact.  Ragged requests
with lengths across the 64-token tiles, several GQA shapes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.attention_helpers import prefill_bounds
from tests.oracle_helpers import bf16_to_f32

pytestmark = pytest.mark.gpu

SCALE = 0.08838834764831845


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _run(w: W.Workload, seed: int = 3):
    k = torch.stack([W.make_kv_layer(w, seed, l, 0) for l in range(w.L)])
    v = torch.stack([W.make_kv_layer(w, seed, l, 1) for l in range(w.L)])
    q = torch.randn((w.L, w.T, w.Hq, 128), generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    lens = torch.tensor(w.lens, dtype=torch.int32)
    pool = libdkv.DevicePool(4, 16)
    out = torch.full((w.L, w.T, w.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    sig = torch.full((w.L, w.T, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    cnt = torch.full((w.T,), -5, dtype=torch.int32, device="cuda")
    libdkv.dkv_init_pool(pool)
    libdkv.dkv_prefill_attention(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), max(w.lens + [0]), SCALE, out, sig, cnt,
                                 pool)
    st = libdkv.dkv_get_status(pool)
    assert st == libdkv.DKV_OK, libdkv.status_string(st)
    rc, o_ref, s_ref, c_ref = oracle.prefill_attention(_bits(q), _bits(k), _bits(v), w.lens, SCALE)
    assert rc == oracle.OK
    assert np.array_equal(cnt.cpu().numpy(), c_ref)
    o_gpu = out.cpu().numpy().astype(np.float64)
    s_gpu = sig.cpu().numpy().astype(np.float64)
    qf = bf16_to_f32(_bits(q)).astype(np.float64)
    kf = bf16_to_f32(_bits(k)).astype(np.float64)
    vf = bf16_to_f32(_bits(v)).astype(np.float64)
    G = w.Hq // w.Hkv
    worst = 0.0
    start = 0
    for n in w.lens:
        for l in range(w.L):
            for qh in range(w.Hq):
                sl = slice(start, start + n)
                ob, sb, _ = prefill_bounds(qf[l, sl, qh], kf[l, sl, qh // G], vf[l, sl, qh // G], SCALE)
                eo = np.abs(o_gpu[l, sl, qh] - o_ref[l, sl, qh])
                es = np.abs(s_gpu[l, sl, qh] - s_ref[l, sl, qh])
                assert np.all(eo <= ob), (n, l, qh, float(eo.max()), float(ob.max()))
                assert np.all(es <= sb), (n, l, qh, float(es.max()), float(sb.max()))
                if n:
                    worst = max(worst, float((eo / ob).max()), float((es / sb).max()))
        start += n
    return worst


def test_prefill_attention_small_ragged():
    w = W.small("pfa", lens=[300, 7, 517, 0, 129])  # G = 3
    _run(w)


@pytest.mark.parametrize("shape", [
    dict(Hq=8, Hkv=2, lens=[65, 64, 1, 133], L=1),      # G = 4, lengths across the 64-query tiles
    dict(Hq=4, Hkv=4, lens=[200, 3], L=1),              # G = 1
    dict(Hq=16, Hkv=2, lens=[90, 257], L=1),            # G = 8
])
def test_prefill_attention_shapes(shape):
    _run(W.small("pfs", **shape))


def test_prefill_attention_feeds_compaction():
    """Its significance sums and counts are the compaction's inputs: classes
    from them agree with the oracle's classes from the oracle's sums, except
    where a token's score is within the sums' error bound of a threshold."""
    # thresholds inside the spread of N x score of these random-query softmaxes
    # (about 0.7 .. 5.4 between the 5th and 95th percentiles): all three classes
    w = W.small("pfc", lens=[300, 129], L=1, Hq=8, Hkv=2, alpha_h=1.7, alpha_l=0.9)
    k = torch.stack([W.make_kv_layer(w, 9, 0, 0)])
    v = torch.stack([W.make_kv_layer(w, 9, 0, 1)])
    q = torch.randn((1, w.T, w.Hq, 128), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    lens = torch.tensor(w.lens, dtype=torch.int32)
    pool = libdkv.DevicePool(w.pool_pages, w.P)
    libdkv.dkv_init_pool(pool)
    sig = torch.empty((1, w.T, w.Hq), dtype=torch.float32, device="cuda")
    cnt = torch.empty((w.T,), dtype=torch.int32, device="cuda")
    out = torch.empty((1, w.T, w.Hq, 128), dtype=torch.float32, device="cuda")
    libdkv.dkv_prefill_attention(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), max(w.lens), SCALE, out, sig, cnt, pool)
    comp = libdkv.Compactor(1, w.R, w.Hq, w.Hkv, w.T, max(w.lens), w.P, w.pool_pages)
    comp.compact({"L": 1, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T, "k": k.cuda(), "v": v.cuda(),
                  "sig_sum": sig, "sig_cnt": cnt, "lens": lens.cuda()}, w.alpha_h, w.alpha_l)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    rc, _, s_ref, c_ref = oracle.prefill_attention(_bits(q), _bits(k), _bits(v), w.lens, SCALE)
    G = w.Hq // w.Hkv
    score = (s_ref / c_ref[None, :, None]).reshape(w.T, w.Hkv, G).max(2)  # [T][Hkv]
    N = np.repeat(np.array(w.lens, dtype=np.float64), w.lens)[:, None]
    want = np.where(score >= w.alpha_h / N, 2, np.where(score >= w.alpha_l / N, 1, 0))
    got = comp.classes.cpu().numpy().reshape(w.T, w.Hkv)
    near = (np.abs(score - w.alpha_h / N) < 1e-4 * w.alpha_h / N) | (np.abs(score - w.alpha_l / N) < 1e-4 * w.alpha_l / N)
    assert np.array_equal(got[~near], want[~near])
    assert (got == 2).any() and (got == 1).any() and (got == 0).any()


@pytest.mark.parametrize("bad_lens,max_len", [
    ([-5, 70, 10], 70),     # a negative earlier length: request 1 would start before the layer
    ([20, 55, 0], 50),      # a length above max_len: its queries past the grid would go uncomputed
    ([20, 30, 10], 64),     # lengths that do not add up to T
])
def test_prefill_attention_rejects_bad_lengths(bad_lens, max_len):
    """Every length is validated before any access: DKV_E_LENS is recorded,
    and neither the outputs nor the counts are written."""
    T = 75
    g = torch.Generator().manual_seed(4)
    q = torch.randn((1, T, 4, 128), generator=g).to(torch.bfloat16).cuda()
    k = torch.randn((1, T, 2, 128), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((1, T, 2, 128), generator=g).to(torch.bfloat16).cuda()
    pool = libdkv.DevicePool(4, 16)
    libdkv.dkv_init_pool(pool)
    out = torch.full((1, T, 4, 128), 7.0, dtype=torch.float32, device="cuda")
    sig = torch.empty((1, T, 4), dtype=torch.float32, device="cuda")
    cnt = torch.full((T,), -5, dtype=torch.int32, device="cuda")
    lens = torch.tensor(bad_lens, dtype=torch.int32, device="cuda")
    libdkv.dkv_prefill_attention(q, k, v, lens, max_len, SCALE, out, sig, cnt, pool)
    assert libdkv.dkv_get_status(pool) == libdkv.DKV_E_LENS
    assert torch.all(out == 7.0) and torch.all(cnt == -5)
    # the same buffers with valid lengths then work
    lens = torch.tensor([20, 45, 10], dtype=torch.int32, device="cuda")
    libdkv.dkv_prefill_attention(q, k, v, lens, 64, SCALE, out, sig, cnt, pool)
    assert libdkv.dkv_get_status(pool) == libdkv.DKV_OK
    assert cnt[0].item() == 20 and cnt[20].item() == 45
