"""Prefill attention at the full Llama shape (32 layers, 16 requests of 4096
tokens, 32 query / 8 KV heads), in the launch configuration the bench times:
one dkv_prefill_attention over every layer.

Checked on every output:
- the counts are exactly N - i;
- every output is finite;
- each query row's probabilities sum to 1, so the significance sums of a
  (layer, request, query head) add up to the request's length (in fp32, to a
  relative 1e-4).
Checked against the oracle's double-precision result, inside the bound
derived from the kernel's fp32 arithmetic (tests/attention_helpers.py), on
whole (layer, request, query head) slices: every output row and every
significance sum of the slice, the oracle running on that slice alone (keys
and queries of one request, one head pair)."""
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
SLICES = [(0, 0, 0), (31, 15, 31), (17, 6, 9)]  # (layer, request, query head)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def test_prefill_attention_full_llama():
    w = W.get("llama")
    dev = torch.device("cuda", 0)
    seed = W.SEED_BASE + 77
    k = torch.empty((w.L, w.T, w.Hkv, 128), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    q = torch.empty((w.L, w.T, w.Hq, 128), dtype=torch.bfloat16, device=dev)
    for l in range(w.L):
        k[l] = W.make_kv_layer(w, seed, l, 0, dev)
        v[l] = W.make_kv_layer(w, seed, l, 1, dev)
        q[l] = W.prefill_queries(w, seed, l, dev)
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    out = torch.full((w.L, w.T, w.Hq, 128), float("nan"), dtype=torch.float32, device=dev)
    sig = torch.full((w.L, w.T, w.Hq), float("nan"), dtype=torch.float32, device=dev)
    cnt = torch.full((w.T,), -5, dtype=torch.int32, device=dev)
    pool = libdkv.DevicePool(1, 16, dev)
    libdkv.dkv_init_pool(pool)
    libdkv.dkv_prefill_attention(q, k, v, lens, max(w.lens), SCALE, out, sig, cnt, pool)
    torch.cuda.synchronize()
    st = libdkv.dkv_get_status(pool)
    assert st == libdkv.DKV_OK, libdkv.status_string(st)

    # counts, finiteness and probability mass, over everything
    starts = np.concatenate([[0], np.cumsum(w.lens)])
    want_cnt = np.concatenate([np.arange(n, 0, -1) for n in w.lens]).astype(np.int32)
    assert np.array_equal(cnt.cpu().numpy(), want_cnt)
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(sig).all())
    for r, n in enumerate(w.lens):
        mass = sig[:, starts[r]:starts[r] + n, :].double().sum(dim=1)  # [L][Hq]
        assert torch.allclose(mass, torch.full_like(mass, float(n)), rtol=1e-4, atol=0), (r, n)

    # whole slices against the oracle
    G = w.Hq // w.Hkv
    for l, r, qh in SLICES:
        n = w.lens[r]
        sl = slice(int(starts[r]), int(starts[r]) + n)
        qs = q[l, sl, qh:qh + 1].unsqueeze(0)                 # [1][n][1][128]
        ks = k[l, sl, qh // G:qh // G + 1].unsqueeze(0)
        vs = v[l, sl, qh // G:qh // G + 1].unsqueeze(0)
        rc, o_ref, s_ref, c_ref = oracle.prefill_attention(_bits(qs), _bits(ks), _bits(vs), [n], SCALE)
        assert rc == oracle.OK
        ob, sb, _ = prefill_bounds(bf16_to_f32(_bits(qs[0, :, 0])).astype(np.float64),
                                   bf16_to_f32(_bits(ks[0, :, 0])).astype(np.float64),
                                   bf16_to_f32(_bits(vs[0, :, 0])).astype(np.float64), SCALE)
        eo = np.abs(out[l, sl, qh].cpu().numpy().astype(np.float64) - o_ref[0, :, 0])
        es = np.abs(sig[l, sl, qh].cpu().numpy().astype(np.float64) - s_ref[0, :, 0])
        assert np.all(eo <= ob), (l, r, qh, float(eo.max()), float(ob.max()))
        assert np.all(es <= sb), (l, r, qh, float(es.max()), float(sb.max()))
