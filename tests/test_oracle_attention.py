"""Pins for the oracle's decode attention over the unified pages (reading M),
CPU only.

Each test ties it to something other than itself:
- a zero query reduces softmax to the uniform average of the dequantised values;
- a held token plus the step's new token has the two-token closed form;
- rows on exact integer grids dequantise exactly, so the output equals
  attention over the original bf16 rows, taken with scipy's softmax on the
  positions the prefill's classes keep (not from the pages);
- the page placement does not matter (a permuted free list gives the same bits);
- empty units and new-token-only units.

Source: DiffKV (arXiv 2412.03131), Figure 7 and section 6.1 (attention over the
mixed-precision unified pages); Pith review, "What carries the argument"
(significance is the average attention a token receives).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.decode_helpers import list_slots, slot_codes
from tests.oracle_helpers import bf16_to_f32, f16, run_oracle


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _attn(w, pool, tab, q, cap, scale=0.0883883476, k_new=None, v_new=None, new_lens=None, ctx=None):
    a = {"L": w.L, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "cap": cap, "layer0": 0, "n_layers": w.L,
         "q": _bits(q), "k_new": None if k_new is None else _bits(k_new),
         "v_new": None if v_new is None else _bits(v_new),
         "new_lens": None if new_lens is None else np.asarray(new_lens, np.int32),
         "ctx_lens": np.asarray(w.lens if ctx is None else ctx, np.int32), "scale": scale}
    st, out, p = oracle.decode_attention(a, pool, tab)
    assert st == oracle.OK
    return out, p


def _held_values(w, pool, tab, u):
    """Dequantised V rows and positions of a unit's held tokens, parsed from
    the page bytes by the test's own parser (fp32 fma emulated in fp64 then
    rounded once: exact, as c*s+z has at most 24+11 significant bits)."""
    vs, pos = [], []
    for li, high in ((0, True), (1, False)):
        n = int(tab.unit_hdr[u][li])
        for s in list_slots(pool.pages, tab.fwd[u], tab.unit_hdr[u], w.P)[li][:n]:
            _, vq, meta = slot_codes(s[:3], high)
            vsc, vz = f16(meta[2]).astype(np.float64), f16(meta[3]).astype(np.float64)
            vs.append((vq.astype(np.float64) * vsc + vz).astype(np.float32))
            pos.append(s[3])
    return np.array(vs, np.float64).reshape(-1, 128), pos


def test_zero_query_gives_uniform_weights_and_mean_value():
    w = W.small("att0", L=1, lens=[300, 7, 0, 129], Hq=6, Hkv=2)
    st, pool, tab = run_oracle(w, W.to_numpy(W.make_inputs(w, 3)))
    assert st == oracle.OK
    q = torch.zeros((1, w.R, w.Hq, 128), dtype=torch.bfloat16)
    out, p = _attn(w, pool, tab, q, cap=max(w.lens))
    G = w.Hq // w.Hkv
    for r in range(w.R):
        for qh in range(w.Hq):
            u = r * w.Hkv + qh // G
            v, pos = _held_values(w, pool, tab, u)
            if not pos:
                assert not out[0, r, qh].any() and not p[0, r * max(w.lens):(r + 1) * max(w.lens), qh].any()
                continue
            np.testing.assert_allclose(out[0, r, qh], v.mean(0), rtol=1e-12, atol=1e-12)
            row = p[0, r * max(w.lens):(r + 1) * max(w.lens), qh]
            np.testing.assert_allclose(row[pos], 1.0 / len(pos), rtol=1e-13)
            assert np.count_nonzero(row) == len(pos)


def _grid_inputs(w, seed):
    """Rows on exact integer grids: K8V4 tokens K in 0..255, V in 0..15; K4V2
    tokens K in 0..15, V in 0..3 (every row reaching both ends of its range,
    so scale 1 and zero 0); the class chosen by the significance sums: x10,
    x0.5 and x0.01 the threshold average, i.e. K8V4, K4V2, pruned."""
    inp = W.make_inputs(w, seed)
    g = torch.Generator().manual_seed(seed)
    T, Hkv = w.T, w.Hkv
    tier = torch.randint(0, 3, (T,), generator=g)  # 0 pruned, 1 K4V2, 2 K8V4
    kmax = torch.where(tier == 2, 255, 15)[:, None, None]
    vmax = torch.where(tier == 2, 15, 3)[:, None, None]
    k = (torch.rand((T, Hkv, 128), generator=g) * (kmax + 1)).floor().clamp(max=kmax)
    v = (torch.rand((T, Hkv, 128), generator=g) * (vmax + 1)).floor().clamp(max=vmax)
    k[:, :, 0], k[:, :, 1] = 0, kmax[:, :, 0]
    v[:, :, 0], v[:, :, 1] = 0, vmax[:, :, 0]
    inp["k"] = k[None].to(torch.bfloat16)
    inp["v"] = v[None].to(torch.bfloat16)
    lens = torch.tensor(w.lens)
    req = torch.repeat_interleave(torch.arange(w.R), lens)
    N = lens[req].to(torch.float32)
    f = torch.tensor([0.01, 0.5, 10.0])[tier]
    inp["sig_sum"] = (inp["sig_cnt"].to(torch.float32) * f * w.alpha_h / N)[None, :, None].expand(1, T, w.Hq).contiguous()
    return inp, tier


@pytest.mark.parametrize("with_new", [False, True])
def test_exact_grid_matches_attention_over_the_original_rows(with_new):
    w = W.small("attg", L=1, lens=[200, 33, 90, 1], Hq=8, Hkv=2, n_outlier=0)
    inp, tier = _grid_inputs(w, 11)
    st, pool, tab = run_oracle(w, W.to_numpy(inp))
    assert st == oracle.OK
    cls = tab.classes.reshape(w.T, w.Hkv)
    assert set(np.unique(cls)) == {0, 1, 2}
    q = W.decode_queries(w, 1, 5)
    scale = 1.0 / 512
    cap = max(w.lens) + 1
    kn = vn = None
    nl = [1, 0, 1, 1] if with_new else None
    if with_new:
        kn = torch.randint(-4, 5, (1, w.R, w.Hkv, 128), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
        vn = torch.randint(-4, 5, (1, w.R, w.Hkv, 128), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    out, p = _attn(w, pool, tab, q, cap, scale=scale, k_new=kn, v_new=vn, new_lens=nl)
    kf = bf16_to_f32(_bits(inp["k"][0])).astype(np.float64)
    vf = bf16_to_f32(_bits(inp["v"][0])).astype(np.float64)
    qf = bf16_to_f32(_bits(q[0])).astype(np.float64)
    G = w.Hq // w.Hkv
    start = np.concatenate([[0], np.cumsum(w.lens)[:-1]])
    for r in range(w.R):
        for qh in range(w.Hq):
            h = qh // G
            rows = start[r] + np.nonzero(cls[start[r]:start[r] + w.lens[r], h])[0]  # held positions
            K, V, pos = kf[rows, h], vf[rows, h], list(rows - start[r])
            if with_new and nl[r]:
                K = np.vstack([K, bf16_to_f32(_bits(kn[0, r, h]))[None].astype(np.float64)])
                V = np.vstack([V, bf16_to_f32(_bits(vn[0, r, h]))[None].astype(np.float64)])
                pos.append(w.lens[r])
            if len(pos) == 0:
                assert not out[0, r, qh].any()
                continue
            pw = softmax(scale * (K @ qf[r, qh]))
            np.testing.assert_allclose(out[0, r, qh], pw @ V, rtol=1e-12, atol=1e-12)
            row = p[0, r * cap:(r + 1) * cap, qh]
            np.testing.assert_allclose(row[pos], pw, rtol=1e-12, atol=1e-300)
            assert np.count_nonzero(row) == np.count_nonzero(pw)


def test_one_held_token_and_the_new_token_closed_form():
    """p_new = 1 / (1 + exp(l_held - l_new)) with both logits known exactly."""
    w = W.small("att2", L=1, lens=[1], Hq=2, Hkv=1, n_outlier=0)
    inp = W.make_inputs(w, 1)
    k = torch.zeros((1, 1, 1, 128))
    k[..., 0], k[..., 1] = 0.0, 255.0  # codes 0 and 255, scale 1: exact
    v = torch.zeros((1, 1, 1, 128))
    v[..., 1] = 15.0
    inp["k"], inp["v"] = k.to(torch.bfloat16), v.to(torch.bfloat16)
    inp["sig_sum"] = torch.full((1, 1, 2), 10.0)
    st, pool, tab = run_oracle(w, W.to_numpy(inp))
    assert st == oracle.OK and tab.unit_hdr[0][0] == 1
    q = torch.zeros((1, 1, 2, 128))
    q[0, 0, 0, 1] = 0.5    # held logit 0.5 * 255 * scale; new logit 0.5 * 2 * scale
    q[0, 0, 1, 1] = -1.0
    kn = torch.zeros((1, 1, 1, 128))
    kn[..., 1] = 2.0
    vn = torch.zeros((1, 1, 1, 128))
    vn[..., 0] = 3.0
    scale = 1.0 / 64
    out, p = _attn(w, pool, tab, q.to(torch.bfloat16), cap=2, scale=scale, k_new=kn.to(torch.bfloat16),
                   v_new=vn.to(torch.bfloat16), new_lens=[1], ctx=[1])
    for qh, qq in ((0, 0.5), (1, -1.0)):
        ph = 1.0 / (1.0 + np.exp(scale * qq * (2.0 - 255.0)))  # weight of the held token
        np.testing.assert_allclose(p[0, :2, qh], [ph, 1.0 - ph], rtol=1e-14)
        np.testing.assert_allclose(out[0, 0, qh, :2], [3.0 * (1 - ph), 15.0 * ph], rtol=1e-14)
        assert not out[0, 0, qh, 2:].any()


def test_page_placement_does_not_matter():
    w = W.small("attp", L=2, lens=[300, 7, 517, 0, 129])
    n = W.to_numpy(W.make_inputs(w, 4))
    st, pool_a, tab_a = run_oracle(w, n)
    pool_b = oracle.Pool(w.pool_pages, w.P)
    pool_b.free_list[:] = np.random.default_rng(0).permutation(w.pool_pages).astype(np.int32)
    st2, pool_b, tab_b = run_oracle(w, n, pool=pool_b)
    assert st == st2 == oracle.OK and not np.array_equal(tab_a.fwd, tab_b.fwd)
    q = W.decode_queries(w, 2, 9)
    oa, pa = _attn(w, pool_a, tab_a, q, cap=517)
    ob, pb = _attn(w, pool_b, tab_b, q, cap=517)
    assert np.array_equal(oa, ob) and np.array_equal(pa, pb)
    # probabilities sum to one per attended (layer, request, query head)
    sums = pa.reshape(2, w.R, 517, w.Hq).sum(2)
    for r, n_r in enumerate(w.lens):
        if n_r:
            np.testing.assert_allclose(sums[:, r], 1.0, rtol=1e-13)


def test_empty_unit_and_new_token_only():
    """A request holding nothing attends to nothing (zero output), or only to
    its new token (weight 1, output = its V)."""
    w = W.small("atte", L=1, lens=[0, 5], Hq=2, Hkv=1)
    st, pool, tab = run_oracle(w, W.to_numpy(W.make_inputs(w, 2)))
    assert st == oracle.OK
    q = W.decode_queries(w, 1, 1)
    out, p = _attn(w, pool, tab, q, cap=8)
    assert not out[0, 0].any() and not p[0, :8].any()
    kn = W.decode_queries(W.small("x", L=1, lens=[0, 5], Hq=1, Hkv=1), 1, 2)
    vn = W.decode_queries(W.small("x", L=1, lens=[0, 5], Hq=1, Hkv=1), 1, 3)
    out, p = _attn(w, pool, tab, q, cap=8, k_new=kn, v_new=vn, new_lens=[1, 0])
    np.testing.assert_array_equal(out[0, 0, 0], bf16_to_f32(_bits(vn[0, 0, 0])))
    np.testing.assert_array_equal(p[0, 0, :], [1.0, 1.0])
