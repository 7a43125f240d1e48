"""Pins for the oracle's prefill attention with significance accumulation
(reading S), CPU only.

- A zero query makes the causal softmax uniform: p(i, j) = 1 / (i + 1), so a
  key's significance sum is the harmonic difference H_n - H_j and each output
  is the mean of the values so far.
- Two tokens have the logistic closed form.
- On the tiny configuration the significance sums equal the input generator's
  own fp64 causal-softmax computation (torch), given the same bf16 queries.
- Every query's probabilities sum to one, so a request's significance sums add
  up to its length.

Source: DiffKV (arXiv 2412.03131), Pith review, "What carries the argument"
(significance is the average attention a token receives from the tokens after
it) and Referee Report, major comment 2 (the average is over N - i scores).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.oracle_helpers import bf16_to_f32

SCALE = 1.0 / math.sqrt(128)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _kv(w, seed):
    k = torch.stack([W.make_kv_layer(w, seed, l, 0) for l in range(w.L)])
    v = torch.stack([W.make_kv_layer(w, seed, l, 1) for l in range(w.L)])
    return k, v


def test_zero_query_harmonic_closed_form():
    w = W.small("pa0", L=1, lens=[37, 1, 0, 12], Hq=4, Hkv=2)
    k, v = _kv(w, 3)
    q = torch.zeros((1, w.T, w.Hq, 128), dtype=torch.bfloat16)
    st, out, sig, cnt = oracle.prefill_attention(_bits(q), _bits(k), _bits(v), w.lens, SCALE)
    assert st == oracle.OK
    vf = bf16_to_f32(_bits(v)).astype(np.float64)
    G = w.Hq // w.Hkv
    start = 0
    for n in w.lens:
        H = [math.fsum(1.0 / m for m in range(1, i + 1)) for i in range(n + 1)]
        for j in range(n):
            assert cnt[start + j] == n - j
            np.testing.assert_allclose(sig[0, start + j], H[n] - H[j], rtol=1e-13)
        for qh in range(w.Hq):
            prefix = np.cumsum(vf[0, start:start + n, qh // G], axis=0) / np.arange(1, n + 1)[:, None]
            np.testing.assert_allclose(out[0, start:start + n, qh], prefix, rtol=1e-12, atol=1e-13)
        start += n


def test_two_tokens_logistic():
    w = W.small("pa2", L=1, lens=[2], Hq=1, Hkv=1, n_outlier=0)
    k = torch.zeros((1, 2, 1, 128))
    k[0, 0, 0, 0], k[0, 1, 0, 0] = 3.0, -1.0
    v = torch.zeros((1, 2, 1, 128))
    v[0, 0, 0, 5], v[0, 1, 0, 5] = 2.0, 7.0
    q = torch.zeros((1, 2, 1, 128))
    q[0, :, 0, 0] = 0.5
    st, out, sig, cnt = oracle.prefill_attention(_bits(q.to(torch.bfloat16)), _bits(k.to(torch.bfloat16)),
                                                 _bits(v.to(torch.bfloat16)), w.lens, 0.25)
    assert st == oracle.OK
    p10 = 1.0 / (1.0 + math.exp(0.25 * 0.5 * (-1.0 - 3.0)))  # query 1's weight on key 0
    np.testing.assert_allclose(sig[0, :, 0], [1.0 + p10, 1.0 - p10], rtol=1e-14)
    np.testing.assert_allclose(out[0, 0, 0, 5], 2.0, rtol=1e-15)
    np.testing.assert_allclose(out[0, 1, 0, 5], 2.0 * p10 + 7.0 * (1.0 - p10), rtol=1e-14)
    assert list(cnt) == [2, 1]


def test_tiny_significance_equals_the_generators_softmax(monkeypatch):
    w = W.get("tiny")
    k, v = _kv(w, W.SEED_BASE)
    q32 = W.make_queries(w, W.SEED_BASE, 0)
    qb = q32.to(torch.bfloat16)
    monkeypatch.setattr(W, "make_queries", lambda w_, s_, l_: qb.to(torch.float32))
    want = W._softmax_sig_layer(w, W.SEED_BASE, 0, "cpu", k[0]).to(torch.float64).numpy()
    st, out, sig, cnt = oracle.prefill_attention(_bits(qb[None]), _bits(k), _bits(v), w.lens, SCALE)
    assert st == oracle.OK
    # the generator rounds its fp64 sums to fp32 once
    np.testing.assert_allclose(sig[0], want, rtol=2.0 ** -23, atol=1e-30)
    assert np.array_equal(cnt, W.sig_cnt_prefill(w).numpy())


def test_significance_mass_is_the_number_of_queries():
    w = W.small("pam", L=2, lens=[300, 7, 129], Hq=6, Hkv=2)
    k, v = _kv(w, 5)
    q = torch.randn((2, w.T, 6, 128), generator=torch.Generator().manual_seed(4))
    st, out, sig, cnt = oracle.prefill_attention(_bits(q.to(torch.bfloat16)), _bits(k), _bits(v), w.lens, SCALE)
    assert st == oracle.OK
    start = 0
    for n in w.lens:
        np.testing.assert_allclose(sig[:, start:start + n].sum(1), float(n), rtol=1e-12)
        start += n
