"""Test-side helpers for decode attention: a vectorised parser of a unit's
held tokens from raw page bytes (codes, fp16 scale / zero, positions), and the
error bound the GPU's fp32 attention is held to against the oracle's double
result.  No attention is computed here."""
from __future__ import annotations

import numpy as np

from tests.oracle_helpers import Layout, unpack

U = 2.0 ** -24  # fp32 unit roundoff


def unit_tokens(pages: np.ndarray, fwd_row: np.ndarray, hdr, P: int, scheme: int = 0):
    """Held tokens of a unit in list order (high list, then low list):
    (K codes [n,128], V codes [n,128], k_s, k_z, v_s, v_z [n] float64,
    positions [n] int64).  `pages` is indexable by the forward row's ids; the
    page layout and code widths are those of the bit-width scheme."""
    lay = Layout(P, scheme)
    n_hi, n_lo, p_hi, p_lo = (int(x) for x in hdr)
    parts = []
    for n, ids, per, high in ((n_hi, fwd_row[:p_hi], P, True), (n_lo, fwd_row[p_hi:p_hi + p_lo], 2 * P, False)):
        if n == 0:
            continue
        kb, vb = lay.kbits(high), lay.vbits(high)
        pg = np.stack([pages[int(i)] for i in ids])                     # [pages, page bytes]
        kbytes = 16 * kb
        vbytes = 16 * vb
        vbase = lay.v_off(high, 0)
        kc = pg[:, :per * kbytes].reshape(-1, kbytes)[:n]
        vc = pg[:, vbase:vbase + per * vbytes].reshape(-1, vbytes)[:n]
        meta = pg[:, lay.meta:lay.meta + 8 * per].reshape(-1, 8)[:n].copy().view(np.uint16)
        pos = pg[:, lay.pos:lay.pos + 4 * per].reshape(-1, 4)[:n].copy().view(np.int32)[:, 0]
        kq = unpack(kc.reshape(-1), kb).reshape(n, 128)
        vq = unpack(vc.reshape(-1), vb).reshape(n, 128)
        m = meta.view(np.float16).astype(np.float64)
        parts.append((kq, vq, m[:, 0], m[:, 1], m[:, 2], m[:, 3], pos.astype(np.int64)))
    if not parts:
        z = np.zeros((0, 128), np.uint8)
        e = np.zeros(0)
        return z, z, e, e, e, e, np.zeros(0, np.int64)
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(7))


def attention_bounds(q: np.ndarray, scale: float, toks, new_kv, p: np.ndarray):
    """Error bounds of the GPU's fp32 decode attention of one query head.

    q: [128] float64 (the bf16 query); toks: unit_tokens(...) of its KV head;
    new_kv: None or (k [128], v [128]) float64 of the new token (attended
    last); p: the oracle's probabilities in the same order.
    Returns (bound on |out - out_oracle| per channel [128], bound on
    |p_gpu - p| per token [n]).

    The model (u = 2^-24): a logit is a sum of at most 16 fused products per
    lane, a butterfly of at most 4 additions, then s*(q.c) + z*(sum q) and the
    scale, so |dl_t| <= 32 u scale sum_d |q_d| (c_td s_t + |z_t|) (|q_d||k_d|
    for the new token); exp(l - M) adds u |l - M| + 2 ulp; the denominator and
    the outputs are fp32 sums of at most n + 32 terms.  The relative error of
    p_t is then rho_t = expm1(eta_t) + expm1(sum_s p_s eta_s) + (n + 16) u with
    eta_t = |dl_t| + u |l_t - M| + 2^-19 (the exponential and up to six
    rescalings of running sums by exponential factors), and the output error is
    sum_t p_t (rho_t + (n + 32) u) (c_td s_vt + |z_vt|).  Both bounds are
    doubled to cover second-order terms."""
    kq, vq, ks, kz, vs, vz, _ = toks
    qa = np.abs(q)
    kabs = (kq.astype(np.float64) * ks[:, None] + np.abs(kz)[:, None]) @ qa
    vabs = vq.astype(np.float64) * vs[:, None] + np.abs(vz)[:, None]
    if new_kv is not None:
        kabs = np.append(kabs, np.abs(new_kv[0]) @ qa)
        vabs = np.vstack([vabs, np.abs(new_kv[1])[None]])
    n = kabs.size
    if n == 0:
        return np.zeros(128), np.zeros(0)
    dl = 32 * U * scale * kabs
    with np.errstate(divide="ignore"):
        lm = np.where(p > 0, -np.log(np.where(p > 0, p, 1.0) / p.max()), 200.0)
    eta = dl + U * np.minimum(lm, 200.0) + 2.0 ** -19  # exp, and up to 6 rescales by exp factors
    rho = np.expm1(eta) + np.expm1(float(p @ eta)) + (n + 16) * U
    out_b = 2.0 * ((p * (rho + (n + 32) * U)) @ vabs)
    return out_b, 2.0 * rho * p


def prefill_bounds(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """Error bounds of the GPU's causal prefill attention of one (request,
    query head): q [n][128], k, v [n][128] float64 (the bf16 values).

    Products of bf16 values are exact; the logits are fp32 sums of 128 of them
    on the tensor cores: |dl_ij| <= 64 u scale sum_d |q_id| |k_jd|.  The
    kernel forms p = 2^(s scale log2e - (m_i + log2 l_i)) with one rounded
    multiply-add: the exponent adds u |ln p_ij| + u |lse_i| + 2^-23 ln l_i
    (lse_i = m_i + ln l_i, natural units).  The probabilities then carry
    rho_ij as in attention_bounds (exponential, normaliser); the outputs are fp32 sums over n keys of p rounded to bf16
    (relative error at most 2^-8 more) times the bf16 v, and a significance
    sum adds n fp32 probabilities in fp32 (atomics in any order).
    Returns (bound on |out| errors [n][128], bound on |sig_sum| errors [n],
    the probabilities p [n][n] in double)."""
    n = q.shape[0]
    if n == 0:
        return np.zeros((0, 128)), np.zeros(0), np.zeros((0, 0))
    lg = scale * (q @ k.T)
    mask = np.tril(np.ones((n, n), dtype=bool))
    lg = np.where(mask, lg, -np.inf)
    mx = lg.max(1, keepdims=True)
    e = np.exp(lg - mx)
    p = e / e.sum(1, keepdims=True)
    dl = 64 * U * scale * (np.abs(q) @ np.abs(k).T)
    lsum = e.sum(1, keepdims=True)
    lse = mx + np.log(lsum)  # the row's normaliser, natural log
    with np.errstate(invalid="ignore", divide="ignore"):
        # the exponent s scale log2e - (m + log2 l): rounded once (u |ln p|),
        # plus the rounding of m + log2 l (u |lse|) and of log2 l (2 ulp)
        eta = np.where(mask, dl + U * np.minimum(lse - lg, 200.0) + U * np.abs(lse) + 2.0 ** -23 * np.log(lsum)
                       + 2.0 ** -19, 0.0)
    rho = np.expm1(eta) + np.expm1((p * eta).sum(1, keepdims=True)) + (n + 16) * U
    rho = np.where(mask, rho, 0.0)
    out_b = 2.0 * ((p * (rho + (n + 32) * U + 2.0 ** -8)) @ np.abs(v) + 2.0 ** -24)
    sig_b = 2.0 * ((p * rho).sum(0) + (n + 8) * U * p.sum(0))
    return out_b, sig_b, p
