"""GPU parity of the prefill classification on its edge cases, for every
kernel that classifies: the per-token kernels of the common head shapes
(Hq, G) = (32, 4), (28, 7), (40, 5), (64, 8), (12, 4) and the staged kernel
(G = 4 with Hq = 8, G = 3 with Hq = 6).

DiffKV, Pith review, "What carries the argument": a token's significance is
the average attention it receives from later tokens, max-aggregated over the
query heads of its KV head, compared with alpha_h / N and alpha_l / N; a
count of 0 keeps the token K8V4.  Planted on top of the seeded inputs:
- counts of 0, and negative counts (the reduce takes the smallest sum then);
- summed scores a few ulps either side of n * thr for both thresholds, where
  the kernels' reciprocal test must hand over to the IEEE division;
- NaN (some or all of a head's query heads), +-inf, signed zeros, 3e38;
- thresholds below 2^-100 (alpha 1e-28 / 1e-31), decided by division only.
Everything is compared bit for bit with the oracle: classes, tables, cursors,
every live page.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.gpu_helpers import assert_same_state, fetch, make_compactor, oracle_state, to_device
from tests.oracle_helpers import run_oracle

pytestmark = pytest.mark.gpu

LENS = [300, 7, 517, 0, 129, 128]
SHAPES = [
    dict(Hq=32, Hkv=8), dict(Hq=28, Hkv=4), dict(Hq=40, Hkv=8), dict(Hq=64, Hkv=8),
    dict(Hq=12, Hkv=3), dict(Hq=8, Hkv=2), dict(Hq=6, Hkv=2),
]


def _ulps(x: np.float32, k: int) -> np.float32:
    d = np.float32(np.inf) if k > 0 else np.float32(-np.inf)
    for _ in range(abs(k)):
        x = np.nextafter(x, d, dtype=np.float32)
    return np.float32(x)


def plant_edges(w: W.Workload, inp: dict, alpha_h: float, alpha_l: float, seed: int) -> dict:
    """Edge values written over a seeded sample of tokens (about a third, plus
    the first and last token of every request and the tokens either side of
    each 128-token tile boundary)."""
    rng = np.random.default_rng(seed)
    sig = inp["sig_sum"].numpy().copy()   # [L][T][Hq]
    cnt = inp["sig_cnt"].numpy().copy()   # [T]
    G = w.Hq // w.Hkv
    starts = np.concatenate([[0], np.cumsum(w.lens)])
    for r, N in enumerate(w.lens):
        if N == 0:
            continue
        s0 = int(starts[r])
        toks = set(rng.choice(N, size=max(1, N // 3), replace=False).tolist())
        toks |= {0, N - 1} | {b + d for b in range(128, N, 128) for d in (-1, 0) if 0 <= b + d < N}
        thr = [np.float32(alpha_h) / np.float32(N), np.float32(alpha_l) / np.float32(N)]
        for i in sorted(toks):
            t = s0 + i
            kind = int(rng.integers(0, 8))
            if kind == 0:
                cnt[t] = 0
                continue
            if kind == 1:
                cnt[t] = -int(rng.integers(1, 9))
                sig[:, t, :] = rng.standard_normal((w.L, w.Hq)).astype(np.float32) * np.float32(1.0 / N)
                continue
            n = int(cnt[t])
            for l in range(w.L):
                for h in range(w.Hkv):
                    grp = sig[l, t, h * G:(h + 1) * G]
                    if kind in (2, 3):       # max a few ulps from n * thr
                        base = np.float32(thr[kind - 2] * np.float32(n))
                        top = _ulps(base, int(rng.integers(-3, 4)))
                        grp[:] = np.minimum(grp, top)
                        grp[int(rng.integers(0, G))] = top
                    elif kind == 4:          # NaN in some or all of the group
                        m = rng.random(G) < (1.0 if h % 2 else 0.5)
                        grp[m] = np.nan
                    elif kind == 5:
                        grp[int(rng.integers(0, G))] = np.inf if rng.random() < 0.5 else -np.inf
                    elif kind == 6:
                        grp[:] = np.where(rng.random(G) < 0.5, np.float32(0.0), np.float32(-0.0))
                    else:
                        grp[int(rng.integers(0, G))] = np.float32(3e38)
    out = dict(inp)
    out["sig_sum"] = torch.from_numpy(sig)
    out["sig_cnt"] = torch.from_numpy(cnt)
    return out


@pytest.mark.parametrize("alphas", [(1.0, 0.2), (1e-28, 1e-31)], ids=["plain", "tiny"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"hq{s['Hq']}-hkv{s['Hkv']}" for s in SHAPES])
def test_classification_edges_bit_exact(shape, alphas):
    w = W.small("edges", L=2, lens=LENS, P=16, **shape)
    ah, al = alphas
    inp = plant_edges(w, W.make_inputs(w, seed=31), ah, al, seed=shape["Hq"] * 7 + shape["Hkv"])
    comp = make_compactor(w)
    pool = oracle.Pool(comp.pool.F, w.P)
    comp.compact(to_device(inp), ah, al)
    st = libdkv.dkv_get_status(comp.pool)
    so, pool, tab = run_oracle(w, W.to_numpy(inp), ah, al, pool=pool)
    assert st == so == oracle.OK
    gpu = fetch(comp)
    assert_same_state(gpu, oracle_state(pool, tab))
    # the planted edges reach every class
    cls = gpu["classes"].reshape(-1)[: w.L * w.T * w.Hkv]
    assert set(np.unique(cls).tolist()) <= {0, 1, 2}
