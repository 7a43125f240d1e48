"""Hand-built bf16 token rows that drive the per-token quantiser into its edge
cases, and batches made of them.

Input design only: nothing here quantises.  Rows are built from exact
grids (zero point z and a power-of-two step s, so every value below is exact
in bf16 and every quotient (x - z) / s is exact in fp32), so the quantiser's
result on them has a plain closed form the oracle pins check (ties to even,
clamping, scale underflow).  The same rows are fed to the CUDA path and to
the oracle, and the tests compare every byte.

Row kinds (each 128 channels, channel order shuffled):
  tie8 / tie4 / tie2   the end points z and z + n s plus points z + (k + 1/2) s
                       exactly half way between two codes of that width
  near8 / near4        the tie points moved one bf16 ulp up or down
  grid8 / grid4 / grid2 the exact grid z + k s
  const                one value repeated (scale 0), including -0 and +-65280
  underflow            span / n below half the smallest binary16 subnormal:
                       the scale is raised to 2^-24
  clamp                span / n just above 2^-24 rounds down to 2^-24: the top
                       codes need clamping
  subnormal_min        a minimum inside the binary16 subnormal range that
                       binary16 does not hold exactly (z != min)
  fp16_max             rows that reach -65280 and / or 65280, the bf16 values
                       nearest the binary16 limit 65504 (bf16 holds no 65504)
  signed_zero          -0 and +0 as the extremes
  scaled               N(0,1) rows times 2^e, e from -30 to 13
"""
from __future__ import annotations

import numpy as np
import torch

from differentiated_kv_cache_dkv_gb300 import workloads as W


def bf16_bits_exact(x) -> np.ndarray:
    """bf16 bit patterns of float32 values that bf16 holds exactly."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def bf16_bits_rne(x) -> np.ndarray:
    """bf16 bit patterns of float32 values, rounded to nearest even."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _is_bf16(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, dtype=np.float32).view(np.uint32) & 0xFFFF) == 0


def _fill(vals: np.ndarray, fixed: list, rng) -> np.ndarray:
    """128 values: `fixed` first, the rest drawn from `vals`, shuffled."""
    out = np.empty(128, dtype=np.float32)
    out[:len(fixed)] = fixed
    out[len(fixed):] = rng.choice(vals, size=128 - len(fixed))
    return rng.permutation(out)


def tie_row(b: int, z: float, s: float, rng) -> np.ndarray:
    n = (1 << b) - 1
    k = np.arange(n)
    cand = (np.float64(z) + (k + 0.5) * s).astype(np.float32)
    cand = cand[_is_bf16(cand)]
    assert cand.size > 0
    return _fill(cand, [z, z + n * s], rng)


def grid_row(b: int, z: float, s: float, rng) -> np.ndarray:
    n = (1 << b) - 1
    cand = (np.float64(z) + np.arange(n + 1) * s).astype(np.float32)
    cand = cand[_is_bf16(cand)]
    return _fill(cand, [z, z + n * s], rng)


def near_row(b: int, z: float, s: float, rng) -> np.ndarray:
    """Tie points moved one bf16 ulp towards or away from zero."""
    row = tie_row(b, z, s, rng)
    bits = bf16_bits_exact(row).astype(np.int32)
    step = rng.choice([-1, 1], size=128)
    mid = (row != np.float32(z)) & (row != np.float32(z + ((1 << b) - 1) * s)) & (row != 0)
    bits = np.where(mid, bits + step, bits)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def kinds(rng) -> dict:
    """{name: [row values float32 [128], ...]} for every edge kind."""
    out = {}
    out["tie8"] = [tie_row(8, -1.0, 2.0 ** -5, rng), tie_row(8, 0.0, 2.0 ** -9, rng),
                   tie_row(8, -3.0, 2.0 ** -4, rng)]
    out["tie4"] = [tie_row(4, -0.5, 2.0 ** -3, rng), tie_row(4, 0.125, 2.0 ** -6, rng),
                   tie_row(4, -96.0, 8.0, rng)]
    out["tie2"] = [tie_row(2, 0.25, 2.0 ** -2, rng), tie_row(2, -1.5, 1.0, rng), tie_row(2, 0.0, 2.0 ** -12, rng)]
    out["near8"] = [near_row(8, -1.0, 2.0 ** -5, rng)]
    out["near4"] = [near_row(4, -0.5, 2.0 ** -3, rng), near_row(2, 0.25, 2.0 ** -2, rng)]
    out["grid8"] = [grid_row(8, -1.0, 2.0 ** -5, rng)]
    out["grid4"] = [grid_row(4, -0.5, 2.0 ** -3, rng)]
    out["grid2"] = [grid_row(2, 4.0, 2.0, rng)]
    out["const"] = [np.full(128, c, dtype=np.float32) for c in (0.0, -0.0, 1.5, -65280.0, 65280.0, 2.0 ** -20, -3.0)]
    under = np.full(128, 2.0 ** -12, dtype=np.float32)
    under[rng.integers(128)] = np.float32(2.0 ** -12 + 2.0 ** -19)  # the next bf16 above: span 2^-19
    out["underflow"] = [under]
    # span 356 * 2^-24: span / 255 = 1.396 * 2^-24 rounds to 2^-24, so codes
    # above 255 would be needed; multiples of 2^-24 keep every value exact
    clamp = (rng.integers(0, 357, size=128) * 2.0 ** -24).astype(np.float32)
    clamp[:2] = [0.0, 356 * 2.0 ** -24]
    clamp = np.where(_is_bf16(clamp), clamp, np.float32(0.0))
    out["clamp"] = [rng.permutation(clamp)]
    # minimum -(2^-20 + 2^-27): binary16 holds only multiples of 2^-24 there
    sub = np.float32(-(2.0 ** -20 + 2.0 ** -27))
    vals = (sub + rng.integers(0, 64, size=128) * 2.0 ** -22).astype(np.float32)
    vals = np.where(_is_bf16(vals), vals, sub)
    vals[0] = sub
    out["subnormal_min"] = [rng.permutation(vals)]
    wide = bf16_bits_rne(rng.uniform(-65504.0, 65504.0, size=128).astype(np.float32))
    wide = (wide.astype(np.uint32) << 16).view(np.float32)
    wide = np.clip(wide, -65280.0, 65280.0).astype(np.float32)
    wide[:2] = [-65280.0, 65280.0]
    top = _fill(np.array([65280.0, 65024.0, 64768.0, 64512.0], dtype=np.float32), [65280.0, 64512.0], rng)
    bot = _fill(np.array([-65280.0, -65024.0, -1.0], dtype=np.float32), [-65280.0], rng)
    out["fp16_max"] = [rng.permutation(wide), top, bot]
    sz1 = _fill(np.array([0.0, 0.5, 0.25, 1.0], dtype=np.float32), [-0.0, 0.0, 1.0], rng)        # min -0 / +0
    sz2 = _fill(np.array([-0.0, -0.75, -2.0], dtype=np.float32), [-0.0, 0.0, -2.0], rng)         # max +0 / -0
    sz3 = rng.permutation(np.where(rng.random(128) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32))
    sz4 = np.full(128, -0.0, dtype=np.float32)
    sz4[rng.integers(128)] = np.float32(2.0 ** -30)
    out["signed_zero"] = [sz1, sz2, sz3, sz4]
    scaled = []
    for e in (-30, -24, -20, -16, -14, -12, -3, 0, 6, 13):
        x = rng.standard_normal(128).astype(np.float32) * np.float32(2.0 ** e)
        x = (bf16_bits_rne(np.clip(x, -65280.0, 65280.0)).astype(np.uint32) << 16).view(np.float32)
        scaled.append(x.astype(np.float32))
    out["scaled"] = scaled
    for name, rows in out.items():
        for r in rows:
            assert r.shape == (128,) and _is_bf16(r).all() and np.all(np.abs(r) <= 65504.0), name
    return out


def all_rows(rng) -> list:
    """Every edge row once, as (kind, float32 values)."""
    return [(k, r) for k, rows in kinds(rng).items() for r in rows]


def edge_batch(lens, Hq: int, Hkv: int, seed: int = 0, L: int = 1, P: int = 16,
               class_mix=(0.45, 0.35, 0.20)):
    """A prefill batch whose K and V rows are all edge rows (every kind appears
    in K and in V, at both classes), with significance sums that put each
    token row in a chosen class at alpha_h = 1, alpha_l = 0.2: scores 4/N
    (K8V4), 0.5/N (K4V2) or 0.02/N (pruned).

    Returns (workload, inputs as torch tensors on the CPU, the class each row
    was aimed at [L][T][Hkv])."""
    rng = np.random.default_rng(seed)
    w = W.small("edges", L=L, Hq=Hq, Hkv=Hkv, lens=list(lens), P=P, alpha_h=1.0, alpha_l=0.2)
    rows = all_rows(rng)
    T = w.T
    nrow = L * T * Hkv
    pick_k = np.concatenate([rng.permutation(len(rows)) for _ in range(-(-nrow // len(rows)))])[:nrow]
    pick_v = np.concatenate([rng.permutation(len(rows)) for _ in range(-(-nrow // len(rows)))])[:nrow]
    kx = np.stack([rows[i][1] for i in pick_k]).reshape(L, T, Hkv, 128)
    vx = np.stack([rows[i][1] for i in pick_v]).reshape(L, T, Hkv, 128)
    aim = rng.choice([2, 1, 0], size=(L, T, Hkv), p=list(class_mix)).astype(np.uint8)
    level = np.where(aim == 2, 4.0, np.where(aim == 1, 0.5, 0.02))
    N = np.repeat(np.array(w.lens, dtype=np.float64), w.lens)           # [T]
    cnt = W.sig_cnt_prefill(w).numpy().astype(np.float64)             # [T]
    G = Hq // Hkv
    sig = np.repeat(level / N[None, :, None] * cnt[None, :, None], G, axis=2).astype(np.float32)
    to_t = lambda a: torch.from_numpy(bf16_bits_exact(a).view(np.int16).copy()).view(torch.bfloat16)  # noqa: E731
    inp = {"L": L, "R": w.R, "Hq": Hq, "Hkv": Hkv, "T": T, "k": to_t(kx), "v": to_t(vx),
           "sig_sum": torch.from_numpy(sig), "sig_cnt": W.sig_cnt_prefill(w),
           "lens": torch.tensor(w.lens, dtype=torch.int32)}
    return w, inp, aim


def new_token_rows(L: int, R: int, Hkv: int, seed: int) -> tuple:
    """bf16 [L][R][Hkv][128] K and V of new tokens, drawn from the edge rows."""
    rng = np.random.default_rng(seed)
    rows = all_rows(rng)
    n = L * R * Hkv
    kx = np.stack([rows[i][1] for i in rng.integers(0, len(rows), size=n)]).reshape(L, R, Hkv, 128)
    vx = np.stack([rows[i][1] for i in rng.integers(0, len(rows), size=n)]).reshape(L, R, Hkv, 128)
    to_t = lambda a: torch.from_numpy(bf16_bits_exact(a).view(np.int16).copy()).view(torch.bfloat16)  # noqa: E731
    return to_t(kx), to_t(vx)


def dequant_bound(s: np.ndarray, nbits: int, span=0.0) -> np.ndarray:
    """Largest |x - (z + q s)| the quantiser allows for a row of scale s
    (float64, elementwise), derived from its fp32 arithmetic:
      - rounding x - z and the quotient by s moves t = (x - z) / s by at most
        (n + 1/2) 2^-23 for t <= n + 1/2, so a code is off its real value by at
        most 1/2 + (n + 1/2) 2^-23;
      - a binary16 subnormal scale (s < 2^-14) can round down from (max -
        min) / n by up to 2^-25, and a subnormal minimum can round by up to
        2^-25, so the top codes may clamp: up to (n + 1) 2^-25 more;
      - a scale lowered from infinity to 65504 (1-bit codes of a span above
        65519: `span` = max - min of the row) clamps the top codes: up to
        span - n s more;
      - 1e-6 absolute, as the method states its bound.
    """
    n = (1 << nbits) - 1
    s = np.asarray(s, dtype=np.float64)
    b = s * (0.5 + (n + 0.5) * 2.0 ** -23) + 1e-6
    b = b + np.maximum(0.0, np.asarray(span, dtype=np.float64) - n * s)
    return b + np.where(s < 2.0 ** -14, (n + 1) * 2.0 ** -25, 0.0)
