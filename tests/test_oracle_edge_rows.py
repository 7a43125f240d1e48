"""Pins for the oracle's quantiser on hand-built edge rows (CPU only).

Each row is built on an exact grid (tests/edge_rows.py), so the result the
quantiser must give has a closed form in exact rational arithmetic:
  - at a tie (x - z)/s = k + 1/2 the code is the even neighbour;
  - one bf16 ulp off a tie the code is the nearest integer;
  - exact grids give the grid index, constant rows give scale 0 and code 0;
  - a span whose (max - min)/n underflows binary16 gets the scale 2^-24;
  - a scale that rounds below (max - min)/n clamps the top codes at n;
  - a zero extreme is +0, whichever zero the row holds (reading Q1 step 1);
and every dequantised value is within the error bound derived from the fp32
arithmetic (tests/edge_rows.dequant_bound).

Quantiser source: the per-token asymmetric min/max quantiser the DiffKV review
cites (KIVI), with the fp16 scale and zero and fp32 round-half-to-even of the
method's statement.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import edge_rows as E
from tests.oracle_helpers import f16


def _q(row_f32: np.ndarray, bits: int):
    st, q, s16, z16 = oracle.quant_row(E.bf16_bits_exact(row_f32), bits)
    assert st == oracle.OK
    return q, s16, z16


def _even_round(fr: Fraction) -> int:
    return round(fr)  # Python rounds a Fraction half to even


@pytest.mark.parametrize("bits,z,s", [(8, -1.0, 2.0 ** -5), (8, 0.0, 2.0 ** -9), (8, -3.0, 2.0 ** -4),
                                      (4, -0.5, 2.0 ** -3), (4, 0.125, 2.0 ** -6), (4, -96.0, 8.0),
                                      (2, 0.25, 2.0 ** -2), (2, -1.5, 1.0), (2, 0.0, 2.0 ** -12)])
def test_ties_round_to_even(bits, z, s):
    rng = np.random.default_rng(bits)
    row = E.tie_row(bits, z, s, rng)
    q, s16, z16 = _q(row, bits)
    assert f16([s16])[0] == np.float32(s) and f16([z16])[0] == np.float32(z)
    n = (1 << bits) - 1
    ties = 0
    for x, c in zip(row, q):
        t = (Fraction(float(x)) - Fraction(z)) / Fraction(s)
        assert c == min(max(_even_round(t), 0), n), (x, c, t)
        ties += t.denominator == 2
    assert ties > 100  # nearly every element sits on a tie


@pytest.mark.parametrize("bits,z,s", [(8, -1.0, 2.0 ** -5), (4, -0.5, 2.0 ** -3), (2, 0.25, 2.0 ** -2)])
def test_one_ulp_off_a_tie_rounds_to_nearest(bits, z, s):
    rng = np.random.default_rng(10 + bits)
    row = E.near_row(bits, z, s, rng)
    q, s16, z16 = _q(row, bits)
    assert f16([s16])[0] == np.float32(s) and f16([z16])[0] == np.float32(z)
    for x, c in zip(row, q):
        t = (Fraction(float(x)) - Fraction(z)) / Fraction(s)
        assert c == min(max(_even_round(t), 0), (1 << bits) - 1)


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_exact_grid_codes(bits):
    z, s = {8: (-1.0, 2.0 ** -5), 4: (-0.5, 2.0 ** -3), 2: (4.0, 2.0)}[bits]
    row = E.grid_row(bits, z, s, np.random.default_rng(bits))
    q, s16, z16 = _q(row, bits)
    assert np.array_equal(q.astype(np.float64), (row.astype(np.float64) - z) / s)


def test_clamped_top_codes():
    """Span 356 * 2^-24: (max - min)/255 = 1.396 * 2^-24 rounds to the
    subnormal 2^-24, so values above 255.5 * 2^-24 clamp to code 255."""
    row = E.kinds(np.random.default_rng(0))["clamp"][0]
    q, s16, z16 = _q(row, 8)
    assert s16 == 0x0001 and z16 == 0x0000
    k = np.round(row.astype(np.float64) * 2.0 ** 24).astype(np.int64)
    assert np.array_equal(q, np.minimum(k, 255))
    assert (k > 255).any()
    # at 4 bits the scale is 24 * 2^-24 (356/15 = 23.7): no clamping
    q4, s4, _ = _q(row, 4)
    assert s4 == 24 and np.array_equal(q4, [_even_round(Fraction(int(x), 24)) for x in k])


def test_subnormal_minimum_zero_point():
    """A minimum of -(2^-20 + 2^-27): binary16 rounds it to -16 * 2^-24, so z
    is not the minimum, and the minimum's code is rint(-1/8) = 0."""
    row = E.kinds(np.random.default_rng(0))["subnormal_min"][0]
    q, s16, z16 = _q(row, 8)
    assert z16 == 0x8010  # -16 * 2^-24
    s = Fraction(int(s16), 1 << 24)
    z = Fraction(-16, 1 << 24)
    for x, c in zip(row, q):
        assert c == min(max(_even_round((Fraction(float(x)) - z) / s), 0), 255)


def test_constant_rows():
    for c in (0.0, -0.0, 1.5, -65280.0, 65280.0, 2.0 ** -20, -3.0):
        row = np.full(128, c, dtype=np.float32)
        for bits in (8, 4, 2):
            q, s16, z16 = _q(row, bits)
            assert s16 == 0 and not q.any()
            assert z16 == np.array([c + 0.0], dtype=np.float16).view(np.uint16)[0]  # -0 stored as +0


def test_underflowing_span_gets_smallest_scale():
    """Span 2^-19 (32 units of 2^-24).  At 8 bits 32/255 units rounds to 0
    and the scale is raised to 2^-24; at 4 and 2 bits the scale is 32/n units
    rounded to even, and the larger element's code is 32 / scale, clamped."""
    row = E.kinds(np.random.default_rng(0))["underflow"][0]
    for bits in (8, 4, 2):
        n = (1 << bits) - 1
        q, s16, z16 = _q(row, bits)
        want_s = max(_even_round(Fraction(32, n)), 1)
        assert s16 == want_s and f16([z16])[0] == np.float32(2.0 ** -12)
        assert sorted(set(q.tolist())) == [0, min(_even_round(Fraction(32, want_s)), n)]


@pytest.mark.parametrize("first", [-0.0, 0.0])
def test_signed_zero_extremes_are_plus_zero(first):
    """Reading Q1 step 1: IEEE min / max leave the sign of a zero result open,
    so a zero minimum or maximum is taken as +0 whichever zero comes first."""
    other = 0.0 if first == -0.0 else -0.0
    lo = np.full(128, 0.5, dtype=np.float32)
    lo[0], lo[1], lo[2] = first, other, 1.0            # minimum is a zero
    q, s16, z16 = _q(lo, 8)
    assert z16 == 0x0000 and s16 == np.array([np.float32(1.0) / np.float32(255)], np.float16).view(np.uint16)[0]
    hi = np.full(128, -0.75, dtype=np.float32)
    hi[0], hi[1], hi[2] = first, other, -2.0           # maximum is a zero
    q, s16, z16 = _q(hi, 4)
    assert z16 == 0xC000 and f16([s16])[0] == np.float32(np.float16(np.float32(2.0) / np.float32(15)))
    assert q[0] == q[1] == 15                          # both zeros at the top code
    zeros = np.full(128, 0.0, dtype=np.float32)
    zeros[::2] = first
    zeros[1::2] = other
    q, s16, z16 = _q(zeros, 2)
    assert z16 == 0x0000 and s16 == 0 and not q.any()


def test_every_edge_row_within_the_bound():
    """|x - (z + q s)| <= dequant_bound(s, b) at every width, for every edge
    row; the strict 0.5 s + 1e-6 of the method's statement fails only where
    the scale is a binary16 subnormal that rounded down (the clamped rows) or
    an element sits within 2^-15 of a tie."""
    strict_fail = 0
    for kind, row in E.all_rows(np.random.default_rng(3)):
        x = row.astype(np.float64)
        for bits in (8, 4, 2):
            q, s16, z16 = _q(row, bits)
            s, z = float(f16([s16])[0]), float(f16([z16])[0])
            err = np.abs(x - (z + q.astype(np.float64) * s))
            assert np.all(err <= E.dequant_bound(s, bits)), (kind, bits, float(err.max()), s)
            bad = err > 0.5 * s + 1e-6
            if bad.any():
                assert kind == "clamp" or s < 2.0 ** -14, (kind, bits)
                strict_fail += int(bad.sum())
    assert strict_fail > 0  # the clamp row does exceed the strict bound


def test_bound_is_tight_enough_to_catch_a_wrong_code():
    """A code one off anywhere breaks the bound (so the GPU tests' bound
    check does catch an off-by-one), for scales of every magnitude."""
    # (below about 2e-6 the absolute 1e-6 of the method's bound is wider than
    # a grid step; the exact-grid and tie pins cover those scales)
    for s in (2.0 ** -14, 2.0 ** -5, 1.0, 514.0):
        for bits in (8, 4, 2):
            assert E.dequant_bound(s, bits) < s  # one step of the grid is outside it
