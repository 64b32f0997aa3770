"""Pins of the oracle's number conversions against sources other than itself.

* bf16 rounding: torch's CPU cast on every upper half with every deciding low
  half, and on every low half under a spread of upper halves.
* E4M3 decode: all 127 finite non-negative codes against exact rational
  values of the format's definition and against torch.float8_e4m3fn.
* E4M3 encode: round trip of every code, torch's float8_e4m3fn cast on dense
  samples and on every value near each rounding midpoint, and saturation.
* E2M1 encode: an independent threshold-count formulation of round-to-nearest-
  even on the grid {0, .5, 1, 1.5, 2, 3, 4, 6}, on every bf16 value and dense
  binary32 samples; decode against the grid.
* exp_c: its constants re-derived from the real numbers they name, and its
  error against binary64 exp at most 2 ulp over its whole domain (every bf16
  input, a dense binary32 sample), plus its special cases.
"""
from decimal import Decimal, getcontext
from fractions import Fraction
import math

import numpy as np
import pytest
import torch


# --------------------------------------------------------------------------- #
# bf16                                                                          #
# --------------------------------------------------------------------------- #

def _check_bf16(orc, bits):
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    ours = orc.bf16_bits(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"bf16 mismatch at {vals[bad[:5]]}: {ours[bad[:5]]} vs {ref[bad[:5]]}"


def test_bf16_rounding_every_upper_half(orc):
    """Every one of the 65536 upper halves with every low half that decides a
    rounding (0, 1, just below/at/above the midpoint, all ones) plus 58 random."""
    rng = np.random.default_rng(5)
    lows = np.unique(np.concatenate([
        np.array([0, 1, 0x7FFE, 0x7FFF, 0x8000, 0x8001, 0xFFFE, 0xFFFF], np.uint32),
        rng.integers(0, 1 << 16, 58, dtype=np.uint32)]))
    uppers = np.arange(1 << 16, dtype=np.uint32) << 16
    _check_bf16(orc, (uppers[:, None] | lows[None, :]).ravel())


def test_bf16_rounding_every_low_half(orc):
    """All 65536 low halves under 512 upper halves (every sign/exponent edge and a
    random spread)."""
    rng = np.random.default_rng(6)
    uppers = np.unique(np.concatenate([
        np.array([0x0000, 0x0001, 0x007F, 0x0080, 0x3F80, 0x3F81, 0x7F7F, 0x7F7E,
                  0x8000, 0x8001, 0xBF80, 0xFF7F], np.uint32),
        rng.integers(0, 1 << 16, 500, dtype=np.uint32)])) << 16
    lows = np.arange(1 << 16, dtype=np.uint32)
    _check_bf16(orc, (uppers[:, None] | lows[None, :]).ravel())


def test_bf16_round_half_even_cases(orc):
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1); 1 + 3*2^-8 -> 1 + 2^-6.
    vals = np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 3.0e38 * 1.134], np.float32)
    got = orc.bf16_value(orc.bf16_bits(vals))
    assert got[0] == 1.0 and got[1] == 1 + 2**-6 and got[2] == -1.0
    assert np.isinf(got[3])  # beyond bf16's largest finite value plus half an ulp


# --------------------------------------------------------------------------- #
# E4M3                                                                          #
# --------------------------------------------------------------------------- #

def _e4m3_exact(code):
    e, m = (code >> 3) & 15, code & 7
    if e == 0:
        return Fraction(m, 512)
    return (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def test_e4m3_decode_all_codes(orc):
    torch_vals = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for code in range(0x7F):
        v = orc.e4m3_value(code)
        assert Fraction(v) == _e4m3_exact(code), hex(code)
        assert v == torch_vals[code], hex(code)
    assert orc.e4m3_value(0x7E) == 448.0 and orc.e4m3_value(0x01) == 2.0**-9
    assert orc.e4m3_value(0x08) == 2.0**-6


def test_e4m3_round_trip(orc):
    vals = np.array([orc.e4m3_value(c) for c in range(0x7F)], np.float32)
    assert np.array_equal(orc.e4m3_encode(vals), np.arange(0x7F, dtype=np.uint8))


def _torch_e4m3(vals):
    return torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_near_every_midpoint(orc):
    pts = []
    for c in range(0x7E):
        mid = (float(_e4m3_exact(c)) + float(_e4m3_exact(c + 1))) / 2
        centre = np.float32(mid).view(np.uint32).astype(np.int64)
        pts.append(np.arange(centre - 300, centre + 301))
        v = np.float32(float(_e4m3_exact(c))).view(np.uint32).astype(np.int64)
        pts.append(np.arange(max(v - 50, 0), v + 51))
    bits = np.unique(np.concatenate(pts)).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[(vals >= 0) & (vals < 464.0)]
    assert np.array_equal(orc.e4m3_encode(vals), _torch_e4m3(vals))


def test_e4m3_encode_matches_torch_dense_sample(orc):
    top = np.float32(464.0).view(np.uint32)
    bits = np.arange(0, int(top), 1009, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    assert np.array_equal(orc.e4m3_encode(vals), _torch_e4m3(vals))


def test_e4m3_encode_ties_and_saturation(orc):
    # halfway between consecutive codes goes to the even code
    ties = np.array([1.0625, 1.1875, 2.0**-10, 3 * 2.0**-10, 7.5 * 2.0**-9, 432.0], np.float32)
    assert orc.e4m3_encode(ties).tolist() == [0x38, 0x3A, 0x00, 0x02, 0x08, 0x7E]
    big = np.array([448.0, 463.99, 464.0, 479.0, 480.0, 1e6, 3.4e38, np.inf], np.float32)
    assert (orc.e4m3_encode(big) == 0x7E).all()
    assert orc.e4m3_encode(np.array([0.0, 1e-30, 2.0**-11], np.float32)).tolist() == [0, 0, 0]


# --------------------------------------------------------------------------- #
# E2M1                                                                          #
# --------------------------------------------------------------------------- #

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_by_thresholds(v):
    """RNE on the E2M1 grid as a count of crossed midpoints: a tie goes to the
    even index, so midpoints before an odd index need '>' and before an even
    index need '>='."""
    a = np.abs(v)
    idx = ((a > 0.25).astype(np.uint8) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
           + (a > 2.5) + (a >= 3.5) + (a > 5.0))
    return (idx | (np.signbit(v).astype(np.uint8) << 3)).astype(np.uint8)


def test_e2m1_decode_grid(orc):
    for c in range(16):
        expect = GRID[c & 7] * (-1 if c & 8 else 1)
        assert orc.e2m1_value(c) == expect
    assert math.copysign(1, orc.e2m1_value(8)) == -1


def test_e2m1_encode_every_bf16(orc):
    vals = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    vals = vals[np.isfinite(vals)]
    assert np.array_equal(orc.e2m1_encode(vals), _e2m1_by_thresholds(vals))


def test_e2m1_encode_near_thresholds_and_dense(orc):
    pts = []
    for t in [0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0]:
        c = np.float32(t).view(np.uint32).astype(np.int64)
        pts.append(np.arange(c - 4096, c + 4097))
    pts.append(np.arange(0, 0x41800000, 997))  # every 997th pattern of [0, 16)
    bits = np.unique(np.concatenate(pts)).astype(np.uint32)
    vals = np.concatenate([bits.view(np.float32), -bits.view(np.float32)])
    assert np.array_equal(orc.e2m1_encode(vals), _e2m1_by_thresholds(vals))


def test_e2m1_special_values(orc):
    v = np.array([0.0, -0.0, -0.1, 0.25, -0.25, 6.0, 7.0, 1e30, np.inf, -np.inf], np.float32)
    assert orc.e2m1_encode(v).tolist() == [0, 8, 8, 0, 8, 7, 7, 7, 7, 15]


# --------------------------------------------------------------------------- #
# exp_c                                                                         #
# --------------------------------------------------------------------------- #

def _f32_of(x: Fraction) -> float:
    """Correctly rounded binary32 of an exact rational (independent of numpy)."""
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    q = x / Fraction(2) ** (e - 23)
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2):
        n += 1
    return sign * float(Fraction(n) * Fraction(2) ** (e - 23))


def test_exp_constants_are_the_named_reals(orc):
    getcontext().prec = 60
    ln2 = Fraction(Decimal(2).ln())
    k = orc.exp_constants()
    assert k["L2E"] == _f32_of(1 / ln2)
    assert k["C1"] == _f32_of(ln2)
    assert k["C2"] == _f32_of(ln2 - Fraction(k["C1"]))
    for n in range(1, 8):
        assert k[f"P{n}"] == _f32_of(Fraction(1, math.factorial(n))), n


def _ulp_error(got, z):
    exact = np.exp(z.astype(np.float64))
    ref32 = exact.astype(np.float32)
    ulp = np.spacing(np.abs(ref32)).astype(np.float64)
    ulp = np.maximum(ulp, 2.0**-149)
    return np.abs(got.astype(np.float64) - exact) / ulp


def test_exp_c_accuracy_every_bf16_input(orc):
    z = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    z = z[np.isfinite(z) & (z >= -104) & (z <= 88.5)]
    assert np.max(_ulp_error(orc.exp_c(z), z)) <= 2.0


def test_exp_c_accuracy_dense_binary32(orc):
    lo = np.float32(-104.0).view(np.uint32)
    hi = np.float32(88.5).view(np.uint32)
    neg = np.arange(0x80000000, int(lo) + 1, 101, dtype=np.uint64).astype(np.uint32)
    pos = np.arange(0, int(hi) + 1, 101, dtype=np.uint64).astype(np.uint32)
    z = np.concatenate([neg, pos]).view(np.float32)
    assert np.max(_ulp_error(orc.exp_c(z), z)) <= 2.0


def test_exp_c_special_cases(orc):
    z = np.array([0.0, -0.0, 89.0, 88.8, 1e30, -104.5, -1e30, -104.0, -103.9], np.float32)
    got = orc.exp_c(z)
    assert got[0] == 1.0 and got[1] == 1.0
    assert np.isinf(got[2]) and np.isinf(got[3]) and np.isinf(got[4])
    assert got[5] == 0.0 and got[6] == 0.0
    assert got[7] == 0.0            # exp(-104) < 2^-150: rounds to zero
    assert got[8] == 2.0**-149      # exp(-103.9) rounds to the smallest subnormal
    # monotone over a dense sweep of its domain
    sweep = np.linspace(-104, 88.7, 200001, dtype=np.float32)
    assert np.all(np.diff(orc.exp_c(sweep)) >= 0)


def test_swiglu_value_against_binary64(orc):
    rng = np.random.default_rng(11)
    g = (rng.standard_normal(200000) * 3).astype(np.float32)
    u = (rng.standard_normal(200000) * 3).astype(np.float32)
    g = torch.from_numpy(g).bfloat16().float().numpy()
    u = torch.from_numpy(u).bfloat16().float().numpy()
    got = orc.swiglu_value(g, u)
    g64, u64 = g.astype(np.float64), u.astype(np.float64)
    exact = g64 / (1 + np.exp(-g64)) * u64
    # one bf16 rounding of a value within a few binary32 ulps of exact:
    # at most one bf16 ulp away
    ref = torch.from_numpy(exact.astype(np.float32)).bfloat16().float().numpy().astype(np.float64)
    bf16_ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) * 65536
    assert np.all(np.abs(got - ref) <= bf16_ulp + 1e-45)
    # special cases: silu(0) = 0, large gates
    s = orc.swiglu_value(np.array([0.0, 40.0, -200.0], np.float32), np.array([5.0, 2.0, 3.0], np.float32))
    assert s[0] == 0.0 and s[1] == 80.0 and s[2] == 0.0
