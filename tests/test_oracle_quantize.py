"""Pins of the oracle's NVFP4 block quantize, scale layout and dequantize.

What pins them (none of it is the oracle checking itself):
* hand-worked blocks derived from the definitions (tests/golden/hand_block.txt,
  tests/golden/scale_cases.txt);
* hand-derived offsets of the 128x4 layout (tests/golden/swizzle_cases.txt),
  plus the layout being a bijection with zeroed padding rows;
* brute force: every code is the nearest of all 16 E2M1 codes to y * inv, and
  every scale the nearest of all 127 E4M3 values to gsf * amax / 6 (exact
  rationals);
* the error invariant |y - dequant| <= half a grid step x block scale;
* dequantize against the closed form E2M1(c) * E4M3(sf) / gsf computed in
  binary64 (one correctly rounded binary32 result).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import golden_lines


def _hand_block():
    d = {}
    for line in golden_lines("hand_block.txt"):
        key, *vals = line.split()
        d[key] = vals
    return d


def test_hand_worked_block(orc):
    d = _hand_block()
    y = np.array([float(v) for v in d["y"]], np.float32)
    sf, packed = orc.quantize_block(y, float(d["gsf"][0]))
    assert sf == int(d["sf"][0], 16)
    assert packed.tolist() == [int(b, 16) for b in d["codes"]]
    deq = orc.dequantize_rows(np.concatenate([packed, np.zeros(24, np.uint8)]).reshape(1, 32),
                              np.array([[sf, 0, 0, 0]], np.uint8), float(d["gsf"][0]))
    # a 64-wide row: the hand block, then three zero blocks; values and signs of zero
    want = np.array([float(v) for v in d["dequant"]], np.float32)
    assert np.array_equal(deq[0, :16], want)
    assert np.array_equal(np.signbit(deq[0, :16]), np.signbit(want))


@pytest.mark.parametrize("line", list(golden_lines("scale_cases.txt")))
def test_scale_cases(orc, line):
    name, gsf, amax, sf_hex, code_hex, deq = line.split()
    y = np.zeros(16, np.float32)
    y[0] = np.float32(amax)
    sf, packed = orc.quantize_block(y, float(gsf))
    assert sf == int(sf_hex, 16), name
    assert packed[0] & 0xF == int(code_hex, 16), name
    assert all(p == 0 for p in packed[1:]) and packed[0] >> 4 == 0, name
    deqv = orc.dequantize_rows(np.concatenate([packed, np.zeros(24, np.uint8)]).reshape(1, 32),
                               np.array([[sf, 0, 0, 0]], np.uint8), float(gsf))
    assert deqv[0, 0] == np.float32(deq), name


def test_outlier_block_with_tensor_amax_scale(orc):
    gsf = orc.global_scale(1000.0)
    assert gsf == np.float32(2688.0) / np.float32(1000.0)
    rng = np.random.default_rng(3)
    y = (rng.standard_normal(16) * 2).astype(np.float32)
    y[7] = 1000.0
    sf, packed = orc.quantize_block(y, gsf)
    assert sf == 0x7E
    codes = [(b >> (4 * h)) & 0xF for b in packed for h in (0, 1)]
    assert codes[7] == 7
    assert all(c & 7 == 0 for i, c in enumerate(codes) if i != 7)


def test_swizzle_hand_offsets(orc):
    for line in golden_lines("swizzle_cases.txt"):
        r, g, cols, off = line.split()
        want = sum(int(np.prod([int(f) for f in term.split("*")])) for term in off.split("+"))
        assert orc.scale_offset(int(r), int(g), int(cols)) == want, line


@pytest.mark.parametrize("rows,cols", [(1, 64), (127, 64), (128, 128), (129, 192), (300, 448), (64, 256)])
def test_swizzle_bijection_and_padding(orc, rows, cols):
    groups = cols // 16
    pad = orc.padded_rows(rows)
    assert pad % 128 == 0 and pad >= rows and pad - rows < 128
    offs = orc.scale_offsets(np.arange(pad), cols).ravel()
    assert np.array_equal(np.sort(offs), np.arange(pad * groups))
    rng = np.random.default_rng(rows * 1000 + cols)
    sf = rng.integers(1, 0x7F, (rows, groups), dtype=np.uint8)
    out = orc.swizzle_scales(sf, rows, cols)
    real = orc.scale_offsets(np.arange(rows), cols)
    assert np.array_equal(out[real], sf)
    pad_offs = orc.scale_offsets(np.arange(rows, pad), cols).ravel()
    assert (out[pad_offs] == 0).all()


def _e4m3_exact(code):
    e, m = (code >> 3) & 15, code & 7
    if e == 0:
        return Fraction(m, 512)
    return (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


E4M3_VALUES = [_e4m3_exact(c) for c in range(0x7F)]
E2M1_MAG = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]


def _random_blocks(n, seed):
    rng = np.random.default_rng(seed)
    kinds = rng.integers(0, 4, n)
    scale = np.exp(rng.uniform(-12, 6, n))[:, None]
    y = rng.standard_normal((n, 16)) * scale
    y[kinds == 1] = rng.standard_t(3, (int((kinds == 1).sum()), 16)) * scale[kinds == 1]
    y[kinds == 2, 0] *= 50  # one outlier
    y = torch.from_numpy(y.astype(np.float32)).bfloat16().float().numpy()
    gsf = np.exp(rng.uniform(-3, 6, n)).astype(np.float32)
    return y, gsf


def test_brute_force_nearest_scale_and_codes(orc):
    y, gsf = _random_blocks(400, 7)
    for i in range(len(y)):
        g = float(gsf[i])
        sf, packed = orc.quantize_block(y[i], g)
        amax = np.float32(np.abs(y[i]).max())
        s = np.float32(np.float32(g) * np.float32(amax / np.float32(6)))
        target = Fraction(float(s))
        if s >= 448:
            assert sf == 0x7E
        else:
            dists = [abs(v - target) for v in E4M3_VALUES]
            best = min(dists)
            cands = [c for c, dd in enumerate(dists) if dd == best]
            assert sf == (cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0])
        dec = np.float32(np.float32(orc.e4m3_value(sf)) / np.float32(g))
        inv = np.float32(np.float32(1) / dec) if dec != 0 else np.float32(0)
        for j in range(16):
            q = Fraction(float(np.float32(y[i, j] * inv)))
            code = (packed[j // 2] >> (4 * (j % 2))) & 0xF
            mag = code & 7
            if abs(q) >= 6:
                assert mag == 7
            else:
                dists = [abs(abs(q) - v) for v in E2M1_MAG]
                best = min(dists)
                cands = [c for c, dd in enumerate(dists) if dd == best]
                assert mag == (cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0])
            assert (code >> 3) == int(np.signbit(np.float32(y[i, j] * inv)))


def _half_step(a):
    # half the distance between neighbouring E2M1 magnitudes around a (the wider
    # step where a is within a hair of a step boundary)
    return np.where(a < 2 * (1 - 2**-20), 0.25, np.where(a < 4 * (1 - 2**-20), 0.5, 1.0))


def test_dequant_error_invariant(orc):
    y, gsf = _random_blocks(3000, 9)
    for i in range(len(y)):
        g = float(gsf[i])
        row = np.zeros((1, 64), np.float32)
        row[0, :16] = y[i]
        codes, sf = orc.quantize_rows(orc.bf16_bits(row), g)
        deq = orc.dequantize_rows(codes, sf, g)[0, :16].astype(np.float64)
        code = sf[0, 0]
        if not (0x08 <= code < 0x7E):
            continue  # subnormal or saturated scale: relative rounding of the scale is coarser
        dec = orc.e4m3_value(code) / g
        a = np.abs(y[i].astype(np.float64)) / dec
        bound = _half_step(a) * dec * (1 + 2**-20) + 8 * dec * 2**-22
        assert np.all(np.abs(y[i] - deq) <= bound), i


def test_dequant_closed_form(orc):
    rng = np.random.default_rng(4)
    rows, cols = 5, 128
    codes = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    sf = rng.integers(0, 0x7F, (rows, cols // 16), dtype=np.uint8)
    for g in (1.0, 2.688, 1e-3, 37.5):
        got = orc.dequantize_rows(codes, sf, g)
        grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
        nib = np.stack([codes & 0xF, codes >> 4], -1).reshape(rows, cols)
        val = grid[nib & 7] * np.where(nib & 8, -1.0, 1.0)
        sfv = np.array([float(_e4m3_exact(int(c))) for c in sf.ravel()]).reshape(sf.shape)
        want = (val * np.repeat(sfv, 16, axis=1) / np.float64(np.float32(g))).astype(np.float32)
        assert np.array_equal(got, want)
        assert np.array_equal(np.signbit(got), np.signbit(want))


def test_quantize_rows_matches_blocks(orc):
    rng = np.random.default_rng(12)
    x = torch.from_numpy(rng.standard_normal((3, 192)).astype(np.float32)).bfloat16()
    bits = x.view(torch.int16).numpy().view(np.uint16)
    codes, sf = orc.quantize_rows(bits, 3.0)
    xf = x.float().numpy()
    for r in range(3):
        for b in range(12):
            s, p = orc.quantize_block(xf[r, 16 * b:16 * b + 16], 3.0)
            assert sf[r, b] == s and np.array_equal(codes[r, 8 * b:8 * b + 8], p)
