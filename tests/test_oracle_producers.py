"""Pins of the oracle's fused producers (RMSNorm+AdaLN and SwiGLU).

* Dyadic rows where every operation of the RMSNorm + modulation is exact, so
  the result is known as an exact rational: this pins which table entry is
  the shift and which the scale, where eps enters, and the frame lookup.
* Row statistics against binary64 (relative error <= 1e-6, the stated
  tolerance for the fp32 statistics) and the all-ones closed form.
* Modulated and SwiGLU values against binary64 within one bf16 ulp.
* Composition: each producer's codes and scales equal the standalone quantize
  of its own bf16 output.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_adaln_exact_dyadic_rows(orc):
    cols = 64
    rng = np.random.default_rng(21)
    rows = []
    # row 0: 16 entries +-2, rest 0 -> sum of squares 64, mean 1, rstd 1 (eps 0)
    r0 = np.zeros(cols); r0[rng.choice(cols, 16, replace=False)] = rng.choice([-2.0, 2.0], 16)
    # row 1: 16 entries +-8 -> mean 16, rstd 1/4
    r1 = np.zeros(cols); r1[rng.choice(cols, 16, replace=False)] = rng.choice([-8.0, 8.0], 16)
    # row 2: all +-2 -> mean 4, rstd 1/2
    r2 = rng.choice([-2.0, 2.0], cols)
    x = np.stack([r0, r1, r2]).astype(np.float32)
    expect_rstd = [Fraction(1), Fraction(1, 4), Fraction(1, 2)]
    gamma = rng.choice([0.5, 0.75, 1.0, 1.5, 2.0], cols).astype(np.float32)
    table = np.zeros((3, 2, cols), np.float32)
    table[:, 0] = rng.choice([0.0, 0.125, -1.0, 0.5], (3, cols))   # shift
    table[:, 1] = rng.choice([-0.5, 0.0, 0.25, 1.0], (3, cols))    # scale
    frames = np.array([2, 0, 1])
    codes, sf, rstd, y = orc.adaln_rows(_bits(x), _bits(gamma), _bits(table), frames, 0.0, 1.0,
                                        want_y=True)
    for r in range(3):
        assert Fraction(float(rstd[r])) == expect_rstd[r]
        t = frames[r]
        for j in range(cols):
            want = (Fraction(float(x[r, j])) * expect_rstd[r] * Fraction(float(gamma[j]))
                    * (1 + Fraction(float(table[t, 1, j]))) + Fraction(float(table[t, 0, j])))
            assert Fraction(float(_f(y[r, j]))) == want, (r, j)


def test_adaln_eps_enters_the_mean(orc):
    cols = 64
    x = np.zeros((1, cols), np.float32)
    x[0, :12] = 2.0   # sum of squares 48, mean 0.75
    gamma = np.ones(cols, np.float32)
    table = np.zeros((1, 2, cols), np.float32)
    _, _, rstd, _ = orc.adaln_rows(_bits(x), _bits(gamma), _bits(table), [0], 0.25, None)
    assert rstd[0] == 1.0  # 1 / sqrt(0.75 + 0.25)


def test_adaln_rstd_of_ones(orc):
    x = np.ones((1, 256), np.float32)
    _, _, rstd, _ = orc.adaln_rows(_bits(x), _bits(np.ones(256)), _bits(np.zeros((1, 2, 256))),
                                   [0], 1e-6, None)
    want = np.float32(1) / np.sqrt(np.float32(1) + np.float32(1e-6))
    assert rstd[0] == want


@pytest.mark.parametrize("cols", [64, 256, 1088, 7168])
def test_adaln_rstd_against_binary64(orc, cols):
    rng = np.random.default_rng(cols)
    sigma = np.exp(rng.normal(0, 0.5, cols))
    x = (rng.standard_normal((40, cols)) * sigma).astype(np.float32)
    xb = _bits(x)
    _, _, rstd, _ = orc.adaln_rows(xb, _bits(np.ones(cols)), _bits(np.zeros((1, 2, cols))),
                                   np.zeros(40, np.int64), 1e-6, None)
    xf = _f(xb).astype(np.float64)
    exact = 1 / np.sqrt((xf * xf).sum(1) / cols + np.float64(np.float32(1e-6)))
    assert np.max(np.abs(rstd - exact) / exact) <= 1e-6


def test_adaln_values_against_binary64_and_composition(orc):
    rng = np.random.default_rng(31)
    n, cols, frames_n = 48, 256, 4
    x = _bits(rng.standard_normal((n, cols)))
    gamma = _bits(rng.normal(1, 0.1, cols))
    table = _bits(rng.normal(0, 0.2, (frames_n, 2, cols)))
    frames = np.arange(n) // 16 % frames_n
    _, _, rstd, y = orc.adaln_rows(x, gamma, table, frames, 1e-6, None, want_y=True)
    gsf = orc.global_scale(float(np.abs(_f(y)).max()))
    codes, sf, rstd2, y2 = orc.adaln_rows(x, gamma, table, frames, 1e-6, gsf, want_y=True)
    assert np.array_equal(y, y2) and np.array_equal(rstd, rstd2)
    xf, gf, tf = _f(x).astype(np.float64), _f(gamma).astype(np.float64), _f(table).astype(np.float64)
    exact = xf * rstd[:, None] * gf * (1 + tf[frames, 1]) + tf[frames, 0]
    yf = _f(y).astype(np.float64)
    ulp = np.spacing(np.abs(yf).astype(np.float32)).astype(np.float64) * 65536
    assert np.all(np.abs(yf - exact) <= ulp + 1e-30)
    qcodes, qsf = orc.quantize_rows(y, gsf)
    assert np.array_equal(codes, qcodes) and np.array_equal(sf, qsf)


def test_swiglu_composition_and_values(orc):
    rng = np.random.default_rng(41)
    n, cols = 32, 192
    g = _bits(rng.normal(0, 1.5, (n, cols)))
    u = _bits(rng.normal(0, 1.5, (n, cols)))
    _, _, y = orc.swiglu_rows(g, u, None, want_y=True)
    assert np.array_equal(_f(y), orc.swiglu_value(_f(g), _f(u)))
    gsf = orc.global_scale(float(np.abs(_f(y)).max()))
    codes, sf, _ = orc.swiglu_rows(g, u, gsf)
    qcodes, qsf = orc.quantize_rows(y, gsf)
    assert np.array_equal(codes, qcodes) and np.array_equal(sf, qsf)


def test_swiglu_gate_is_the_silu_argument(orc):
    # silu(gate) * up with gate = 0 is 0 whatever up is; up = 0 gives 0 whatever gate is
    g = np.zeros((1, 64), np.float32)
    u = np.full((1, 64), 5.0, np.float32)
    _, _, y = orc.swiglu_rows(_bits(g), _bits(u), None, want_y=True)
    assert (_f(y) == 0).all()
    _, _, y = orc.swiglu_rows(_bits(u), _bits(g), None, want_y=True)
    assert (_f(y) == 0).all()
    # large gate: silu(gate) = gate exactly in binary32
    _, _, y = orc.swiglu_rows(_bits(np.full((1, 64), 40.0)), _bits(np.full((1, 64), 0.5)), None,
                              want_y=True)
    assert (_f(y) == 20.0).all()


def test_threads_give_identical_output(orc):
    rng = np.random.default_rng(51)
    x = _bits(rng.standard_normal((37, 128)))
    a = orc.quantize_rows(x, 2.0, threads=1)
    b = orc.quantize_rows(x, 2.0, threads=4)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))
