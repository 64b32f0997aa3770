"""The oracle's block-scaled NVFP4 GEMM and its SwiGLU + NVFP4 epilogue, against
what fixes them independently:

- hand-worked dot products (tests/golden/gemm_cases.txt), one of them a sum
  that only an exact accumulation rounded once gives;
- the exact rational sum of the dequantized products (each element's value
  from the oracle's dequantize with gsf = 1, itself pinned to the closed forms)
  rounded to binary32 by a rounding written here, over random codes and every
  scale code;
- invariants: the GEMM of (B, A) is the transpose; doubling every scale of A
  doubles acc exactly;
- the epilogue with alpha = 1 on bf16-valued accumulators equals the SwiGLU
  producer's oracle on the value and gate columns; alpha and its bf16 rounding
  checked through a saturated gate (sigma = 1), with numpy binary32 products and
  torch's bf16 rounding.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_lines


def _u32(x) -> np.ndarray:
    return np.asarray(x, np.float32).view(np.uint32)


def _round_f32(q: Fraction) -> np.float32:
    """An exact rational rounded to binary32 (normal range), nearest, ties to even."""
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    scaled = a / Fraction(2) ** (e - 23)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return np.float32(sign * float(Fraction(m) * Fraction(2) ** (e - 23)))


def _cases():
    cases, cur = [], None
    for line in golden_lines("gemm_cases.txt"):
        tok = line.split()
        if tok[0] == "case":
            cur = {"name": tok[1], "k": int(tok[3])}
            cases.append(cur)
        elif tok[0] in ("a", "b", "sfa", "sfb"):
            cur[tok[0]] = np.array([int(t, 16) for t in tok[1:]], np.uint8)[None, :]
        elif tok[0] == "acc":
            cur["acc"] = int(tok[1], 16)
    return cases


CASES = _cases()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_worked_dot_products(case):
    acc = oracle.nvfp4_gemm(case["a"], case["sfa"], case["b"], case["sfb"])
    assert acc.shape == (1, 1)
    assert int(_u32(acc)[0, 0]) == case["acc"], f"{case['name']}: {acc[0, 0]!r}"


def test_rounded_once_not_accumulated_in_binary32():
    """G2's products summed one at a time in binary32 give another result."""
    case = next(c for c in CASES if c["name"] == "G2")
    p = np.float32(2688.0) * np.float32(2688.0)
    for _ in range(3):
        p = np.float32(p + np.float32(0.25))
    assert int(_u32(p)) != case["acc"]


def _random_operands(rng, rows, k, scales=None):
    codes = rng.integers(0, 256, (rows, k // 2), dtype=np.uint8)
    if scales is None:
        sf = rng.integers(0, 0x7F, (rows, k // 16), dtype=np.uint8)
    else:
        sf = rng.choice(np.asarray(scales, np.uint8), (rows, k // 16))
    return codes, sf


def _exact_acc(a_codes, a_sf, b_codes, b_sf):
    """fl(exact sum) from the dequantized element values (exact in binary32 at gsf = 1)."""
    av = oracle.dequantize_rows(a_codes, a_sf, 1.0).astype(np.float64)
    bv = oracle.dequantize_rows(b_codes, b_sf, 1.0).astype(np.float64)
    out = np.empty((av.shape[0], bv.shape[0]), np.float32)
    for i in range(av.shape[0]):
        fa = [Fraction(float(x)) for x in av[i]]
        for j in range(bv.shape[0]):
            s = sum((x * Fraction(float(y)) for x, y in zip(fa, bv[j]) if y != 0.0), Fraction(0))
            out[i, j] = _round_f32(s)
    return out


@pytest.mark.parametrize("k,scales", [(64, None), (128, None), (64, [0x00, 0x01, 0x07, 0x08, 0x7E]),
                                      (192, [0x30, 0x38, 0x40, 0x7E])])
def test_exact_sum_rounded_once(k, scales):
    rng = np.random.default_rng(k + (len(scales) if scales else 0))
    a_codes, a_sf = _random_operands(rng, 5, k, scales)
    b_codes, b_sf = _random_operands(rng, 6, k, scales)
    got = oracle.nvfp4_gemm(a_codes, a_sf, b_codes, b_sf)
    want = _exact_acc(a_codes, a_sf, b_codes, b_sf)
    assert np.array_equal(_u32(got), _u32(want))


def test_transpose_symmetry_and_scale_doubling():
    rng = np.random.default_rng(7)
    k = 256
    a_codes, a_sf = _random_operands(rng, 9, k, list(range(0x08, 0x70)))
    b_codes, b_sf = _random_operands(rng, 11, k, list(range(0x00, 0x7F)))
    ab = oracle.nvfp4_gemm(a_codes, a_sf, b_codes, b_sf)
    ba = oracle.nvfp4_gemm(b_codes, b_sf, a_codes, a_sf)
    assert np.array_equal(_u32(ab), _u32(ba.T))
    # exponent field + 1 doubles every scale of A (all normal, none reaches 0x78)
    doubled = oracle.nvfp4_gemm(a_codes, a_sf + 8, b_codes, b_sf)
    assert np.array_equal(_u32(doubled), _u32(ab * np.float32(2)))


def test_multi_threaded_rows_are_the_single_threaded_ones():
    rng = np.random.default_rng(8)
    a_codes, a_sf = _random_operands(rng, 13, 512)
    b_codes, b_sf = _random_operands(rng, 7, 512)
    one = oracle.nvfp4_gemm(a_codes, a_sf, b_codes, b_sf)
    many = oracle.nvfp4_gemm(a_codes, a_sf, b_codes, b_sf, threads=4)
    assert np.array_equal(_u32(one), _u32(many))


def _bf16(values) -> np.ndarray:
    return torch.as_tensor(np.asarray(values, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def test_epilogue_with_unit_alpha_is_the_swiglu_producer():
    """alpha = 1 and bf16-valued accumulators: u and g are the accumulators
    themselves, so the epilogue is the SwiGLU producer's spec on (gate, up)."""
    rng = np.random.default_rng(9)
    m, f = 6, 256
    up = _bf16(rng.standard_normal((m, f)) * 2)
    gate = _bf16(rng.standard_normal((m, f)) * 4)
    acc = np.empty((m, 2 * f), np.float32)
    acc[:, 0::2] = _val(up)
    acc[:, 1::2] = _val(gate)
    gsf = 0.37
    codes, sf, y = oracle.swiglu_epilogue_rows(acc, 1.0, gsf, want_y=True)
    c2, s2, y2 = oracle.swiglu_rows(gate, up, gsf, want_y=True)
    assert np.array_equal(codes, c2) and np.array_equal(sf, s2) and np.array_equal(y, y2)


def test_epilogue_alpha_and_its_roundings():
    """A gate of 20 has sigma(20) = fl(1 / (1 + e^-20)) = 1 exactly, so y = bf16(fl(20 *
    u)) with u = bf16(fl(alpha * acc_value)); and with u = 1 the gate side is
    g = bf16(fl(alpha * acc_gate)) into the SwiGLU value."""
    rng = np.random.default_rng(10)
    m, f = 4, 128
    alpha = np.float32(0.0123)
    acc_v = (rng.standard_normal((m, f)) * 300).astype(np.float32)
    acc = np.empty((m, 2 * f), np.float32)
    acc[:, 0::2] = acc_v
    acc[:, 1::2] = np.float32(20.0) / alpha          # alpha * that rounds to ~20
    g = _val(_bf16(np.float32(alpha) * acc[:, 1::2]))
    assert (g == np.float32(20.0)).all()
    _, _, y = oracle.swiglu_epilogue_rows(acc, float(alpha), None, want_y=True)
    u = _val(_bf16(alpha * acc_v))
    assert np.array_equal(y, _bf16(np.float32(20.0) * u))

    acc_g = (rng.standard_normal((m, f)) * 500).astype(np.float32)
    acc[:, 0::2] = np.float32(1.0) / alpha
    acc[:, 1::2] = acc_g
    assert (_val(_bf16(alpha * acc[:, 0::2])) == np.float32(1.0)).all()
    _, _, y = oracle.swiglu_epilogue_rows(acc, float(alpha), None, want_y=True)
    gv = _val(_bf16(alpha * acc_g))
    want = _bf16(oracle.swiglu_value(gv, np.ones_like(gv)))
    assert np.array_equal(y, want)


def test_pairs_are_value_then_gate():
    """Column 2j is the value and 2j+1 the gate: swapping them changes y."""
    acc = np.zeros((1, 128), np.float32)
    acc[0, 0::2] = 3.0
    acc[0, 1::2] = -1.0
    _, _, y = oracle.swiglu_epilogue_rows(acc, 1.0, None, want_y=True)
    want = _bf16(oracle.swiglu_value(np.full(64, -1.0, np.float32), np.full(64, 3.0, np.float32)))
    assert np.array_equal(y[0], want)
    assert not np.array_equal(y[0], _bf16(oracle.swiglu_value(np.full(64, 3.0, np.float32),
                                                              np.full(64, -1.0, np.float32))))
