"""The oracle's residual fold + RMSNorm + AdaLN against what fixes it
independently: the fold in numpy binary32 arithmetic with torch's bf16 rounding,
exact hand values, the fp32-row rstd equal to the bf16-row rstd wherever the
values are bf16, the whole norm part equal to the bf16 AdaLN oracle when the
folded residual holds bf16 values, and rstd within 1e-6 of binary64."""
import numpy as np
import pytest
import torch

import oracle


def _bf16(values) -> np.ndarray:
    """float values -> bf16 bit patterns (torch's round to nearest even)."""
    return torch.as_tensor(np.asarray(values, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(bits) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def _inputs(n, cols, frames, seed):
    rng = np.random.default_rng(seed)
    h = (rng.standard_normal((n, cols)) * 2).astype(np.float32)
    o = _bf16(rng.standard_normal((n, cols)))
    bias = _bf16(rng.standard_normal(cols) * 0.1)
    gate = _bf16(rng.standard_normal((frames, cols)) * 0.5)
    gamma = _bf16(1 + rng.standard_normal(cols) * 0.1)
    table = _bf16(rng.standard_normal((frames, 2, cols)) * 0.3)
    fr = rng.integers(0, frames, n)
    return h, o, bias, gate, gamma, table, fr


@pytest.mark.parametrize("with_bias", [True, False])
def test_fold_matches_numpy_binary32(with_bias):
    h, o, bias, gate, gamma, table, fr = _inputs(40, 320, 3, 1)
    h_out, _, _, _, _ = oracle.residual_adaln_rows(h, o, bias if with_bias else None, gate, gamma,
                                                   table, fr, 1e-6, None)
    ov = _val(o)
    u = _val(_bf16(ov + _val(bias)[None, :])) if with_bias else ov  # fl(o + b) in binary32, then bf16
    t = (u * _val(gate)[fr]).astype(np.float32)
    want = (h + t).astype(np.float32)
    assert np.array_equal(h_out.view(np.uint32), want.view(np.uint32))


def test_fold_hand_values():
    cols = 64
    h = np.full((1, cols), 1.5, np.float32)
    o = _bf16(np.full((1, cols), 2.0))
    bias = _bf16(np.full(cols, 0.25))
    gate = _bf16(np.full((1, cols), 0.5))
    gamma, table = _bf16(np.ones(cols)), _bf16(np.zeros((1, 2, cols)))
    h_out, *_ = oracle.residual_adaln_rows(h, o, bias, gate, gamma, table, [0], 1e-6, None)
    assert (h_out == np.float32(2.625)).all()  # 1.5 + bf16(2.25) * 0.5
    # o + bias is rounded to bf16 before the gate: 1 + 3 * 2^-9 -> 1 + 2^-7
    o1 = _bf16(np.ones((1, cols)))
    b1 = _bf16(np.full(cols, 3 * 2.0 ** -9))
    g1 = _bf16(np.ones((1, cols)))
    h0 = np.zeros((1, cols), np.float32)
    h_out, *_ = oracle.residual_adaln_rows(h0, o1, b1, g1, gamma, table, [0], 1e-6, None)
    assert (h_out == np.float32(1 + 2.0 ** -7)).all()


@pytest.mark.parametrize("cols", [64, 256, 1088, 7168])
def test_fp32_rstd_equals_bf16_rstd_on_bf16_rows(cols):
    rng = np.random.default_rng(cols)
    bits = _bf16(rng.standard_normal(cols) * rng.uniform(0.1, 10))
    assert oracle.row_rstd_f32(_val(bits), 1e-6) == oracle.adaln_rows(
        bits[None, :], _bf16(np.ones(cols)), _bf16(np.zeros((1, 2, cols))), [0], 1e-6, None)[2][0]


def test_norm_part_equals_the_bf16_adaln_oracle_when_the_residual_is_bf16():
    """o = 0 and no bias: the fold leaves h unchanged, and h holds bf16 values, so
    rstd, y, codes and scales equal the bf16 AdaLN oracle's on those values."""
    n, cols, frames = 20, 1024, 2
    _, _, _, gate, gamma, table, fr = _inputs(n, cols, frames, 3)
    x = _bf16(np.random.default_rng(4).standard_normal((n, cols)) * 1.7)
    h = _val(x)
    o = np.zeros((n, cols), np.uint16)
    _, _, _, y_ref = oracle.adaln_rows(x, gamma, table, fr, 1e-6, None, want_y=True)
    gsf = oracle.global_scale(float(np.abs(_val(y_ref)).max()))
    h_out, co, so, ro, y = oracle.residual_adaln_rows(h, o, None, gate, gamma, table, fr, 1e-6, gsf,
                                                      want_y=True)
    c2, s2, r2, y2 = oracle.adaln_rows(x, gamma, table, fr, 1e-6, gsf, want_y=True)
    assert np.array_equal(h_out, h)
    assert np.array_equal(ro.view(np.uint32), r2.view(np.uint32))
    assert np.array_equal(y, y2) and np.array_equal(co, c2) and np.array_equal(so, s2)


def test_rstd_within_1e6_of_binary64():
    h, o, bias, gate, gamma, table, fr = _inputs(64, 2048, 2, 5)
    h_out, _, _, rstd, _ = oracle.residual_adaln_rows(h, o, bias, gate, gamma, table, fr, 1e-6, None)
    hd = h_out.astype(np.float64)
    exact = 1 / np.sqrt((hd * hd).mean(1) + np.float64(np.float32(1e-6)))
    assert (np.abs(rstd - exact) / exact).max() <= 1e-6
