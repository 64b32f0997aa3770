"""The oracle's SwiGLU of a value-first packed projection with bias
against what fixes it independently: without a bias it is the separate-tensor
SwiGLU oracle on the two halves (value = up, second half = gate); the bias add
is binary32 addition rounded to bf16 by torch; hand values."""
import numpy as np
import pytest
import torch

import oracle


def _bf16(values) -> np.ndarray:
    return torch.as_tensor(np.asarray(values, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(bits) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("n,f", [(1, 64), (17, 320), (8, 2048)])
def test_without_bias_is_the_swiglu_of_the_halves(n, f):
    rng = np.random.default_rng(f)
    o = _bf16(rng.standard_normal((n, 2 * f)) * 1.5)
    up, gate = o[:, :f], o[:, f:]
    _, _, y = oracle.swiglu_rows(gate, up, None, want_y=True)
    gsf = oracle.global_scale(float(np.abs(_val(y)).max()))
    c1, s1, y1 = oracle.swiglu_packed_rows(o, None, gsf, want_y=True)
    c2, s2, y2 = oracle.swiglu_rows(gate, up, gsf, want_y=True)
    assert np.array_equal(y1, y2) and np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_bias_is_added_in_binary32_and_rounded_to_bf16():
    n, f = 12, 256
    rng = np.random.default_rng(3)
    o = _bf16(rng.standard_normal((n, 2 * f)))
    bias = _bf16(rng.standard_normal(2 * f) * 0.3)
    biased = _bf16(_val(o) + _val(bias)[None, :])  # binary32 sum, torch's bf16 rounding
    _, _, y_packed = oracle.swiglu_packed_rows(o, bias, None, want_y=True)
    _, _, y_split = oracle.swiglu_rows(biased[:, f:], biased[:, :f], None, want_y=True)
    assert np.array_equal(y_packed, y_split)


def test_hand_values():
    f = 64
    # value 1 + bias 3 * 2^-9 rounds to 1 + 2^-7; gate 0 + bias 0 is 0, so y = 0 * ... = 0
    o = np.zeros((1, 2 * f), np.uint16)
    o[0, :f] = _bf16(np.ones(f))
    bias = np.zeros(2 * f, np.uint16)
    bias[:f] = _bf16(np.full(f, 3 * 2.0 ** -9))
    bias[f:] = _bf16(np.full(f, 2.0))  # gate 2: y = bf16(fl(fl(2 * sigma(2)) * (1 + 2^-7)))
    _, _, y = oracle.swiglu_packed_rows(o, bias, None, want_y=True)
    want = oracle.bf16_bits(np.float32(oracle.swiglu_value(2.0, 1 + 2.0 ** -7)))
    assert (y == want).all()
