"""The oracle's dynamic-scale functions (per-call abs-max and the global scale
derived from it) against what the definition fixes: hand values, numpy's own
maximum over torch's bf16 -> fp32 conversion, the closed form 2688 / amax in
numpy binary32, and the readings for amax = 0 and +inf."""
import numpy as np
import pytest
import torch

import oracle


def _bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_amax_hand_values():
    assert oracle.amax_bf16(_bits([0.0, -0.0, 1.5, -3.0, 2.0])) == 3.0
    assert oracle.amax_bf16(_bits([-0.0, 0.0])) == 0.0
    assert oracle.amax_bf16(np.zeros(0, np.uint16)) == 0.0
    assert oracle.amax_bf16(_bits([1.0, -float("inf")])) == float("inf")
    tiny = np.array([0x0001, 0x8003], np.uint16)  # bf16 subnormals: 2^-133 and -3 * 2^-133
    assert oracle.amax_bf16(tiny) == np.float32(3 * 2.0 ** -133)


def test_amax_matches_numpy_on_every_finite_bf16_value():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = bits[(bits & 0x7FFF) < 0x7F80]
    values = torch.from_numpy(finite.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert oracle.amax_bf16(finite) == np.abs(values).max()
    rng = np.random.default_rng(5)
    for _ in range(20):
        sample = rng.choice(finite, size=int(rng.integers(1, 5000)))
        vals = torch.from_numpy(sample.view(np.int16)).view(torch.bfloat16).float().numpy()
        assert oracle.amax_bf16(sample) == np.abs(vals).max()


def test_running_maximum_is_the_maximum_of_the_concatenation():
    rng = np.random.default_rng(9)
    parts = [_bits(rng.standard_normal(n) * s) for n, s in ((100, 1.0), (50, 7.0), (300, 0.1))]
    running = 0.0
    for p in parts:
        running = max(running, oracle.amax_bf16(p))
    assert running == oracle.amax_bf16(np.concatenate(parts))


@pytest.mark.parametrize("amax", [2688.0, 1.0, 6.0, 448.0, 3.0e38, 1.0e-30, 0.1, 12345.678])
def test_global_scale_closed_form(amax):
    a = np.float32(amax)
    assert oracle.global_scale_from_amax(float(a)) == np.float32(2688.0) / a
    assert oracle.global_scale_from_amax(float(a)) == oracle.global_scale(float(a))


def test_global_scale_readings_for_zero_and_inf():
    assert oracle.global_scale_from_amax(0.0) == 1.0
    fmax = np.finfo(np.float32).max
    assert oracle.global_scale_from_amax(float("inf")) == np.float32(2688.0) / fmax
    assert oracle.global_scale_from_amax(2688.0) == 1.0
