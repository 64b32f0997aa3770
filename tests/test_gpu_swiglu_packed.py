"""GPU parity of the SwiGLU of a value-first packed projection with its bias,
through the C ABI: every code and scale byte equals the oracle's,
with and without a bias, through the SiLU table and the direct path, for strided
rows and the 65,280 x 18,944 workload."""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
import workloads
from parity import THREADS, bits, check_full, check_padding, fill, gsf_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _packed(dev, rows, f, seed, pad=0):
    gate, up = workloads.swiglu_inputs(dev, rows=rows, cols=f, seed=seed)
    o = torch.empty((rows, 2 * f + pad), dtype=torch.bfloat16, device=dev)
    o[:, :f] = up
    o[:, f:2 * f] = gate
    gen = torch.Generator(device=dev).manual_seed(seed + 1)
    bias = (torch.randn(2 * f, generator=gen, device=dev) * 0.2).to(torch.bfloat16)
    return o[:, :2 * f], bias


def _check(dev, o, bias, what):
    rows, two_f = o.shape
    f = two_f // 2
    b_bits = None if bias is None else bits(bias)
    _, _, y = oracle.swiglu_packed_rows(bits(o), b_bits, None, want_y=True, threads=THREADS)
    gsf = oracle.global_scale(float(np.abs(oracle.bf16_value(y)).max()))
    codes = fill(torch.empty((rows, f // 2), dtype=torch.uint8, device=dev))
    scales = fill(torch.empty((h3q.padded_rows(rows), f // 16), dtype=torch.uint8, device=dev))
    h3q.h3q_swiglu_packed_nvfp4(o, gsf_tensor(gsf, dev), bias=bias, codes=codes, scales=scales)
    co, so, _ = oracle.swiglu_packed_rows(bits(o), b_bits, gsf, threads=THREADS)
    check_full(codes, scales, rows, f, co, so, what)
    check_padding(scales, rows, f, what)


@pytest.mark.parametrize("rows,f,with_bias,pad", [(1, 64, True, 0), (131, 320, True, 64),
                                                  (257, 18944, True, 0), (64, 1024, False, 0),
                                                  (200, 2048, True, 256)])
def test_shapes(dev, rows, f, with_bias, pad):
    o, bias = _packed(dev, rows, f, seed=rows + f, pad=pad)
    _check(dev, o, bias if with_bias else None, f"packed {rows}x{f} bias={with_bias}")


def test_extreme_gates_with_bias(dev):
    """Gates that the bias pushes out of the SiLU table's window (and beyond +-87),
    so that warps take the direct computation."""
    rows, f = 96, 1024
    o, bias = _packed(dev, rows, f, seed=77)
    g = o[:, f:]
    g[:, ::101] = -95.0
    g[::3, 7::89] = 1.0e-30
    bias[f + 3::64] = torch.tensor(120.0, dtype=torch.bfloat16)
    _check(dev, o, bias, "packed extreme gates")


def test_full_65280x18944(dev):
    o, bias = _packed(dev, 65280, 18944, seed=4)
    _check(dev, o, bias, "packed 65280x18944")
