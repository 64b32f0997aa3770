"""GPU parity of the attention-output quantize at the large-index boundary.

The attention output [B=1, S, H=56, D=128] is quantized along H*D = 7,168.
S = 300,000 gives 2,150,400,000 elements, past 2^31 (the FastVideo commit log's
int64 fix: for 56 x 128 the int32 product wraps from 299,593 tokens on).
"""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
import workloads
from parity import THREADS, bits, check_full, check_padding, check_rows, fill, gsf_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def test_ragged_1000_tokens_every_byte(dev):
    x = workloads.attention_output(dev, tokens=1000)
    gsf = oracle.global_scale(float(x.float().abs().max()))
    codes = fill(torch.empty((1000, 3584), dtype=torch.uint8, device=dev))
    scales = fill(torch.empty((1024, 448), dtype=torch.uint8, device=dev))
    h3q.h3q_quantize_nvfp4(x, gsf_tensor(gsf, dev), codes, scales)
    co, so = oracle.quantize_rows(bits(x), gsf, threads=THREADS)
    check_full(codes, scales, 1000, 7168, co, so, "attention output S=1000")
    check_padding(scales, 1000, 7168, "attention output S=1000")


@pytest.mark.parametrize("tokens", [65280, 300000])
def test_every_row(dev, tokens):
    """Every byte of codes and swizzled scales against the oracle; at S = 300,000 the
    tensor holds 2,150,400,000 elements, so rows past 2^31 elements are included."""
    x = workloads.attention_output(dev, tokens=tokens)
    assert x.numel() > 2**31 or tokens < 299593
    gsf = oracle.global_scale(float(x.abs().max().float()))
    codes = fill(torch.empty((tokens, 3584), dtype=torch.uint8, device=dev))
    scales = fill(torch.empty((h3q.padded_rows(tokens), 448), dtype=torch.uint8, device=dev))
    h3q.h3q_quantize_nvfp4(x, gsf_tensor(gsf, dev), codes, scales)
    co, so = oracle.quantize_rows(bits(x), gsf, threads=THREADS)
    check_full(codes, scales, tokens, 7168, co, so, f"attention output S={tokens}")
    check_padding(scales, tokens, 7168, f"attention output S={tokens}")


def test_dequantize_past_2_31_elements(dev):
    """The dequantize on the S = 300,000 attention output (2,150,400,000 elements, so
    output offsets past 2^31): rows 0-255, the last 256 and 4,096 random rows of its
    fp32 output, bit for bit against the oracle's dequantize of the oracle's codes and
    scales of the same rows."""
    tokens, cols = 300000, 7168
    x = workloads.attention_output(dev, tokens=tokens)
    assert x.numel() > 2**31
    gsf = oracle.global_scale(float(x.abs().max().float()))
    g = gsf_tensor(gsf, dev)
    codes, scales = h3q.h3q_quantize_nvfp4(x, g)
    out = h3q.h3q_dequantize_nvfp4(codes, scales, g)
    del codes, scales
    rng = np.random.default_rng(2031)
    sample = np.unique(np.concatenate([np.arange(256), np.arange(tokens - 256, tokens),
                                       rng.integers(256, tokens - 256, 4096)]))
    assert sample.max() * cols > 2**31
    idx = torch.as_tensor(sample, device=dev)
    got = out.index_select(0, idx).cpu().numpy()
    co, so = oracle.quantize_rows(bits(x.index_select(0, idx)), gsf, threads=THREADS)
    want = oracle.dequantize_rows(co, so, gsf, threads=THREADS)
    bad = np.nonzero((got.view(np.uint32) != want.view(np.uint32)).any(1))[0]
    assert bad.size == 0, f"dequantize differs in rows {sample[bad[:8]].tolist()}"
