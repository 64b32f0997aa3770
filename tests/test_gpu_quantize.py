"""GPU parity of the standalone quantize and the dequantize, through the C ABI."""
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


def _amax_gsf(x):
    return oracle.global_scale(float(x.float().abs().max()))


def test_quantize_8192x7168_student_t_with_planted_blocks(dev):
    """Student-t(3) x 2, 0.1% zero blocks, 0.1% single 1e3 outliers; every byte."""
    x = workloads.quantize_inputs(dev)
    gsf = _amax_gsf(x)
    codes, scales = h3q.h3q_quantize_nvfp4(x, gsf_tensor(gsf, dev))
    co, so = oracle.quantize_rows(bits(x), gsf, threads=THREADS)
    check_full(codes, scales, 8192, 7168, co, so, "quantize 8192x7168")


@pytest.mark.parametrize("rows,cols", [(1, 64), (2, 128), (127, 64), (128, 128), (129, 192),
                                       (300, 448), (257, 576), (64, 7232), (33, 1088),
                                       (520, 512), (131, 18944)])
def test_quantize_shapes(dev, rows, cols):
    x = workloads.quantize_inputs(dev, rows=rows, cols=cols, seed=rows * 7 + cols,
                                  zero_frac=0.02, outlier_frac=0.02)
    gsf = _amax_gsf(x)
    codes = fill(torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev))
    scales = fill(torch.empty((h3q.padded_rows(rows), cols // 16), dtype=torch.uint8, device=dev))
    h3q.h3q_quantize_nvfp4(x, gsf_tensor(gsf, dev), codes, scales)
    co, so = oracle.quantize_rows(bits(x), gsf, threads=THREADS)
    check_full(codes, scales, rows, cols, co, so, f"quantize {rows}x{cols}")
    check_padding(scales, rows, cols, f"quantize {rows}x{cols}")


def test_quantize_strided_view(dev):
    """An input whose rows are spaced wider than its width (ld > cols)."""
    base = workloads.quantize_inputs(dev, rows=200, cols=1024, seed=77)
    x = base[:, 256:768]
    assert x.stride(0) == 1024
    gsf = _amax_gsf(x)
    codes, scales = h3q.h3q_quantize_nvfp4(x, gsf_tensor(gsf, dev))
    co, so = oracle.quantize_rows(bits(x), gsf)
    check_full(codes, scales, 200, 512, co, so, "strided quantize")


def _every_bf16_block_rows(sign_peak=1.0):
    """Rows whose blocks hold 15 bf16 values each plus one element of magnitude 6,
    covering every finite bf16 value v with |v| <= 6.  With gsf = 1 each block's
    scale is 1, so each code is E2M1(v) of one bf16 value."""
    mags = np.arange(0, 0x40C1, dtype=np.uint32) << 16  # +0 .. 6.0
    vals = np.concatenate([mags, mags | 0x80000000]).view(np.float32)
    per = 15
    nblk = -(-vals.size // per)
    padded = np.zeros(nblk * per, np.float32)
    padded[: vals.size] = vals
    blocks = np.zeros((nblk, 16), np.float32)
    blocks[:, :per] = padded.reshape(nblk, per)
    blocks[:, per] = 6.0 * sign_peak
    cols = 7168
    per_row = cols // 16
    nrows = -(-nblk // per_row)
    full = np.zeros((nrows * per_row, 16), np.float32)
    full[:nblk] = blocks
    full[nblk:, 0] = 6.0
    return full.reshape(nrows, cols)


@pytest.mark.parametrize("sign_peak", [1.0, -1.0])
def test_quantize_every_bf16_value_through_e2m1(dev, sign_peak):
    x = torch.from_numpy(_every_bf16_block_rows(sign_peak)).to(torch.bfloat16).to(dev)
    codes, scales = h3q.h3q_quantize_nvfp4(x, gsf_tensor(1.0, dev))
    co, so = oracle.quantize_rows(bits(x), 1.0)
    assert (so == 0x38).all()
    check_full(codes, scales, x.shape[0], x.shape[1], co, so, "every bf16 value")


def test_quantize_scale_sweep(dev):
    """Blocks whose amax sweeps 2^-30 .. 2^20 under several global scales, so that
    every E4M3 scale code, subnormal scales, underflow to a zero scale and
    saturation at 448 all occur."""
    rng = np.random.default_rng(8)
    rows, cols = 256, 4096
    blk = rng.standard_normal((rows * cols // 16, 16)).astype(np.float32)
    amax = np.exp2(rng.uniform(-30, 20, blk.shape[0])).astype(np.float32)
    blk *= (amax / np.abs(blk).max(1))[:, None]
    x = torch.from_numpy(blk.reshape(rows, cols)).to(torch.bfloat16).to(dev)
    seen = set()
    for gsf in (1.0, 0.37, 2.688, 1000.0, 3.0e-4):
        codes, scales = h3q.h3q_quantize_nvfp4(x, gsf_tensor(gsf, dev))
        co, so = oracle.quantize_rows(bits(x), gsf, threads=THREADS)
        check_full(codes, scales, rows, cols, co, so, f"scale sweep gsf={gsf}")
        seen.update(np.unique(so).tolist())
    assert len(seen) == 127, f"only {len(seen)} of the 127 scale codes occurred"


def test_quantize_zero_rows_is_a_noop(dev):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    codes, scales = h3q.h3q_quantize_nvfp4(x, gsf_tensor(1.0, dev))
    assert codes.shape == (0, 128) and scales.shape == (0, 16)


def test_quantize_on_a_side_stream_and_repeated_unsynchronised(dev):
    x = workloads.quantize_inputs(dev, rows=1000, cols=7168, seed=9)
    gsf = gsf_tensor(_amax_gsf(x), dev)
    s = torch.cuda.Stream()
    outs = []
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(6):
            outs.append(h3q.h3q_quantize_nvfp4(x, gsf, stream=s))
    torch.cuda.synchronize()
    co, so = oracle.quantize_rows(bits(x), float(gsf.item()), threads=THREADS)
    for codes, scales in outs:
        check_full(codes, scales, 1000, 7168, co, so, "side-stream repeat")


def test_dequantize_matches_oracle(dev):
    x = workloads.quantize_inputs(dev, rows=300, cols=2048, seed=12)
    gsf = _amax_gsf(x)
    g = gsf_tensor(gsf, dev)
    codes, scales = h3q.h3q_quantize_nvfp4(x, g)
    out = h3q.h3q_dequantize_nvfp4(codes, scales, g)
    co, so = oracle.quantize_rows(bits(x), gsf)
    want = oracle.dequantize_rows(co, so, gsf)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_dequantize_random_codes_every_scale(dev):
    """Random codes under every scale code; global scales that keep every value
    normal and ones that push the small scales' values below the normal range
    (2^120: subnormal and zero results) or the large ones' past it (2^-118: inf)."""
    rng = np.random.default_rng(14)
    rows, cols = 129, 640
    codes = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    sf = rng.integers(0, 0x7F, (rows, cols // 16), dtype=np.uint8)
    scales = oracle.swizzle_scales(sf, rows, cols)
    for gsf in (1.0, 0.001, 123.5, 2.0**120, 2.0**-118):
        out = h3q.h3q_dequantize_nvfp4(torch.from_numpy(codes).to(dev),
                                       torch.from_numpy(scales.reshape(-1, cols // 16)).to(dev),
                                       gsf_tensor(gsf, dev))
        want = oracle.dequantize_rows(codes, sf, gsf)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_outputs_do_not_spill_past_their_buffers(dev):
    """Outputs are carved out of larger sentinel-filled buffers; the guard bytes
    after each must survive and every byte inside must be written."""
    rows, cols = 133, 704
    x = workloads.quantize_inputs(dev, rows=rows, cols=cols, seed=21)
    gsf = _amax_gsf(x)
    nc, ns = rows * cols // 2, h3q.scale_bytes(rows, cols)
    guard = 4096
    cbuf = fill(torch.empty(nc + guard, dtype=torch.uint8, device=dev))
    sbuf = fill(torch.empty(ns + guard, dtype=torch.uint8, device=dev))
    codes = cbuf[:nc].view(rows, cols // 2)
    scales = sbuf[:ns].view(-1, cols // 16)
    h3q.h3q_quantize_nvfp4(x, gsf_tensor(gsf, dev), codes, scales)
    assert (cbuf[nc:] == 0xAB).all() and (sbuf[ns:] == 0xAB).all()
    co, so = oracle.quantize_rows(bits(x), gsf)
    check_full(codes, scales, rows, cols, co, so, "guarded quantize")


def test_quantize_maximum_width(dev):
    """Rows of 2^24 columns, the widest the ABI accepts."""
    x = workloads.quantize_inputs(dev, rows=3, cols=1 << 24, seed=78)
    g = oracle.global_scale(float(x.float().abs().max()))
    codes, scales = h3q.h3q_quantize_nvfp4(x, gsf_tensor(g, dev))
    co, so = oracle.quantize_rows(bits(x), g, threads=THREADS)
    check_full(codes, scales, 3, 1 << 24, co, so, "quantize 3 x 2^24")
