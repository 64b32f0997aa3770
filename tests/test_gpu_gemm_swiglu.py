"""GPU parity of the block-scaled NVFP4 GEMM with the SwiGLU + NVFP4 epilogue
(h3q_gemm_swiglu_nvfp4), through the C ABI.

The operands are the oracle's NVFP4 quantize of seeded bf16 tensors (so no
input of the oracle comes from the CUDA path).  The tensor cores accumulate in
binary32 in their own order, so the kernel's accumulator (written beside the
outputs for this check) is compared with the oracle's exact sum within

    |acc - exact| <= (k/64 + 1) * 2^-22 * sum_k |a_k b_k|

(one binary32 rounding, or truncation, per K = 64 step of the MMA, plus one for
the step's own sum).  Everything after the accumulator is exact arithmetic of
this library, so codes, swizzled scales (padding rows zero) and y must equal
the oracle's epilogue applied to the kernel's own accumulator bit for bit, on
every row.  Against the oracle's epilogue on the exact sum, y must agree
wherever the kernel's accumulator pair equals the exact one.
"""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
import workloads
from parity import THREADS, bits, check_rows, fill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _nvfp4(t: torch.Tensor):
    """The oracle's NVFP4 of a bf16 tensor under its own amax scale: (codes, logical
    scales, gsf)."""
    b = bits(t)
    g = oracle.global_scale(oracle.amax_bf16(b))
    codes, sf = oracle.quantize_rows(b, g, threads=THREADS)
    return codes, sf, g


def _upload(dev, codes, sf):
    rows, half = codes.shape
    return (torch.from_numpy(codes).to(dev),
            torch.from_numpy(oracle.swizzle_scales(sf, rows, 2 * half)).to(dev))


def _abs_sum(a_codes, a_sf, b_codes, b_sf):
    """sum_k |a_k b_k| (exact, rounded once): the codes with their sign bits cleared."""
    return oracle.nvfp4_gemm(a_codes & 0x77, a_sf, b_codes & 0x77, b_sf, threads=THREADS)


def _operands(dev, m, k, f, seed, w_std=None):
    w = workloads.ffn_up_inputs(dev, rows=m, hidden=k, ffn=f, seed=seed, w_std=w_std)
    a_codes, a_sf, ga = _nvfp4(w["x"])
    b_codes, b_sf, gb = _nvfp4(w["w"])
    alpha = float(np.float32(1.0) / (np.float32(ga) * np.float32(gb)))
    return a_codes, a_sf, b_codes, b_sf, alpha


def _run(dev, a_codes, a_sf, b_codes, b_sf, alpha, gsf, want_acc=True):
    m, k = a_codes.shape[0], 2 * a_codes.shape[1]
    n = b_codes.shape[0]
    A, As = _upload(dev, a_codes, a_sf)
    B, Bs = _upload(dev, b_codes, b_sf)
    acc = fill(torch.empty((m, n), dtype=torch.float32, device=dev)) if want_acc else None
    y = fill(torch.empty((m, n // 2), dtype=torch.bfloat16, device=dev))
    codes = fill(torch.empty((m, n // 4), dtype=torch.uint8, device=dev))
    scales = fill(torch.empty((h3q.padded_rows(m), n // 32), dtype=torch.uint8, device=dev))
    h3q.h3q_gemm_swiglu_nvfp4(A, As, B, Bs, torch.tensor([alpha], device=dev),
                              torch.tensor([gsf], device=dev), codes, scales, y=y, acc=acc)
    torch.cuda.synchronize()
    return codes, scales, y, acc


def _check_acc(got, want, bound, k, what):
    tol = bound.astype(np.float64) * ((k / 64 + 1) * 2.0**-22)
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    worst = float(np.max(err / np.maximum(tol, 1e-300)))
    assert np.isfinite(got).all(), f"{what}: non-finite accumulator"
    assert (err <= tol).all(), f"{what}: accumulator off the exact sum by up to {worst:.3g} of the bound"
    return worst, float(np.mean(got.view(np.uint32) == want.view(np.uint32)))


def _gsf_of(acc_exact, alpha):
    _, _, y = oracle.swiglu_epilogue_rows(acc_exact, alpha, None, want_y=True, threads=THREADS)
    return oracle.global_scale(float(np.abs(oracle.bf16_value(y)).max())), y


@pytest.mark.parametrize("m,k,f", [(1, 256, 128), (5, 256, 256), (200, 768, 384), (128, 7168, 128),
                                   (777, 1024, 768), (2000, 256, 512), (300, 2048, 1280)])
def test_every_output_against_the_oracle(dev, m, k, f):
    a_codes, a_sf, b_codes, b_sf, alpha = _operands(dev, m, k, f, seed=m + k + f)
    exact = oracle.nvfp4_gemm(a_codes, a_sf, b_codes, b_sf, threads=THREADS)
    gsf, y_exact = _gsf_of(exact, alpha)
    codes, scales, y, acc = _run(dev, a_codes, a_sf, b_codes, b_sf, alpha, gsf)
    acc_k = acc.cpu().numpy()
    _check_acc(acc_k, exact, _abs_sum(a_codes, a_sf, b_codes, b_sf), k, f"{m}x{k}x{2 * f}")
    # everything after the accumulator, bit for bit on every row
    co, so, yo = oracle.swiglu_epilogue_rows(acc_k, alpha, gsf, want_y=True, threads=THREADS)
    y_k = bits(y)
    assert np.array_equal(y_k, yo), "y differs from the oracle's epilogue of the kernel's accumulator"
    assert np.array_equal(codes.cpu().numpy(), co), "codes differ"
    want_scales = oracle.swizzle_scales(so, m, f)                   # padding rows zero
    assert np.array_equal(scales.cpu().numpy().ravel(), want_scales), "scales differ"
    # against the exact accumulator: equal wherever the value/gate pair is exact
    same = (acc_k.view(np.uint32) == exact.view(np.uint32))
    pair = same[:, 0::2] & same[:, 1::2]
    assert np.array_equal(y_k[pair], y_exact[pair])


def test_ffn_up_65280x7168x37888(dev):
    """The FFN-up workload (65,280 tokens, hidden 7,168, 2 x 18,944 value/gate rows):
    the epilogue bit for bit on every row against the oracle's epilogue of the
    kernel's accumulator; the accumulator against the exact sum on 64 sampled rows
    (the first 32, the last 16, 16 random)."""
    m, k, f = workloads.TOKENS, workloads.HIDDEN, workloads.FFN
    n = 2 * f
    a_codes, a_sf, b_codes, b_sf, alpha = _operands(dev, m, k, f, seed=8)
    rng = np.random.default_rng(37888)
    sample = np.unique(np.concatenate([np.arange(32), np.arange(m - 16, m), rng.integers(32, m - 16, 16)]))
    exact = oracle.nvfp4_gemm(a_codes[sample], a_sf[sample], b_codes, b_sf, threads=THREADS)
    gsf, _ = _gsf_of(exact, alpha)
    codes, scales, y, acc = _run(dev, a_codes, a_sf, b_codes, b_sf, alpha, gsf)
    idx = torch.as_tensor(sample, device=dev)
    worst, frac = _check_acc(acc.index_select(0, idx).cpu().numpy(), exact,
                             _abs_sum(a_codes[sample], a_sf[sample], b_codes, b_sf), k, "ffn-up sampled rows")
    print(f"accumulator: {frac:.4f} of sampled values exact, worst {worst:.3g} of the bound")
    assert h3q.h3q_kernel_error_flag() == 0
    step = 8192
    for r0 in range(0, m, step):
        r1 = min(m, r0 + step)
        acc_k = acc[r0:r1].cpu().numpy()
        co, so, yo = oracle.swiglu_epilogue_rows(acc_k, alpha, gsf, want_y=True, threads=THREADS)
        assert np.array_equal(bits(y[r0:r1]), yo), f"y differs in rows {r0}..{r1}"
        check_rows(codes, scales, np.arange(r0, r1), f, co, so, f"ffn-up rows {r0}..{r1}")


def test_gates_outside_the_silu_table(dev):
    """alpha scaled up and down so gates leave the SiLU table's window (|g| > 127.5,
    and below 2^-25): the direct SwiGLU paths, bit for bit."""
    m, k, f = 256, 512, 256
    a_codes, a_sf, b_codes, b_sf, alpha = _operands(dev, m, k, f, seed=55)
    for scale in (400.0, 1e-9, 3.0):
        al = float(np.float32(alpha * scale))
        codes, scales, y, acc = _run(dev, a_codes, a_sf, b_codes, b_sf, al, 1.0)
        acc_k = acc.cpu().numpy()
        co, so, yo = oracle.swiglu_epilogue_rows(acc_k, al, 1.0, want_y=True, threads=THREADS)
        assert np.array_equal(bits(y), yo) and np.array_equal(codes.cpu().numpy(), co)
        assert np.array_equal(scales.cpu().numpy().ravel(), oracle.swizzle_scales(so, m, f))


def test_zero_operands_and_padding(dev):
    m, k, f = 70, 256, 128
    a_codes = np.zeros((m, k // 2), np.uint8)
    a_sf = np.zeros((m, k // 16), np.uint8)
    b_codes = np.zeros((2 * f, k // 2), np.uint8)
    b_sf = np.full((2 * f, k // 16), 0x38, np.uint8)
    codes, scales, y, acc = _run(dev, a_codes, a_sf, b_codes, b_sf, 1.0, 1.0)
    assert (acc.cpu().numpy() == 0).all() and (bits(y) == 0).all()
    assert (codes.cpu().numpy() == 0).all() and (scales.cpu().numpy() == 0).all()


def test_outputs_stay_inside_their_buffers_and_repeat(dev):
    """Outputs carved out of sentinel-filled buffers: the guard bytes survive, and a
    second launch on a side stream gives the same bytes without the optional outputs."""
    m, k, f = 333, 512, 384
    a_codes, a_sf, b_codes, b_sf, alpha = _operands(dev, m, k, f, seed=77)
    A, As = _upload(dev, a_codes, a_sf)
    B, Bs = _upload(dev, b_codes, b_sf)
    al = torch.tensor([alpha], device=dev)
    g = torch.tensor([0.5], device=dev)
    nc, ns, ny = m * f // 2, h3q.scale_bytes(m, f), m * f
    guard = 4096
    cbuf = fill(torch.empty(nc + guard, dtype=torch.uint8, device=dev))
    sbuf = fill(torch.empty(ns + guard, dtype=torch.uint8, device=dev))
    ybuf = fill(torch.empty(ny + guard, dtype=torch.bfloat16, device=dev))
    codes, scales, y = cbuf[:nc].view(m, f // 2), sbuf[:ns].view(-1, f // 16), ybuf[:ny].view(m, f)
    h3q.h3q_gemm_swiglu_nvfp4(A, As, B, Bs, al, g, codes, scales, y=y)
    torch.cuda.synchronize()
    assert (cbuf[nc:] == 0xAB).all() and (sbuf[ns:] == 0xAB).all()
    assert (ybuf[ny:].view(torch.int16) == torch.tensor(-21589, dtype=torch.int16, device=dev)).all()  # 0xABAB
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        c2, s2 = h3q.h3q_gemm_swiglu_nvfp4(A, As, B, Bs, al, g, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(c2, codes) and torch.equal(s2, scales)
    assert h3q.h3q_kernel_error_flag() == 0
