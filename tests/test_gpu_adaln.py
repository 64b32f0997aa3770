"""GPU parity of the fused RMSNorm + AdaLN -> NVFP4 producer (a), through the C ABI."""
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


def _oracle_gsf(w, frames, rows_sel=None):
    x = w["x"] if rows_sel is None else w["x"][rows_sel]
    _, _, _, y = oracle.adaln_rows(bits(x), bits(w["gamma"]), bits(w["table"]), frames, w["eps"],
                                   None, want_y=True, threads=THREADS)
    return oracle.global_scale(float(np.abs(oracle.bf16_value(y)).max()))


def _run(dev, w, gsf, row_frame=None, rows_per_frame=None):
    rows, cols = w["x"].shape
    codes = fill(torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev))
    scales = fill(torch.empty((h3q.padded_rows(rows), cols // 16), dtype=torch.uint8, device=dev))
    rstd = fill(torch.empty(rows, dtype=torch.float32, device=dev))
    h3q.h3q_rmsnorm_adaln_nvfp4(w["x"], w["gamma"], w["table"], gsf_tensor(gsf, dev),
                                row_frame=row_frame, rows_per_frame=rows_per_frame, eps=w["eps"],
                                codes=codes, scales=scales, row_rstd=rstd)
    return codes, scales, rstd


def test_tiny_64x256(dev):
    """x [64, 256] ~ N(0,1), gamma ~ N(1, 0.1), table [4, 2, 256] ~ N(0, 0.2), frame =
    row // 16, eps 1e-6, gsf from the oracle's max |modulated x|: every byte."""
    w = workloads.tiny_adaln_inputs(dev)
    frames = np.arange(64) // 16
    gsf = _oracle_gsf(w, frames)
    codes, scales, rstd = _run(dev, w, gsf, rows_per_frame=16)
    co, so, ro, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                      w["eps"], gsf)
    check_full(codes, scales, 64, 256, co, so, "tiny adaln")
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32))
    check_padding(scales, 64, 256, "tiny adaln")


@pytest.mark.parametrize("rows,cols,frames_n,rpf", [
    (1, 64, 1, 1), (2, 128, 2, 1), (129, 256, 3, 50), (300, 7168, 3, 100), (70, 8192, 2, 40),
    (40, 16384, 1, 40), (33, 1088, 4, 9), (130, 2560, 2, 65), (255, 7168, 32, 8), (128, 4096, 1, 128)])
def test_shapes(dev, rows, cols, frames_n, rpf):
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=frames_n, rows_per_frame=rpf,
                               seed=rows * 31 + cols)
    frames = np.arange(rows) // rpf
    gsf = _oracle_gsf(w, frames)
    codes, scales, rstd = _run(dev, w, gsf, rows_per_frame=rpf)
    co, so, ro, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                      w["eps"], gsf, threads=THREADS)
    check_full(codes, scales, rows, cols, co, so, f"adaln {rows}x{cols}")
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32))


def test_row_frame_array_and_strided_x(dev):
    rows, cols, frames_n = 200, 2048, 5
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols + 512, frames=frames_n, seed=5)
    w["x"] = w["x"][:, 256:256 + cols]
    w["gamma"] = w["gamma"][:cols].contiguous()
    w["table"] = w["table"][:, :, :cols].contiguous()
    gen = torch.Generator(device="cpu").manual_seed(3)
    rf = torch.randint(0, frames_n, (rows,), generator=gen, dtype=torch.int32)
    gsf = _oracle_gsf(w, rf.numpy())
    codes, scales, rstd = _run(dev, w, gsf, row_frame=rf.to(dev))
    co, so, ro, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), rf.numpy(),
                                      w["eps"], gsf, threads=THREADS)
    check_full(codes, scales, rows, cols, co, so, "adaln row_frame")
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32))


@pytest.mark.parametrize("rows", [1, 2, 3, 4, 5, 7, 457, 1000])
def test_7168_row_frame_array_strided_and_ragged_steps(dev, rows):
    """The 7,168-column kernel (three rows per step, one block per thread) with a
    per-row random frame (frames change inside every step), x as a strided view,
    row counts that leave partial steps and CTAs with one or two rows, and the
    per-row rstd output."""
    cols, frames_n = 7168, 7
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols + 256, frames=frames_n, seed=rows + 70)
    w["x"] = w["x"][:, 128:128 + cols]
    w["gamma"] = w["gamma"][:cols].contiguous()
    w["table"] = w["table"][:, :, :cols].contiguous()
    gen = torch.Generator(device="cpu").manual_seed(rows)
    rf = torch.randint(0, frames_n, (rows,), generator=gen, dtype=torch.int32)
    gsf = _oracle_gsf(w, rf.numpy())
    codes, scales, rstd = _run(dev, w, gsf, row_frame=rf.to(dev))
    co, so, ro, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), rf.numpy(),
                                      w["eps"], gsf, threads=THREADS)
    check_full(codes, scales, rows, cols, co, so, f"adaln 7168 row_frame {rows}")
    check_padding(scales, rows, cols, f"adaln 7168 row_frame {rows}")
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32))


def test_7168_zero_rows_and_eps(dev):
    """All-zero and constant rows at 7,168 columns, eps 0 and 0.5."""
    rows, cols = 96, 7168
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=2, rows_per_frame=48, seed=31)
    w["x"][5:9] = 0
    w["x"][20:23] = -2.5
    for eps in (0.5, 0.0):
        if eps == 0.0:
            w["x"][5:9] = 0.125  # keep rstd finite
        w["eps"] = eps
        frames = np.arange(rows) // 48
        gsf = _oracle_gsf(w, frames)
        codes, scales, rstd = _run(dev, w, gsf, rows_per_frame=48)
        co, so, ro, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                          eps, gsf, threads=THREADS)
        check_full(codes, scales, rows, cols, co, so, f"adaln 7168 eps={eps}")
        assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32))


def test_eps_and_constant_rows(dev):
    """All-zero rows (rstd = 1/sqrt(eps)), constant rows and a large eps."""
    rows, cols = 64, 512
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=1, rows_per_frame=rows, seed=8)
    w["x"][:8] = 0
    w["x"][8:16] = 1.5
    for eps in (1e-6, 0.5, 0.0):
        if eps == 0.0:
            w["x"][:8] = 0.25  # keep rstd finite
        w["eps"] = eps
        frames = np.zeros(rows, np.int64)
        gsf = _oracle_gsf(w, frames)
        codes, scales, rstd = _run(dev, w, gsf, rows_per_frame=rows)
        co, so, ro, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                          eps, gsf)
        check_full(codes, scales, rows, cols, co, so, f"adaln eps={eps}")
        assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32))


def test_full_65280x7168_every_row(dev):
    """The 65,280 x 7,168 workload (32 frames of 2,040 tokens, per-channel LogNormal
    scales) in the launch configuration the benchmark times: every byte of the codes
    and of the swizzled scales, and every row's rstd, against the oracle."""
    w = workloads.adaln_inputs(dev)
    rows, cols = w["x"].shape
    frames = np.arange(rows) // w["rows_per_frame"]
    calib = workloads.sample_rows(rows, seed=3).numpy()
    gsf = _oracle_gsf(w, calib // w["rows_per_frame"], torch.as_tensor(calib, device=dev))
    codes, scales, rstd = _run(dev, w, gsf, rows_per_frame=w["rows_per_frame"])
    co, so, ro, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                      w["eps"], gsf, threads=THREADS)
    check_full(codes, scales, rows, cols, co, so, "adaln 65280x7168")
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32))


def test_rstd_within_stated_tolerance_of_binary64(dev):
    w = workloads.adaln_inputs(dev, rows=256, cols=7168, seed=17)
    frames = np.arange(256) // 2040
    gsf = _oracle_gsf(w, frames)
    _, _, rstd = _run(dev, w, gsf, rows_per_frame=2040)
    xf = oracle.bf16_value(bits(w["x"])).astype(np.float64)
    exact = 1 / np.sqrt((xf * xf).mean(1) + np.float64(np.float32(1e-6)))
    rel = np.abs(rstd.cpu().numpy() - exact) / exact
    assert rel.max() <= 1e-6


def test_repeated_unsynchronised(dev):
    w = workloads.adaln_inputs(dev, rows=1024, cols=7168, frames=2, rows_per_frame=512, seed=11)
    frames = np.arange(1024) // 512
    gsf = gsf_tensor(_oracle_gsf(w, frames), dev)
    outs = [h3q.h3q_rmsnorm_adaln_nvfp4(w["x"], w["gamma"], w["table"], gsf, rows_per_frame=512)
            for _ in range(5)]
    torch.cuda.synchronize()
    co, so, _, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                     w["eps"], float(gsf.item()), threads=THREADS)
    for codes, scales in outs:
        check_full(codes, scales, 1024, 7168, co, so, "adaln repeat")


def test_maximum_width(dev):
    """Rows of 2^24 columns, the widest the ABI accepts (the generic kernel: x read
    twice, tables per row)."""
    rows, cols = 2, 1 << 24
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=1, rows_per_frame=rows, seed=77)
    frames = np.zeros(rows, np.int64)
    gsf = _oracle_gsf(w, frames)
    codes, scales, rstd = _run(dev, w, gsf, rows_per_frame=rows)
    co, so, ro, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"],
                                      gsf, threads=THREADS)
    check_full(codes, scales, rows, cols, co, so, "adaln 2 x 2^24")
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32))
