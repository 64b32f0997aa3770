"""GPU parity of the residual fold + RMSNorm + AdaLN -> NVFP4 producer, through
the C ABI: the folded residual written back to h (every fp32 bit), the codes and
swizzled scales (every byte, padding rows zero) and each row's rstd equal the
oracle's."""
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


def _oracle(w, frames, gsf, want_y=False):
    return oracle.residual_adaln_rows(
        w["h"].cpu().numpy(), bits(w["o"]), None if w["bias"] is None else bits(w["bias"]),
        bits(w["gate"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"], gsf, want_y=want_y,
        threads=THREADS)


def _gsf(w, frames):
    _, _, _, _, y = _oracle(w, frames, None, want_y=True)
    return oracle.global_scale(float(np.abs(oracle.bf16_value(y)).max()))


def _run(dev, w, gsf, **frame_args):
    rows, cols = w["o"].shape
    codes = fill(torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev))
    scales = fill(torch.empty((h3q.padded_rows(rows), cols // 16), dtype=torch.uint8, device=dev))
    rstd = fill(torch.empty(rows, dtype=torch.float32, device=dev))
    h3q.h3q_residual_rmsnorm_adaln_nvfp4(w["h"], w["o"], w["gate"], w["gamma"], w["table"],
                                         gsf_tensor(gsf, dev), bias=w["bias"], eps=w["eps"],
                                         codes=codes, scales=scales, row_rstd=rstd, **frame_args)
    return codes, scales, rstd


def _check(dev, w, frames, gsf, codes, scales, rstd, h_after, what):
    rows, cols = w["o"].shape
    h_ref, co, so, ro, _ = _oracle(w, frames, gsf)
    assert np.array_equal(h_after.cpu().numpy().view(np.uint32), h_ref.view(np.uint32)), f"{what}: h"
    check_full(codes, scales, rows, cols, co, so, what)
    check_padding(scales, rows, cols, what)
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), ro.view(np.uint32)), f"{what}: rstd"


@pytest.mark.parametrize("rows,cols,frames_n,rpf,with_bias", [
    (1, 64, 1, 1, True), (130, 256, 3, 50, True), (257, 1024, 2, 200, False), (100, 2048, 4, 25, True),
    (300, 4096, 2, 150, True), (457, 7168, 3, 160, True), (64, 8192, 1, 64, False),
    (33, 1088, 4, 9, True), (99, 2560, 2, 50, False),
    # the 7,168-column ring kernel: one row per CTA, no bias, frames changing inside a CTA's rows
    (1, 7168, 1, 1, False), (5, 7168, 2, 3, True), (151, 7168, 2, 100, False), (1000, 7168, 4, 300, True)])
def test_shapes(dev, rows, cols, frames_n, rpf, with_bias):
    w = workloads.residual_inputs(dev, rows=rows, cols=cols, frames=frames_n, rows_per_frame=rpf,
                                  seed=rows + cols, bias=with_bias)
    frames = np.arange(rows) // rpf
    gsf = _gsf(w, frames)
    h_before = w["h"].clone()
    codes, scales, rstd = _run(dev, w, gsf, rows_per_frame=rpf)
    h_after, w["h"] = w["h"], h_before  # the oracle folds the original h
    _check(dev, w, frames, gsf, codes, scales, rstd, h_after, f"residual {rows}x{cols}")


def test_row_frame_array_and_strided_views(dev):
    rows, cols, frames_n = 300, 7168, 5
    w = workloads.residual_inputs(dev, rows=rows, cols=cols + 512, frames=frames_n, seed=9)
    w["h"] = w["h"][:, 256:256 + cols]
    w["o"] = w["o"][:, 128:128 + cols]
    w["bias"] = w["bias"][:cols].contiguous()
    w["gate"] = w["gate"][:, :cols].contiguous()
    w["gamma"] = w["gamma"][:cols].contiguous()
    w["table"] = w["table"][:, :, :cols].contiguous()
    rf = torch.randint(0, frames_n, (rows,), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    gsf = _gsf(w, rf.numpy())
    h_before = w["h"].clone()
    codes, scales, rstd = _run(dev, w, gsf, row_frame=rf.to(dev))
    h_after = w["h"]
    w["h"] = h_before
    _check(dev, w, rf.numpy(), gsf, codes, scales, rstd, h_after, "residual row_frame strided")


def test_full_65280x7168_every_row(dev):
    """The 65,280 x 7,168 workload (32 frames of 2,040 tokens) in the configuration
    the benchmark times: every bit of the folded residual and every output byte."""
    w = workloads.residual_inputs(dev)
    rows = w["o"].shape[0]
    rpf = w["rows_per_frame"]
    frames = np.arange(rows) // rpf
    h_before = w["h"].cpu().numpy()
    gsf = 90.0  # about 2688 / max |y| of this workload (the scale's exact value is immaterial)
    codes, scales, rstd = _run(dev, w, gsf, rows_per_frame=rpf)
    h_after = w["h"]
    w["h"] = torch.from_numpy(h_before)
    _check(dev, w, frames, gsf, codes, scales, rstd, h_after, "residual 65280x7168")
