"""GPU parity of the dynamic and calibrated global scales, through
the C ABI: each producer's abs-max pass equals the oracle's max |y| over the
same bf16 outputs, the device global scale equals the oracle's, the running
maximum folds across calls, and the chained dynamic call (abs-max pass, scale,
producer -- no host synchronisation) writes the oracle's codes and scales."""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
import workloads
from parity import THREADS, bits, check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _f32(v: float) -> int:
    return int(np.float32(v).view(np.uint32))


def _eq(got: torch.Tensor, want: float, what: str):
    g = float(got.item())
    assert _f32(g) == _f32(want), f"{what}: {g!r} != {want!r}"


@pytest.mark.parametrize("rows,cols,strided", [(1, 64, False), (333, 7168, True), (8192, 7168, False), (1000, 18944, False),
                          (70, 1088, True)])
def test_amax_bf16(dev, rows, cols, strided):
    x = workloads.quantize_inputs(dev, rows=rows, cols=cols + (256 if strided else 0), seed=rows)
    if strided:
        x = x[:, 128:128 + cols]
    amax = h3q.h3q_amax_bf16(x)
    _eq(amax, oracle.amax_bf16(bits(x)), f"amax {rows}x{cols}")


def test_running_maximum_folds_across_calls(dev):
    a = workloads.attention_output(dev, tokens=500) * 3
    b = workloads.attention_output(dev, tokens=700)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    h3q.h3q_amax_bf16(b, amax)
    h3q.h3q_amax_bf16(a, amax)
    want = max(oracle.amax_bf16(bits(a)), oracle.amax_bf16(bits(b)))
    _eq(amax, want, "running max")
    amax.fill_(1.0e30)  # a larger running value is kept
    h3q.h3q_amax_bf16(a, amax)
    _eq(amax, 1.0e30, "kept")
    empty = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    h3q.h3q_amax_bf16(empty, amax)  # no rows: nothing launched, amax unchanged
    _eq(amax, 1.0e30, "empty")


def _adaln_amax_oracle(w, frames):
    _, _, _, y = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                   w["eps"], None, want_y=True, threads=THREADS)
    return oracle.amax_bf16(y)


@pytest.mark.parametrize("rows,cols", [(5, 64), (130, 256), (257, 1024), (100, 2048), (300, 4096),
                                       (457, 7168), (64, 8192), (40, 16384), (33, 1088), (99, 2560)])
def test_adaln_amax_every_route(dev, rows, cols):
    """Widths covering every kernel (128-thread resident kernels of 1..8 chunks per
    lane, guarded and guard-free, the 7,168-column block kernel, the generic one)."""
    rpf = max(1, rows // 3)
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=(rows + rpf - 1) // rpf,
                               rows_per_frame=rpf, seed=rows * 7 + cols)
    amax = h3q.h3q_rmsnorm_adaln_amax(w["x"], w["gamma"], w["table"], rows_per_frame=rpf, eps=w["eps"])
    _eq(amax, _adaln_amax_oracle(w, np.arange(rows) // rpf), f"adaln amax {rows}x{cols}")


def test_adaln_amax_row_frame_strided(dev):
    rows, cols = 200, 7168
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols + 512, frames=5, seed=12)
    w["x"] = w["x"][:, 256:256 + cols]
    w["gamma"] = w["gamma"][:cols].contiguous()
    w["table"] = w["table"][:, :, :cols].contiguous()
    rf = torch.randint(0, 5, (rows,), generator=torch.Generator().manual_seed(2), dtype=torch.int32)
    amax = h3q.h3q_rmsnorm_adaln_amax(w["x"], w["gamma"], w["table"], row_frame=rf.to(dev), eps=w["eps"])
    _eq(amax, _adaln_amax_oracle(w, rf.numpy()), "adaln amax row_frame")


@pytest.mark.parametrize("rows", [1, 2, 3, 4, 5, 7, 458, 1001])
def test_adaln_amax_7168_ragged_steps(dev, rows):
    """The 7,168-column block kernel's abs-max instance (its own warp roles) on CTAs of
    one or a few 3-row steps, the last one short, with a row -> frame array."""
    cols, frames_n = 7168, 7
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=frames_n, seed=rows + 90)
    rf = torch.randint(0, frames_n, (rows,), generator=torch.Generator().manual_seed(rows), dtype=torch.int32)
    amax = h3q.h3q_rmsnorm_adaln_amax(w["x"], w["gamma"], w["table"], row_frame=rf.to(dev), eps=w["eps"])
    _eq(amax, _adaln_amax_oracle(w, rf.numpy()), f"adaln amax 7168 ragged {rows}")


@pytest.mark.parametrize("rows,cols,extreme", [(3, 64, False), (131, 320, True), (257, 18944, False),
                                               (64, 8192, True)])
def test_swiglu_amax(dev, rows, cols, extreme):
    gate, up = workloads.swiglu_inputs(dev, rows=rows, cols=cols, seed=rows + cols)
    if extreme:  # gates outside the SiLU table's window send warps to the direct path
        gate.view(-1)[::97] = torch.tensor(-95.0, dtype=torch.bfloat16)
        gate.view(-1)[5::89] = torch.tensor(1.0e-30, dtype=torch.bfloat16)
    amax = h3q.h3q_swiglu_amax(gate, up)
    _, _, y = oracle.swiglu_rows(bits(gate), bits(up), None, want_y=True, threads=THREADS)
    _eq(amax, oracle.amax_bf16(y), f"swiglu amax {rows}x{cols}")


@pytest.mark.parametrize("a", [0.0, 1.0, 2688.0, 6.5, 3.0e38, float("inf"), 1.0e-30, 12345.678, 448.0])
def test_global_scale_from_amax(dev, a):
    amax = torch.tensor([a], dtype=torch.float32, device=dev)
    gsf = h3q.h3q_global_scale_from_amax(amax)
    _eq(gsf, oracle.global_scale_from_amax(a), f"gsf({a})")


def test_dynamic_quantize_chain(dev):
    x = workloads.quantize_inputs(dev, rows=1000, cols=7168, seed=33)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    h3q.h3q_amax_bf16(x, amax)
    gsf = h3q.h3q_global_scale_from_amax(amax)
    codes, scales = h3q.h3q_quantize_nvfp4(x, gsf)
    g = oracle.global_scale_from_amax(oracle.amax_bf16(bits(x)))
    co, so = oracle.quantize_rows(bits(x), g, threads=THREADS)
    check_full(codes, scales, 1000, 7168, co, so, "dynamic quantize")


def test_dynamic_swiglu_chain(dev):
    gate, up = workloads.swiglu_inputs(dev, rows=300, cols=18944, seed=8)
    amax = h3q.h3q_swiglu_amax(gate, up)
    codes, scales = h3q.h3q_swiglu_nvfp4(gate, up, h3q.h3q_global_scale_from_amax(amax))
    _, _, y = oracle.swiglu_rows(bits(gate), bits(up), None, want_y=True, threads=THREADS)
    g = oracle.global_scale_from_amax(oracle.amax_bf16(y))
    co, so, _ = oracle.swiglu_rows(bits(gate), bits(up), g, threads=THREADS)
    check_full(codes, scales, 300, 18944, co, so, "dynamic swiglu")


def test_dynamic_adaln_65280x7168_every_row(dev):
    """The 65,280 x 7,168 AdaLN workload with a per-call abs-max instead of the
    calibrated static scale: the abs-max, the scale, every row's rstd handed from
    the abs-max pass to the second pass, and every byte of the outputs of both
    second passes (the producer forming its own statistics, and the one taking the
    abs-max pass's rstd)."""
    w = workloads.adaln_inputs(dev)
    rows, cols = w["x"].shape
    rpf = w["rows_per_frame"]
    rstd = torch.empty(rows, dtype=torch.float32, device=dev)
    amax = h3q.h3q_rmsnorm_adaln_amax(w["x"], w["gamma"], w["table"], rows_per_frame=rpf, eps=w["eps"],
                                      row_rstd=rstd)
    gsf = h3q.h3q_global_scale_from_amax(amax)
    codes, scales = h3q.h3q_rmsnorm_adaln_nvfp4(w["x"], w["gamma"], w["table"], gsf, rows_per_frame=rpf,
                                                eps=w["eps"])
    codes2, scales2 = h3q.h3q_rmsnorm_adaln_nvfp4_from_rstd(w["x"], w["gamma"], w["table"], rstd, gsf,
                                                            rows_per_frame=rpf)
    frames = np.arange(rows) // rpf
    _, _, _, y = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"],
                                   None, want_y=True, threads=THREADS)
    a = oracle.amax_bf16(y)
    _eq(amax, a, "full-size amax")
    g = oracle.global_scale_from_amax(a)
    _eq(gsf, g, "full-size gsf")
    co, so, rstd_o, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"],
                                          g, threads=THREADS)
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), rstd_o.view(np.uint32)), "abs-max pass rstd"
    check_full(codes, scales, rows, cols, co, so, "dynamic adaln 65280x7168")
    check_full(codes2, scales2, rows, cols, co, so, "dynamic adaln from rstd 65280x7168")


def test_adaln_7168_short_frames(dev):
    """The 7,168-column block kernel with two rows per frame and about 30 rows per
    CTA: each lane's rows three apart cross one or two frame boundaries a step, in
    the abs-max pass (which takes its rows downwards) and in both producers.  The
    pass's maximum and rstd, and the codes and scales of the producer forming its
    own statistics and of the one given the rstd, against the oracle."""
    rows, cols, rpf = 4561, 7168, 2
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=(rows + rpf - 1) // rpf, rows_per_frame=rpf,
                               seed=77)
    frames = np.arange(rows) // rpf
    rstd = torch.empty(rows, dtype=torch.float32, device=dev)
    amax = h3q.h3q_rmsnorm_adaln_amax(w["x"], w["gamma"], w["table"], rows_per_frame=rpf, eps=w["eps"],
                                      row_rstd=rstd)
    gsf = h3q.h3q_global_scale_from_amax(amax)
    c1, s1 = h3q.h3q_rmsnorm_adaln_nvfp4_from_rstd(w["x"], w["gamma"], w["table"], rstd, gsf, rows_per_frame=rpf)
    c2, s2 = h3q.h3q_rmsnorm_adaln_nvfp4(w["x"], w["gamma"], w["table"], gsf, rows_per_frame=rpf, eps=w["eps"])
    _, _, _, y = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"],
                                   None, want_y=True, threads=THREADS)
    _eq(amax, oracle.amax_bf16(y), "adaln amax short frames")
    g = oracle.global_scale_from_amax(oracle.amax_bf16(y))
    co, so, rstd_o, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"],
                                          g, threads=THREADS)
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), rstd_o.view(np.uint32)), "abs-max pass rstd"
    check_full(c1, s1, rows, cols, co, so, "adaln from rstd, short frames")
    check_full(c2, s2, rows, cols, co, so, "adaln, short frames")


@pytest.mark.parametrize("rows,cols,use_row_frame", [(5, 64, False), (130, 256, True), (257, 1024, False),
                                                     (100, 2048, True), (1, 7168, False), (4, 7168, True),
                                                     (457, 7168, False), (458, 7168, True), (64, 8192, False),
                                                     (40, 16384, True), (33, 1088, False)])
def test_adaln_from_rstd_every_route(dev, rows, cols, use_row_frame):
    """The abs-max pass's row_rstd equals the oracle's rstd bit for bit, and the
    producer given it writes the oracle's codes and scales, on every kernel route
    (resident kernels, the 7,168-column block kernel with its short last steps, the
    generic one), with rows_per_frame and with a row -> frame array."""
    frames_n = 5
    rpf = max(1, (rows + frames_n - 1) // frames_n)
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=frames_n, rows_per_frame=rpf,
                               seed=rows * 3 + cols)
    if use_row_frame:
        rf = torch.randint(0, frames_n, (rows,), generator=torch.Generator().manual_seed(rows), dtype=torch.int32)
        frames = rf.numpy()
        kw = {"row_frame": rf.to(dev)}
    else:
        frames = np.arange(rows) // rpf
        kw = {"rows_per_frame": rpf}
    rstd = torch.empty(rows, dtype=torch.float32, device=dev)
    amax = h3q.h3q_rmsnorm_adaln_amax(w["x"], w["gamma"], w["table"], eps=w["eps"], row_rstd=rstd, **kw)
    gsf = h3q.h3q_global_scale_from_amax(amax)
    codes, scales = h3q.h3q_rmsnorm_adaln_nvfp4_from_rstd(w["x"], w["gamma"], w["table"], rstd, gsf, **kw)
    _, _, _, y = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"],
                                   None, want_y=True, threads=THREADS)
    g = oracle.global_scale_from_amax(oracle.amax_bf16(y))
    _eq(gsf, g, f"gsf {rows}x{cols}")
    co, so, rstd_o, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"],
                                          g, threads=THREADS)
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), rstd_o.view(np.uint32)), f"rstd {rows}x{cols}"
    check_full(codes, scales, rows, cols, co, so, f"adaln from rstd {rows}x{cols}")
