"""The host-buffer call of the RMSNorm + AdaLN -> NVFP4 producer
(h3q_rmsnorm_adaln_nvfp4_host, through HostPipeline): pinned host inputs and
outputs, chunks of 128-row multiples, the copies inside the library call.  Its
outputs must equal the oracle's byte for byte (small cases) and the single
device-buffer call's (the 65,280 x 7,168 workload)."""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
import workloads
from nvfp4_activation_quantize_gb300.host import HostPipeline
from parity import THREADS, bits, check_full, gsf_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _host_outputs(rows, cols):
    codes = torch.full((rows, cols // 2), 0xAB, dtype=torch.uint8).pin_memory()
    scales = torch.full((h3q.padded_rows(rows), cols // 16), 0xAB, dtype=torch.uint8).pin_memory()
    return codes, scales


def _gsf(w, frames):
    _, _, _, y = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                   w["eps"], None, want_y=True, threads=THREADS)
    return oracle.global_scale(float(np.abs(oracle.bf16_value(y)).max()))


@pytest.mark.parametrize("rows,cols,rpf,chunk", [
    (300, 1024, 100, 128),     # ragged last chunk (44 rows), frames across chunk edges
    (1000, 2048, 77, 256),     # more chunks than slots
    (128, 512, 128, 128),      # one chunk
    (5, 7168, 2, 8192),        # fewer rows than a tile
    (1300, 640, 1300, 128),    # eleven chunks through three slots
])
def test_matches_oracle(dev, rows, cols, rpf, chunk):
    w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=(rows + rpf - 1) // rpf,
                               rows_per_frame=rpf, seed=rows + cols)
    frames = np.arange(rows) // rpf
    gsf = _gsf(w, frames)
    pipe = HostPipeline(dev, max_cols=cols, chunk_rows=chunk)
    hc, hs = _host_outputs(rows, cols)
    hx = w["x"].cpu().pin_memory()
    pipe.rmsnorm_adaln_nvfp4(hx, w["gamma"].cpu(), w["table"].cpu(), gsf_tensor(gsf, "cpu"), hc, hs,
                             rows_per_frame=rpf, eps=w["eps"])
    torch.cuda.current_stream(dev).synchronize()
    co, so, _, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames,
                                     w["eps"], gsf, threads=THREADS)
    check_full(hc, hs, rows, cols, co, so, f"host pipeline {rows}x{cols}")


def test_host_row_frame_and_reuse(dev):
    """A host row_frame array, then the same pipeline reused for another shape."""
    pipe = HostPipeline(dev, max_cols=4096, chunk_rows=256)
    for rows, cols, seed in ((700, 4096, 1), (513, 1024, 2)):
        w = workloads.adaln_inputs(dev, rows=rows, cols=cols, frames=6, seed=seed)
        rf = torch.randint(0, 6, (rows,), generator=torch.Generator().manual_seed(seed),
                           dtype=torch.int32)
        gsf = _gsf(w, rf.numpy())
        hc, hs = _host_outputs(rows, cols)
        pipe.rmsnorm_adaln_nvfp4(w["x"].cpu().pin_memory(), w["gamma"], w["table"],
                                 gsf_tensor(gsf, dev), hc, hs, row_frame=rf, eps=w["eps"])
        torch.cuda.synchronize()
        co, so, _, _ = oracle.adaln_rows(bits(w["x"]), bits(w["gamma"]), bits(w["table"]),
                                         rf.numpy(), w["eps"], gsf, threads=THREADS)
        check_full(hc, hs, rows, cols, co, so, f"host pipeline reuse {rows}x{cols}")


def test_full_65280x7168_equals_device_call(dev):
    """The 65,280 x 7,168 workload in the benchmark's host-buffer configuration
    (2,048-row chunks, three slots), and in 8,192-row chunks, twice each: every
    result equals the device-buffer call's bytes, which the every-row oracle test
    pins."""
    w = workloads.adaln_inputs(dev)
    rows, cols = w["x"].shape
    g = gsf_tensor(150.0, dev)
    ref_c, ref_s = h3q.h3q_rmsnorm_adaln_nvfp4(w["x"], w["gamma"], w["table"], g,
                                               rows_per_frame=w["rows_per_frame"], eps=w["eps"])
    hx, hg, ht = (w[k].cpu().pin_memory() for k in ("x", "gamma", "table"))
    for chunk in (2048, 8192):
        pipe = HostPipeline(dev, max_cols=cols, chunk_rows=chunk)
        for _ in range(2):
            hc, hs = _host_outputs(rows, cols)
            pipe.rmsnorm_adaln_nvfp4(hx, hg, ht, g, hc, hs, rows_per_frame=w["rows_per_frame"],
                                     eps=w["eps"])
            torch.cuda.synchronize()
            assert torch.equal(hc, ref_c.cpu())
            assert torch.equal(hs, ref_s.cpu())


def test_rejects_bad_shapes(dev):
    pipe = HostPipeline(dev, max_cols=256, chunk_rows=128)
    x = torch.zeros((10, 512), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="max_cols"):
        pipe.rmsnorm_adaln_nvfp4(x, None, None, None, *_host_outputs(10, 512), rows_per_frame=1)
    x = torch.zeros((10, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="codes_host"):
        pipe.rmsnorm_adaln_nvfp4(x, None, None, None, *_host_outputs(11, 256), rows_per_frame=1)
    with pytest.raises(ValueError):
        HostPipeline(dev, max_cols=256, chunk_rows=100)
