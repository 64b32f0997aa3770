"""h3q_quantize_nvfp4_dynamic: the dynamic quantize whose abs-max pass keeps its
partial maxima in a device array inside the library instead of caller scratch.

On the GPU it must write what the existing entry points write for the same
input -- h3q_amax_bf16 into a zeroed scalar, h3q_global_scale_from_amax, then
h3q_quantize_nvfp4 -- on two calls in a row, the second on a smaller input with
a smaller abs-max, so that partial maxima left behind by the first call would
show.  On the host, its argument checks run before any CUDA call.

(The file is named to be collected last: the scratch array is shared by every
call in the process, and the test must pass after all the others too.)
"""
import numpy as np
import pytest
import torch

import nvfp4_activation_quantize_gb300 as h3q
import oracle
import workloads
from nvfp4_activation_quantize_gb300 import build as libbuild
from parity import bits


def _f32(t: torch.Tensor) -> int:
    return int(np.float32(float(t.item())).view(np.uint32))


@pytest.mark.gpu
def test_matches_the_existing_entry_points_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    big = workloads.quantize_inputs(dev, rows=3000, cols=7168, seed=41)            # abs-max 1000
    small = (workloads.attention_output(dev, tokens=10, seed=42) * 0.5).contiguous()  # far smaller
    gsf = torch.empty(1, dtype=torch.float32, device=dev)
    for x in (big, small):
        rows, cols = x.shape
        codes = torch.full((rows, cols // 2), 0xAB, dtype=torch.uint8, device=dev)
        scales = torch.full((h3q.padded_rows(rows), cols // 16), 0xAB, dtype=torch.uint8, device=dev)
        h3q.h3q_quantize_nvfp4_dynamic(x, gsf, codes, scales)

        amax = torch.zeros(1, dtype=torch.float32, device=dev)
        h3q.h3q_amax_bf16(x, amax)
        ref_gsf = h3q.h3q_global_scale_from_amax(amax)
        ref_codes, ref_scales = h3q.h3q_quantize_nvfp4(x, ref_gsf)
        torch.cuda.synchronize()

        assert _f32(gsf) == _f32(ref_gsf), f"global scale {gsf.item()} != {ref_gsf.item()}"
        assert _f32(gsf) == int(np.float32(oracle.global_scale_from_amax(oracle.amax_bf16(bits(x))))
                                .view(np.uint32))
        assert torch.equal(codes, ref_codes), f"codes differ for {rows} x {cols}"
        assert torch.equal(scales, ref_scales), f"scales differ for {rows} x {cols}"


@pytest.mark.gpu
def test_a_call_leaves_device_memory_as_it_found_it():
    """After a first call on the device, further calls change no free-memory count:
    the partial maxima go to the library's own array, and nothing is allocated."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    x = workloads.attention_output(dev, tokens=2048, seed=43)
    rows, cols = x.shape
    gsf = torch.empty(1, dtype=torch.float32, device=dev)
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((h3q.padded_rows(rows), cols // 16), dtype=torch.uint8, device=dev)
    lib = h3q.library()
    stream = torch.cuda.current_stream(dev).cuda_stream

    def call():
        rc = lib.h3q_quantize_nvfp4_dynamic(x.data_ptr(), cols, rows, cols, gsf.data_ptr(),
                                            codes.data_ptr(), scales.data_ptr(), stream)
        assert rc == h3q.H3Q_OK, h3q.h3q_last_error()

    call()
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info(dev)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info(dev)
    assert free_after == free_before, f"free device memory moved by {free_before - free_after} bytes"


def test_host_checks_run_before_any_cuda_call():
    libbuild.build()
    lib = h3q.library()
    f = lib.h3q_quantize_nvfp4_dynamic
    # (x, ld, rows, cols, global_scale, codes, scales, stream)
    assert f(None, 256, 4, 256, 0x400000, 0x500000, 0x600000, None) == h3q.H3Q_ERR_INVALID_ARGUMENT
    assert f(0x100010, 256, 4, 256, 0x400000, 0x500000, 0x600000, None) == 1  # x not 32-byte aligned
    assert f(0x100000, 256, 4, 100, 0x400000, 0x500000, 0x600000, None) == 1  # cols % 64
    assert f(0x100000, 256, 4, 256, None, 0x500000, 0x600000, None) == 1      # no global scale
    assert f(0x100000, 256, 4, 256, 0x500004, 0x500000, 0x600000, None) == 1  # scale inside codes
    assert "overlap" in h3q.h3q_last_error()
    assert f(None, 256, 0, 256, None, None, None, None) == h3q.H3Q_OK          # no rows: no-op
    if not torch.cuda.is_available():
        assert f(0x100000, 256, 4, 256, 0x400000, 0x500000, 0x600000, None) == h3q.H3Q_ERR_CUDA
