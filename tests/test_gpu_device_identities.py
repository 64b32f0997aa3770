"""The kernels' division-free routines against CUDA's correctly rounded operations,
exhaustively on the GPU: the Markstein reciprocal used for the SiLU sigmoid over
every binary32 in [1, 2^126), the once-corrected fl(a/6) of the block scale
over every bf16 value, and the one-instruction bf16 sum (the bias adds and the
RoPE sum) against the binary32 sum rounded to bf16 over every pair of bf16
values, and the hardware bf16, E2M1 and E4M3 conversions the kernels use against
integer formulations of the formats over every binary32 pattern
(tests/device/identities.cu, compiled here with the library's own flags)."""
import os
import subprocess

import pytest
import torch

from nvfp4_activation_quantize_gb300 import build as libbuild

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_division_free_routines_match_cuda(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = str(tmp_path / "identities")
    flags = [f for f in libbuild.NVCC_FLAGS if f not in ("-Xcompiler", "-fPIC", "-Xptxas", "-v")]
    subprocess.run([libbuild._nvcc(), *flags, os.path.join(HERE, "device", "identities.cu"), "-o", exe],
                   check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "rcp_rn_ge1 mismatches 0" in res.stdout and "amax_over_six mismatches 0" in res.stdout
    assert "add_bf16x2 mismatches 0 of 4294967296" in res.stdout
    assert "e2m1 mismatches 0; bf16 mismatches 0; e4m3 mismatches 0" in res.stdout
