"""The C ABI without a GPU: libh3q.so builds and loads, exports every function
include/h3q.h declares, and rejects invalid arguments on the host before any
CUDA call.  (Compute calls need a GPU; they live in the -m gpu tests.)"""
import ctypes
import os
import re

import pytest

import nvfp4_activation_quantize_gb300 as h3q
from nvfp4_activation_quantize_gb300 import build as libbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "h3q.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return h3q.library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(h3q_\w+)\s*\(", text, flags=re.M)
    inline = set(re.findall(r"static inline [^(]*?(h3q_\w+)\s*\(", text))
    return sorted(set(names) - inline)


def test_header_declares_the_four_calls():
    names = _declared_functions()
    for fn in ("h3q_quantize_nvfp4", "h3q_rmsnorm_adaln_nvfp4", "h3q_swiglu_nvfp4",
               "h3q_dequantize_nvfp4", "h3q_last_error", "h3q_abi_version"):
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    for fn in _declared_functions():
        assert hasattr(lib, fn), f"{fn} is declared in h3q.h but not exported"
    assert lib.h3q_abi_version() == 4


def _q(lib, x=0x10000, ld=256, rows=4, cols=256, gsf=0x20000, codes=0x30000, scales=0x40000):
    return lib.h3q_quantize_nvfp4(x, ld, rows, cols, gsf, codes, scales, None)


def test_quantize_rejects_bad_arguments_on_the_host(lib):
    # none of these pointers is dereferenced: validation fails first
    assert _q(lib, cols=100) == h3q.H3Q_ERR_INVALID_ARGUMENT
    assert "multiple of 64" in h3q.h3q_last_error()
    assert _q(lib, cols=0) == 1
    assert _q(lib, rows=-1) == 1
    assert _q(lib, x=None) == 1
    assert _q(lib, x=0x10010) == 1 and "32-byte" in h3q.h3q_last_error()
    assert _q(lib, ld=200) == 1
    assert _q(lib, ld=264) == 1
    assert _q(lib, codes=None) == 1
    assert _q(lib, scales=0x40004) == 1
    assert _q(lib, gsf=None) == 1
    assert _q(lib, codes=0x10000 + 64) == 1 and "overlap" in h3q.h3q_last_error()
    assert _q(lib, cols=1 << 25, ld=1 << 25) == 1


def test_zero_rows_is_a_noop_without_a_gpu(lib):
    assert _q(lib, rows=0, x=None, codes=None, scales=None, gsf=None) == h3q.H3Q_OK
    assert h3q.h3q_last_error() == ""


def test_adaln_rejects_bad_arguments_on_the_host(lib):
    def call(**kw):
        a = dict(x=0x100000, ld=256, gamma=0x200000, table=0x300000, frames=4, row_frame=None,
                 rpf=16, eps=1e-6, rows=64, cols=256, gsf=0x400000, codes=0x500000,
                 scales=0x600000, rstd=None)
        a.update(kw)
        return lib.h3q_rmsnorm_adaln_nvfp4(a["x"], a["ld"], a["gamma"], a["table"], a["frames"],
                                           a["row_frame"], a["rpf"], a["eps"], a["rows"], a["cols"],
                                           a["gsf"], a["codes"], a["scales"], a["rstd"], None)

    assert call(rpf=0) == 1
    assert call(rpf=15) == 1 and "modulation table" in h3q.h3q_last_error()
    assert call(frames=0) == 1
    assert call(eps=float("nan")) == 1
    assert call(eps=-1.0) == 1
    assert call(gamma=None) == 1
    assert call(table=0x300010) == 1
    assert call(row_frame=0x700002) == 1
    assert call(rstd=0x600000 + 8) == 1  # rstd inside the scales buffer
    assert call(codes=0x300000) == 1     # codes over the table


def test_swiglu_and_dequantize_reject_bad_arguments_on_the_host(lib):
    assert lib.h3q_swiglu_nvfp4(0x100000, 256, None, 256, 8, 256, 0x400000, 0x500000, 0x600000,
                                None) == 1
    assert lib.h3q_swiglu_nvfp4(0x100000, 256, 0x200000, 8, 8, 256, 0x400000, 0x500000,
                                0x600000, None) == 1
    assert lib.h3q_dequantize_nvfp4(0x100000, 0x200000, 8, 256, 0x300000, 0x400010, None) == 1
    assert lib.h3q_dequantize_nvfp4(0x100000, 0x200000, 8, 96, 0x300000, 0x400000, None) == 1


def test_valid_call_without_a_gpu_reports_a_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = _q(lib)
    assert rc == h3q.H3Q_ERR_CUDA, h3q.h3q_last_error()
    assert "CUDA error" in h3q.h3q_last_error()


def test_python_binding_refuses_host_tensors():
    import torch

    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        h3q.h3q_quantize_nvfp4(x, torch.ones(1))


def test_dynamic_scale_calls_reject_bad_arguments_on_the_host(lib):
    # h3q_amax_bf16(x, ld, rows, cols, amax, stream)
    assert lib.h3q_amax_bf16(0x100000, 256, 4, 256, None, None) == 1
    assert "amax" in h3q.h3q_last_error()
    assert lib.h3q_amax_bf16(0x100000, 256, 4, 256, 0x200002, None) == 1
    assert lib.h3q_amax_bf16(0x100000, 256, 4, 256, 0x100010, None) == 1  # inside x
    assert lib.h3q_amax_bf16(0x100000, 256, 4, 100, 0x200000, None) == 1
    assert lib.h3q_amax_bf16(None, 256, 0, 256, None, None) == h3q.H3Q_OK  # no rows: no-op
    # h3q_rmsnorm_adaln_amax(x, ld, gamma, table, frames, row_frame, rpf, eps, rows, cols, amax,
    #                        row_rstd, stream)
    args = [0x100000, 256, 0x200000, 0x300000, 4, None, 16, 1e-6, 64, 256, 0x400000, None, None]
    bad = list(args); bad[6] = 15
    assert lib.h3q_rmsnorm_adaln_amax(*bad) == 1 and "modulation table" in h3q.h3q_last_error()
    bad = list(args); bad[10] = None
    assert lib.h3q_rmsnorm_adaln_amax(*bad) == 1
    bad = list(args); bad[10] = 0x300004  # inside the table
    assert lib.h3q_rmsnorm_adaln_amax(*bad) == 1 and "overlaps" in h3q.h3q_last_error()
    bad = list(args); bad[7] = -1.0
    assert lib.h3q_rmsnorm_adaln_amax(*bad) == 1
    bad = list(args); bad[11] = 0x500002  # row_rstd misaligned
    assert lib.h3q_rmsnorm_adaln_amax(*bad) == 1 and "row_rstd" in h3q.h3q_last_error()
    bad = list(args); bad[11] = 0x400000  # row_rstd on amax
    assert lib.h3q_rmsnorm_adaln_amax(*bad) == 1 and "overlaps" in h3q.h3q_last_error()
    bad = list(args); bad[11] = 0x100100  # row_rstd inside x
    assert lib.h3q_rmsnorm_adaln_amax(*bad) == 1 and "overlaps" in h3q.h3q_last_error()
    # h3q_swiglu_amax(gate, ldg, up, ldu, rows, cols, amax, stream)
    assert lib.h3q_swiglu_amax(0x100000, 256, None, 256, 8, 256, 0x400000, None) == 1
    assert lib.h3q_swiglu_amax(0x100000, 256, 0x200000, 256, 8, 256, 0x200100, None) == 1
    # h3q_global_scale_from_amax(amax, gsf, stream)
    assert lib.h3q_global_scale_from_amax(None, 0x100000, None) == 1
    assert lib.h3q_global_scale_from_amax(0x100000, None, None) == 1
    assert lib.h3q_global_scale_from_amax(0x100001, 0x100000, None) == 1


def test_dynamic_scale_call_without_a_gpu_reports_a_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.h3q_amax_bf16(0x100000, 256, 4, 256, 0x200000, None) == h3q.H3Q_ERR_CUDA
    assert lib.h3q_global_scale_from_amax(0x100000, 0x200000, None) == h3q.H3Q_ERR_CUDA


def test_residual_fold_rejects_bad_arguments_on_the_host(lib):
    # (h, ld_h, o, ld_o, bias, gate, gamma, table, frames, row_frame, rpf, eps, rows, cols,
    #  gsf, codes, scales, row_rstd, stream)
    good = [0x1000000, 256, 0x2000000, 256, None, 0x3000000, 0x3100000, 0x3200000, 4, None, 16,
            1e-6, 64, 256, 0x4000000, 0x5000000, 0x6000000, None, None]
    f = lib.h3q_residual_rmsnorm_adaln_nvfp4

    def call(**kw):
        a = list(good)
        names = ["h", "ld_h", "o", "ld_o", "bias", "gate", "gamma", "table", "frames", "row_frame",
                 "rpf", "eps", "rows", "cols", "gsf", "codes", "scales", "rstd", "stream"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(cols=16384, ld_h=16384, ld_o=16384) == 1 and "8,192" in h3q.h3q_last_error()
    assert call(h=None) == 1
    assert call(h=0x1000010) == 1                       # h not 32-byte aligned
    assert call(ld_h=260) == 1                          # ld_h not a multiple of 8
    assert call(gate=None) == 1
    assert call(bias=0x3000010) == 1                    # bias not 32-byte aligned
    assert call(rpf=15) == 1 and "modulation table" in h3q.h3q_last_error()
    assert call(o=0x1000000 + 512) == 1 and "overlap" in h3q.h3q_last_error()   # o inside h
    assert call(codes=0x1000000 + 4096) == 1                                     # codes inside h
    assert call(rows=0, h=None, o=None) == h3q.H3Q_OK


def test_swiglu_packed_rejects_bad_arguments_on_the_host(lib):
    # (o, ld_o, bias, rows, f, gsf, codes, scales, stream)
    f = lib.h3q_swiglu_packed_nvfp4
    assert f(0x1000000, 512, None, 8, 256, 0x4000000, 0x5000000, 0x6000000, None) in (0, 2)
    assert f(0x1000000, 500, None, 8, 256, 0x4000000, 0x5000000, 0x6000000, None) == 1  # ld < 2F
    assert f(0x1000000, 512, 0x2000010, 8, 256, 0x4000000, 0x5000000, 0x6000000, None) == 1
    assert f(0x1000000, 512, None, 8, 100, 0x4000000, 0x5000000, 0x6000000, None) == 1   # F % 64
    assert f(0x1000000, 512, None, 8, 256, 0x4000000, 0x1000100, 0x6000000, None) == 1   # codes in o
    assert f(None, 512, None, 0, 256, None, None, None, None) == h3q.H3Q_OK


def test_qkv_epilogue_rejects_bad_arguments_on_the_host(lib):
    # (q, ld_q, k, ld_k, v, ld_v, bias_q, bias_k, bias_v, cos, sin, rot, interleaved, rows, heads,
    #  head_dim, eps, q_out, k_out, v_out, stream): 8 rows of 2 heads of 128
    names = ["q", "ld_q", "k", "ld_k", "v", "ld_v", "bq", "bk", "bv", "cos", "sin", "rot", "ilv", "rows",
             "heads", "hd", "eps", "qo", "ko", "vo", "stream"]
    good = [0x1000000, 256, 0x1100000, 256, 0x1200000, 256, 0x2000000, 0x2100000, 0x2200000,
            0x3000000, 0x3100000, 64, 0, 8, 2, 128, 1e-6, 0x4000000, 0x4100000, 0x4200000, None]
    f = lib.h3q_qkv_epilogue

    def call(**kw):
        a = list(good)
        for name, value in kw.items():
            a[names.index(name)] = value
        return f(*a)

    assert call() in (0, 2)
    assert call(hd=96, ld_q=192, ld_k=192, ld_v=192) == 1 and "head_dim" in h3q.h3q_last_error()
    assert call(rot=24) == 1 and "rot" in h3q.h3q_last_error()
    assert call(rot=144) == 1                                          # rot > head_dim
    assert call(heads=0) == 1
    assert call(eps=float("nan")) == 1
    assert call(ld_k=200) == 1                                          # ld < H * HD
    assert call(k=0x1100010) == 1                                       # k not 32-byte aligned
    assert call(bv=None) == 1
    assert call(cos=None) == 1 and "cos" in h3q.h3q_last_error()
    assert call(rot=0, cos=None, sin=None) in (0, 2)                    # no rotation, no tables
    assert call(sin=0x3100008) == 1                                     # sin not 16-byte aligned
    assert call(vo=0x1000000 + 256) == 1 and "overlap" in h3q.h3q_last_error()  # v_out inside q
    assert call(ko=0x4000000 + 4096 - 16) == 1 and "overlap" in h3q.h3q_last_error()  # k_out on q_out
    assert call(qo=0x3000000) == 1                                      # q_out on cos
    assert call(ilv=1) in (0, 2) and call(ilv=2) == 1 and "interleaved" in h3q.h3q_last_error()
    assert call(rows=0, q=None, k=None, v=None) == h3q.H3Q_OK


def test_python_binding_of_the_qkv_epilogue_refuses_host_tensors():
    import torch

    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    b = torch.zeros(256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        h3q.h3q_qkv_epilogue(x, x, x, (b, b, b), None, None, 2, 1e-6)


def test_host_call_rejects_bad_arguments_on_the_host(lib):
    # (x_host, rows, cols, gamma, table, frames, row_frame, rpf, eps, gsf, codes_host, scales_host,
    #  workspace, workspace_bytes, chunk_rows, stream)
    names = ["x", "rows", "cols", "gamma", "table", "frames", "rf", "rpf", "eps", "gsf", "codes", "scales",
             "ws", "wsb", "chunk", "stream"]
    need = h3q.host_workspace_bytes(256, 512, 1000, True)
    good = [0x7000000, 1000, 512, 0x1000000, 0x1100000, 4, None, 250, 1e-6, 0x1200000, 0x7100000,
            0x7200000, 0x2000000, need, 256, None]
    f = lib.h3q_rmsnorm_adaln_nvfp4_host

    def call(**kw):
        a = list(good)
        for name, value in kw.items():
            a[names.index(name)] = value
        return f(*a)

    assert call() in (0, 2)
    assert call(chunk=200) == 1 and "chunk_rows" in h3q.h3q_last_error()
    assert call(wsb=need - 1) == 1 and "workspace" in h3q.h3q_last_error()
    assert call(ws=0x2000010) == 1                                    # workspace not 256-byte aligned
    assert call(x=None) == 1
    assert call(rpf=200) == 1 and "modulation table" in h3q.h3q_last_error()
    assert call(codes=0x7000000 + 4096) == 1 and "overlap" in h3q.h3q_last_error()  # codes inside x
    assert call(ws=0x1000000 - 512) == 1 and "workspace" in h3q.h3q_last_error()      # workspace on gamma
    assert call(rows=0, x=None) == h3q.H3Q_OK


def test_gemm_swiglu_host_checks_run_before_any_cuda_call():
    """h3q_gemm_swiglu_nvfp4 rejects shapes, alignment and overlaps on the host."""
    lib = h3q.library()
    f = lib.h3q_gemm_swiglu_nvfp4
    A, AS, B, BS, AL, G, C, S = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x500010, 0x600000, 0x700000
    # (a, a_scales, m, k, b, b_scales, n, alpha, gsf, codes, scales, y, acc, stream)
    assert f(A, AS, 4, 128, B, BS, 256, AL, G, C, S, None, None, None) == 1       # k % 256
    assert f(A, AS, 4, 256, B, BS, 200, AL, G, C, S, None, None, None) == 1       # n % 256
    assert f(A, AS, -1, 256, B, BS, 256, AL, G, C, S, None, None, None) == 1      # m < 0
    assert f(A + 8, AS, 4, 256, B, BS, 256, AL, G, C, S, None, None, None) == 1   # a not 16-byte aligned
    assert f(A, AS, 4, 256, B, BS, 256, None, G, C, S, None, None, None) == 1     # no alpha
    assert f(A, AS, 4, 256, B, BS, 256, AL, G, C, S, C + 16, None, None) == 1     # y inside codes
    assert "overlap" in h3q.h3q_last_error()
    assert f(A, AS, 4, 256, B, BS, 256, AL, G, A, S, None, None, None) == 1       # codes over a
    assert f(None, None, 0, 256, None, None, 256, None, None, None, None, None, None, None) == 0  # m = 0


def test_from_rstd_producer_rejects_bad_arguments_on_the_host(lib):
    # h3q_rmsnorm_adaln_nvfp4_from_rstd(x, ld, gamma, table, frames, row_frame, rpf, row_rstd, rows, cols,
    #                                   gsf, codes, scales, stream)
    args = [0x100000, 256, 0x200000, 0x300000, 4, None, 16, 0x500000, 64, 256, 0x600000, 0x700000,
            0x800000, None]
    bad = list(args); bad[7] = None
    assert lib.h3q_rmsnorm_adaln_nvfp4_from_rstd(*bad) == 1 and "row_rstd" in h3q.h3q_last_error()
    bad = list(args); bad[7] = 0x500002
    assert lib.h3q_rmsnorm_adaln_nvfp4_from_rstd(*bad) == 1 and "aligned" in h3q.h3q_last_error()
    bad = list(args); bad[7] = 0x700010  # row_rstd inside the codes
    assert lib.h3q_rmsnorm_adaln_nvfp4_from_rstd(*bad) == 1 and "overlaps" in h3q.h3q_last_error()
    bad = list(args); bad[6] = 15
    assert lib.h3q_rmsnorm_adaln_nvfp4_from_rstd(*bad) == 1 and "modulation table" in h3q.h3q_last_error()
    bad = list(args); bad[9] = 100
    assert lib.h3q_rmsnorm_adaln_nvfp4_from_rstd(*bad) == 1
    bad = list(args); bad[0] = None
    assert lib.h3q_rmsnorm_adaln_nvfp4_from_rstd(*bad) == 1
    bad = list(args); bad[8] = 0
    assert lib.h3q_rmsnorm_adaln_nvfp4_from_rstd(*bad) == h3q.H3Q_OK  # no rows: no-op
