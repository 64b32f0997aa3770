"""h3q -- fused NVFP4 activation producers for GB300 (sm_103a).

A thin Python binding of the C ABI in ``include/h3q.h`` (``libh3q.so``, built
in-tree by :func:`nvfp4_activation_quantize_gb300.build.build`).  The functions
carry the C names and only marshal torch CUDA tensors into the C calls; every
step of the computation runs in the library's CUDA kernels.  There is no CPU
fallback: if the library is missing or no GPU is present the calls raise.

Outputs that are not passed in are allocated here with ``torch.empty`` in the
shapes of the ABI (codes ``[rows, cols/2]`` uint8, scales
``[pad128(rows), cols/16]`` uint8 in the 128x4 swizzled layout).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "H3Q_OK", "H3Q_ERR_INVALID_ARGUMENT", "H3Q_ERR_CUDA", "H3QError", "library", "library_path",
    "padded_rows", "scale_bytes", "h3q_quantize_nvfp4", "h3q_rmsnorm_adaln_nvfp4",
    "h3q_swiglu_nvfp4", "h3q_dequantize_nvfp4", "h3q_last_error", "h3q_abi_version",
    "h3q_amax_bf16", "h3q_rmsnorm_adaln_amax", "h3q_rmsnorm_adaln_nvfp4_from_rstd", "h3q_swiglu_amax",
    "h3q_global_scale_from_amax",
    "h3q_quantize_nvfp4_dynamic", "h3q_residual_rmsnorm_adaln_nvfp4", "h3q_swiglu_packed_nvfp4",
    "h3q_qkv_epilogue", "h3q_rmsnorm_adaln_nvfp4_host", "host_workspace_bytes",
    "h3q_gemm_swiglu_nvfp4", "h3q_kernel_error_flag",
]

H3Q_OK = 0
H3Q_ERR_INVALID_ARGUMENT = 1
H3Q_ERR_CUDA = 2

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SIGNATURES = {
    "h3q_quantize_nvfp4": [_P, _I64, _I64, _I64, _P, _P, _P, _P],
    "h3q_rmsnorm_adaln_nvfp4": [_P, _I64, _P, _P, _I64, _P, _I64, ctypes.c_float, _I64, _I64,
                                _P, _P, _P, _P, _P],
    "h3q_swiglu_nvfp4": [_P, _I64, _P, _I64, _I64, _I64, _P, _P, _P, _P],
    "h3q_dequantize_nvfp4": [_P, _P, _I64, _I64, _P, _P, _P],
    "h3q_amax_bf16": [_P, _I64, _I64, _I64, _P, _P],
    "h3q_rmsnorm_adaln_amax": [_P, _I64, _P, _P, _I64, _P, _I64, ctypes.c_float, _I64, _I64, _P, _P, _P],
    "h3q_rmsnorm_adaln_nvfp4_from_rstd": [_P, _I64, _P, _P, _I64, _P, _I64, _P, _I64, _I64, _P, _P, _P, _P],
    "h3q_swiglu_amax": [_P, _I64, _P, _I64, _I64, _I64, _P, _P],
    "h3q_global_scale_from_amax": [_P, _P, _P],
    "h3q_quantize_nvfp4_dynamic": [_P, _I64, _I64, _I64, _P, _P, _P, _P],
    "h3q_swiglu_packed_nvfp4": [_P, _I64, _P, _I64, _I64, _P, _P, _P, _P],
    "h3q_residual_rmsnorm_adaln_nvfp4": [_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _P, _I64,
                                         ctypes.c_float, _I64, _I64, _P, _P, _P, _P, _P],
    "h3q_rmsnorm_adaln_nvfp4_host": [_P, _I64, _I64, _P, _P, _I64, _P, _I64, ctypes.c_float, _P, _P, _P, _P,
                                     _I64, _I64, _P],
    "h3q_qkv_epilogue": [_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _P, _P, _I64, ctypes.c_int, _I64, _I64,
                         _I64, ctypes.c_float, _P, _P, _P, _P],
    "h3q_gemm_swiglu_nvfp4": [_P, _P, _I64, _I64, _P, _P, _I64, _P, _P, _P, _P, _P, _P, _P],
    "h3q_kernel_error_flag": [_P],
}

_lock = threading.Lock()
_lib = None


class H3QError(RuntimeError):
    """A nonzero status from the library, with its message."""

    def __init__(self, fn: str, code: int, message: str):
        super().__init__(f"{fn} returned {code}: {message}")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def library():
    """The loaded ``libh3q.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with nvfp4_activation_quantize_gb300.build.build() "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(path)
            for name, args in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.h3q_last_error.argtypes = []
            lib.h3q_last_error.restype = ctypes.c_char_p
            lib.h3q_abi_version.argtypes = []
            lib.h3q_abi_version.restype = ctypes.c_int
            _lib = lib
    return _lib


def h3q_last_error() -> str:
    return library().h3q_last_error().decode()


def h3q_abi_version() -> int:
    return library().h3q_abi_version()


def padded_rows(rows: int) -> int:
    return (rows + 127) // 128 * 128


def scale_bytes(rows: int, cols: int) -> int:
    return padded_rows(rows) * (cols // 16)


def host_workspace_bytes(chunk_rows: int, cols: int, rows: int, with_frames: bool) -> int:
    """Device workspace bytes of h3q_rmsnorm_adaln_nvfp4_host (h3q_host_workspace_bytes in
    include/h3q.h): three staging slots, then the frames when they come from rows_per_frame."""
    a = lambda n: (n + 255) // 256 * 256  # noqa: E731
    slot = a(chunk_rows * cols * 2) + a(chunk_rows * cols // 2) + a(chunk_rows * cols // 16)
    return 3 * slot + (a(rows * 4) if with_frames else 0)


def _check(fn: str, rc: int) -> None:
    if rc != H3Q_OK:
        raise H3QError(fn, rc, h3q_last_error())


def _cuda_tensor(name, t, dtype, device=None):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library takes device pointers)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _rows_view(name, t, dtype, device=None):
    """A 2-D view with unit column stride; returns (tensor, rows, cols, ld)."""
    _cuda_tensor(name, t, dtype, device)
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D with contiguous rows")
    ld = t.stride(0) if t.shape[0] > 1 else t.shape[1]
    return t, t.shape[0], t.shape[1], ld


def _contiguous(name, t, dtype, shape, device):
    _cuda_tensor(name, t, dtype, device)
    if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous with shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _outputs(device, rows, cols, codes, scales):
    import torch

    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    if scales is None:
        scales = torch.empty((padded_rows(rows), cols // 16), dtype=torch.uint8, device=device)
    _contiguous("codes", codes, torch.uint8, (rows, cols // 2), device)
    _contiguous("scales", scales, torch.uint8, (padded_rows(rows), cols // 16), device)
    return codes, scales


def _gsf(global_scale, device):
    import torch

    _cuda_tensor("global_scale", global_scale, torch.float32, device)
    if global_scale.numel() != 1:
        raise ValueError("global_scale must hold one fp32 value")
    return global_scale


def _stream(stream, device) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def h3q_quantize_nvfp4(x, global_scale, codes=None, scales=None, stream=None):
    """Standalone NVFP4 quantize of bf16 x [rows, cols]; returns (codes, scales)."""
    import torch

    x, rows, cols, ld = _rows_view("x", x, torch.bfloat16)
    dev = x.device
    codes, scales = _outputs(dev, rows, cols, codes, scales)
    gsf = _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_quantize_nvfp4(x.data_ptr(), ld, rows, cols, gsf.data_ptr(),
                                          codes.data_ptr(), scales.data_ptr(), _stream(stream, dev))
    _check("h3q_quantize_nvfp4", rc)
    return codes, scales


def h3q_rmsnorm_adaln_nvfp4(x, gamma, mod_table, global_scale, *, row_frame=None,
                            rows_per_frame=None, eps=1e-6, codes=None, scales=None, row_rstd=None,
                            stream=None):
    """RMSNorm (fp32 statistics) + AdaLN modulation + NVFP4 of bf16 x [rows, cols].

    ``mod_table`` is bf16 [frames, 2, cols] ([t, 0] shift, [t, 1] scale); the frame
    of a row is ``row_frame[row]`` (int32 CUDA tensor) or ``row // rows_per_frame``.
    ``row_rstd`` (fp32 [rows], optional) receives each row's rstd.
    Returns (codes, scales).
    """
    import torch

    x, rows, cols, ld = _rows_view("x", x, torch.bfloat16)
    dev = x.device
    _contiguous("gamma", gamma, torch.bfloat16, (cols,), dev)
    _cuda_tensor("mod_table", mod_table, torch.bfloat16, dev)
    if mod_table.dim() != 3 or mod_table.shape[1:] != (2, cols) or not mod_table.is_contiguous():
        raise ValueError("mod_table must be contiguous [frames, 2, cols]")
    frames = mod_table.shape[0]
    rf_ptr = None
    if row_frame is not None:
        _contiguous("row_frame", row_frame, torch.int32, (rows,), dev)
        rf_ptr = row_frame.data_ptr()
        rows_per_frame = 0
    elif rows_per_frame is None:
        raise ValueError("give row_frame or rows_per_frame")
    rstd_ptr = None
    if row_rstd is not None:
        _contiguous("row_rstd", row_rstd, torch.float32, (rows,), dev)
        rstd_ptr = row_rstd.data_ptr()
    codes, scales = _outputs(dev, rows, cols, codes, scales)
    gsf = _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_rmsnorm_adaln_nvfp4(
            x.data_ptr(), ld, gamma.data_ptr(), mod_table.data_ptr(), frames, rf_ptr,
            int(rows_per_frame), float(eps), rows, cols, gsf.data_ptr(), codes.data_ptr(),
            scales.data_ptr(), rstd_ptr, _stream(stream, dev))
    _check("h3q_rmsnorm_adaln_nvfp4", rc)
    return codes, scales


def h3q_swiglu_nvfp4(gate, up, global_scale, codes=None, scales=None, stream=None):
    """NVFP4 of bf16(silu(gate) * up) for bf16 gate, up [rows, cols]; returns (codes, scales)."""
    import torch

    gate, rows, cols, ldg = _rows_view("gate", gate, torch.bfloat16)
    dev = gate.device
    up, rows_u, cols_u, ldu = _rows_view("up", up, torch.bfloat16, dev)
    if (rows_u, cols_u) != (rows, cols):
        raise ValueError("gate and up must have the same shape")
    codes, scales = _outputs(dev, rows, cols, codes, scales)
    gsf = _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_swiglu_nvfp4(gate.data_ptr(), ldg, up.data_ptr(), ldu, rows, cols,
                                        gsf.data_ptr(), codes.data_ptr(), scales.data_ptr(),
                                        _stream(stream, dev))
    _check("h3q_swiglu_nvfp4", rc)
    return codes, scales


def h3q_dequantize_nvfp4(codes, scales, global_scale, out=None, stream=None):
    """fp32 [rows, cols] = E2M1(code) * E4M3(scale) / gsf (checking path)."""
    import torch

    _cuda_tensor("codes", codes, torch.uint8)
    dev = codes.device
    if codes.dim() != 2 or not codes.is_contiguous():
        raise ValueError("codes must be contiguous [rows, cols/2]")
    rows, cols = codes.shape[0], codes.shape[1] * 2
    _contiguous("scales", scales, torch.uint8, (padded_rows(rows), cols // 16), dev)
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    _contiguous("out", out, torch.float32, (rows, cols), dev)
    gsf = _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_dequantize_nvfp4(codes.data_ptr(), scales.data_ptr(), rows, cols,
                                            gsf.data_ptr(), out.data_ptr(), _stream(stream, dev))
    _check("h3q_dequantize_nvfp4", rc)
    return out


# --------------------------------------------------------------------------- #
# dynamic and calibrated global scales                                          #
# --------------------------------------------------------------------------- #

def _amax_buffer(amax, device):
    import torch

    if amax is None:
        amax = torch.zeros(1, dtype=torch.float32, device=device)
    _cuda_tensor("amax", amax, torch.float32, device)
    if amax.numel() != 1:
        raise ValueError("amax must hold one fp32 value")
    return amax


def h3q_amax_bf16(x, amax=None, stream=None):
    """Fold max |x| of bf16 x [rows, cols] into the fp32 device scalar ``amax``
    (a new zero scalar when None); returns amax."""
    import torch

    x, rows, cols, ld = _rows_view("x", x, torch.bfloat16)
    amax = _amax_buffer(amax, x.device)
    with torch.cuda.device(x.device):
        rc = library().h3q_amax_bf16(x.data_ptr(), ld, rows, cols, amax.data_ptr(),
                                     _stream(stream, x.device))
    _check("h3q_amax_bf16", rc)
    return amax


def h3q_rmsnorm_adaln_amax(x, gamma, mod_table, *, row_frame=None, rows_per_frame=None, eps=1e-6,
                           amax=None, row_rstd=None, stream=None):
    """Fold max |y| of the RMSNorm + AdaLN output y (the bf16 values the producer
    quantizes, same arguments) into ``amax``; returns amax.  ``row_rstd`` (fp32
    [rows], optional) receives each row's rstd, for h3q_rmsnorm_adaln_nvfp4_from_rstd."""
    import torch

    x, rows, cols, ld = _rows_view("x", x, torch.bfloat16)
    dev = x.device
    _contiguous("gamma", gamma, torch.bfloat16, (cols,), dev)
    _cuda_tensor("mod_table", mod_table, torch.bfloat16, dev)
    if mod_table.dim() != 3 or mod_table.shape[1:] != (2, cols) or not mod_table.is_contiguous():
        raise ValueError("mod_table must be contiguous [frames, 2, cols]")
    rf_ptr = None
    if row_frame is not None:
        _contiguous("row_frame", row_frame, torch.int32, (rows,), dev)
        rf_ptr = row_frame.data_ptr()
        rows_per_frame = 0
    elif rows_per_frame is None:
        raise ValueError("give row_frame or rows_per_frame")
    amax = _amax_buffer(amax, dev)
    rstd_ptr = None
    if row_rstd is not None:
        _contiguous("row_rstd", row_rstd, torch.float32, (rows,), dev)
        rstd_ptr = row_rstd.data_ptr()
    with torch.cuda.device(dev):
        rc = library().h3q_rmsnorm_adaln_amax(
            x.data_ptr(), ld, gamma.data_ptr(), mod_table.data_ptr(), mod_table.shape[0], rf_ptr,
            int(rows_per_frame), float(eps), rows, cols, amax.data_ptr(), rstd_ptr, _stream(stream, dev))
    _check("h3q_rmsnorm_adaln_amax", rc)
    return amax


def h3q_rmsnorm_adaln_nvfp4_from_rstd(x, gamma, mod_table, row_rstd, global_scale, *, row_frame=None,
                                      rows_per_frame=None, codes=None, scales=None, stream=None):
    """The RMSNorm + AdaLN producer with each row's rstd given (fp32 [rows], e.g. the
    abs-max pass's ``row_rstd``): the statistics are not formed again.  Returns
    (codes, scales)."""
    import torch

    x, rows, cols, ld = _rows_view("x", x, torch.bfloat16)
    dev = x.device
    _contiguous("gamma", gamma, torch.bfloat16, (cols,), dev)
    _cuda_tensor("mod_table", mod_table, torch.bfloat16, dev)
    if mod_table.dim() != 3 or mod_table.shape[1:] != (2, cols) or not mod_table.is_contiguous():
        raise ValueError("mod_table must be contiguous [frames, 2, cols]")
    _contiguous("row_rstd", row_rstd, torch.float32, (rows,), dev)
    rf_ptr = None
    if row_frame is not None:
        _contiguous("row_frame", row_frame, torch.int32, (rows,), dev)
        rf_ptr = row_frame.data_ptr()
        rows_per_frame = 0
    elif rows_per_frame is None:
        raise ValueError("give row_frame or rows_per_frame")
    codes, scales = _outputs(dev, rows, cols, codes, scales)
    gsf = _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_rmsnorm_adaln_nvfp4_from_rstd(
            x.data_ptr(), ld, gamma.data_ptr(), mod_table.data_ptr(), mod_table.shape[0], rf_ptr,
            int(rows_per_frame), row_rstd.data_ptr(), rows, cols, gsf.data_ptr(), codes.data_ptr(),
            scales.data_ptr(), _stream(stream, dev))
    _check("h3q_rmsnorm_adaln_nvfp4_from_rstd", rc)
    return codes, scales


def h3q_swiglu_amax(gate, up, amax=None, stream=None):
    """Fold max |bf16(silu(gate) * up)| into ``amax``; returns amax."""
    import torch

    gate, rows, cols, ldg = _rows_view("gate", gate, torch.bfloat16)
    dev = gate.device
    up, rows_u, cols_u, ldu = _rows_view("up", up, torch.bfloat16, dev)
    if (rows_u, cols_u) != (rows, cols):
        raise ValueError("gate and up must have the same shape")
    amax = _amax_buffer(amax, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_swiglu_amax(gate.data_ptr(), ldg, up.data_ptr(), ldu, rows, cols,
                                       amax.data_ptr(), _stream(stream, dev))
    _check("h3q_swiglu_amax", rc)
    return amax


def h3q_global_scale_from_amax(amax, global_scale=None, stream=None):
    """The global scale fl(2688 / amax) computed on the device from the fp32 scalar
    ``amax`` (0 gives 1; +inf is clamped); returns the fp32 scalar written."""
    import torch

    _cuda_tensor("amax", amax, torch.float32)
    dev = amax.device
    if global_scale is None:
        global_scale = torch.empty(1, dtype=torch.float32, device=dev)
    _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_global_scale_from_amax(amax.data_ptr(), global_scale.data_ptr(),
                                                  _stream(stream, dev))
    _check("h3q_global_scale_from_amax", rc)
    return global_scale


def h3q_quantize_nvfp4_dynamic(x, global_scale=None, codes=None, scales=None, stream=None):
    """NVFP4 of bf16 x [rows, cols] under its own per-call abs-max scale, with the
    abs-max pass's scratch inside the library (no caller scratch, no allocation
    there).  Returns (codes, scales, global_scale); global_scale is the fp32 device
    scalar the call wrote.  Calls overlapping on one device race on that scratch."""
    import torch

    x, rows, cols, ld = _rows_view("x", x, torch.bfloat16)
    dev = x.device
    codes, scales = _outputs(dev, rows, cols, codes, scales)
    if global_scale is None:
        global_scale = torch.empty(1, dtype=torch.float32, device=dev)
    _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_quantize_nvfp4_dynamic(x.data_ptr(), ld, rows, cols,
                                                  global_scale.data_ptr(), codes.data_ptr(),
                                                  scales.data_ptr(), _stream(stream, dev))
    _check("h3q_quantize_nvfp4_dynamic", rc)
    return codes, scales, global_scale


def h3q_residual_rmsnorm_adaln_nvfp4(h, o, gate_table, gamma, mod_table, global_scale, *, bias=None,
                                     row_frame=None, rows_per_frame=None, eps=1e-6, codes=None,
                                     scales=None, row_rstd=None, stream=None):
    """Residual fold + RMSNorm + AdaLN -> NVFP4: h (fp32 [rows, cols], updated in place)
    += bf16(o + bias) * gate_table[frame], then the AdaLN producer on the folded h.
    ``gate_table`` bf16 [frames, cols]; ``mod_table`` bf16 [frames, 2, cols].
    Returns (codes, scales)."""
    import torch

    _cuda_tensor("h", h, torch.float32)
    dev = h.device
    if h.dim() != 2 or (h.shape[1] > 1 and h.stride(1) != 1):
        raise ValueError("h must be 2-D with contiguous rows")
    rows, cols = h.shape
    ld_h = h.stride(0) if rows > 1 else cols
    o, rows_o, cols_o, ld_o = _rows_view("o", o, torch.bfloat16, dev)
    if (rows_o, cols_o) != (rows, cols):
        raise ValueError("o must have the shape of h")
    bias_ptr = None
    if bias is not None:
        _contiguous("bias", bias, torch.bfloat16, (cols,), dev)
        bias_ptr = bias.data_ptr()
    _cuda_tensor("gate_table", gate_table, torch.bfloat16, dev)
    if gate_table.dim() != 2 or gate_table.shape[1] != cols or not gate_table.is_contiguous():
        raise ValueError("gate_table must be contiguous [frames, cols]")
    _contiguous("gamma", gamma, torch.bfloat16, (cols,), dev)
    _cuda_tensor("mod_table", mod_table, torch.bfloat16, dev)
    if (mod_table.dim() != 3 or mod_table.shape[1:] != (2, cols) or not mod_table.is_contiguous()
            or mod_table.shape[0] != gate_table.shape[0]):
        raise ValueError("mod_table must be contiguous [frames, 2, cols], frames as gate_table")
    rf_ptr = None
    if row_frame is not None:
        _contiguous("row_frame", row_frame, torch.int32, (rows,), dev)
        rf_ptr = row_frame.data_ptr()
        rows_per_frame = 0
    elif rows_per_frame is None:
        raise ValueError("give row_frame or rows_per_frame")
    rstd_ptr = None
    if row_rstd is not None:
        _contiguous("row_rstd", row_rstd, torch.float32, (rows,), dev)
        rstd_ptr = row_rstd.data_ptr()
    codes, scales = _outputs(dev, rows, cols, codes, scales)
    gsf = _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_residual_rmsnorm_adaln_nvfp4(
            h.data_ptr(), ld_h, o.data_ptr(), ld_o, bias_ptr, gate_table.data_ptr(), gamma.data_ptr(),
            mod_table.data_ptr(), mod_table.shape[0], rf_ptr, int(rows_per_frame), float(eps), rows,
            cols, gsf.data_ptr(), codes.data_ptr(), scales.data_ptr(), rstd_ptr, _stream(stream, dev))
    _check("h3q_residual_rmsnorm_adaln_nvfp4", rc)
    return codes, scales


def h3q_swiglu_packed_nvfp4(o, global_scale, bias=None, codes=None, scales=None, stream=None):
    """SwiGLU of the value-first packed projection o [rows, 2F] (value, then gate)
    with its bias [2F] (or None) added and rounded to bf16 first; returns (codes, scales)
    of the [rows, F] output."""
    import torch

    o, rows, two_f, ld = _rows_view("o", o, torch.bfloat16)
    dev = o.device
    if two_f % 2:
        raise ValueError("o must have an even number of columns")
    f = two_f // 2
    bias_ptr = None
    if bias is not None:
        _contiguous("bias", bias, torch.bfloat16, (two_f,), dev)
        bias_ptr = bias.data_ptr()
    codes, scales = _outputs(dev, rows, f, codes, scales)
    gsf = _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_swiglu_packed_nvfp4(o.data_ptr(), ld, bias_ptr, rows, f, gsf.data_ptr(),
                                               codes.data_ptr(), scales.data_ptr(), _stream(stream, dev))
    _check("h3q_swiglu_packed_nvfp4", rc)
    return codes, scales


def h3q_qkv_epilogue(q, k, v, biases, cos, sin, heads, eps, outs=None, interleaved=False, stream=None):
    """QKV epilogue of projected q, k, v [rows, heads * HD] bf16 (bias not yet added):
    returns (q_out, k_out, v_out), each bf16 [rows, heads, HD], with q and k biased,
    RMS-normed per head and rotated (RoPE on each head's first ROT values, cos and
    sin bf16 [rows, ROT], None for ROT = 0: rotate-half pairs (i, i + ROT/2), or
    pairs (2j, 2j + 1) with ``interleaved``) and v biased."""
    import torch

    q, rows, d, ld_q = _rows_view("q", q, torch.bfloat16)
    dev = q.device
    k, rows_k, d_k, ld_k = _rows_view("k", k, torch.bfloat16, dev)
    v, rows_v, d_v, ld_v = _rows_view("v", v, torch.bfloat16, dev)
    if (rows_k, d_k) != (rows, d) or (rows_v, d_v) != (rows, d):
        raise ValueError("q, k and v must have the same shape")
    if heads < 1 or d % heads:
        raise ValueError("the columns of q must split into heads")
    hd = d // heads
    b = [_contiguous(n, t, torch.bfloat16, (d,), dev) for n, t in zip(("bias_q", "bias_k", "bias_v"), biases)]
    rot, cos_ptr, sin_ptr = 0, None, None
    if cos is not None or sin is not None:
        rot = cos.shape[-1] if cos.dim() == 2 else -1
        _contiguous("cos", cos, torch.bfloat16, (rows, rot), dev)
        _contiguous("sin", sin, torch.bfloat16, (rows, rot), dev)
        cos_ptr, sin_ptr = cos.data_ptr(), sin.data_ptr()
    if outs is None:
        outs = [torch.empty((rows, heads, hd), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    outs = [_contiguous(n, t, torch.bfloat16, (rows, heads, hd), dev)
            for n, t in zip(("q_out", "k_out", "v_out"), outs)]
    with torch.cuda.device(dev):
        rc = library().h3q_qkv_epilogue(q.data_ptr(), ld_q, k.data_ptr(), ld_k, v.data_ptr(), ld_v,
                                        b[0].data_ptr(), b[1].data_ptr(), b[2].data_ptr(), cos_ptr,
                                        sin_ptr, rot, int(bool(interleaved)), rows, heads, hd, float(eps),
                                        outs[0].data_ptr(),
                                        outs[1].data_ptr(), outs[2].data_ptr(), _stream(stream, dev))
    _check("h3q_qkv_epilogue", rc)
    return outs[0], outs[1], outs[2]


def h3q_rmsnorm_adaln_nvfp4_host(x_host, gamma, mod_table, global_scale, codes_host, scales_host, workspace, *,
                                 row_frame=None, rows_per_frame=None, eps=1e-6, chunk_rows=8192, stream=None):
    """RMSNorm + AdaLN -> NVFP4 on host buffers: x_host (contiguous bf16 [rows, cols] in
    host memory, pinned for the copies to overlap) into host codes [rows, cols/2] and
    scales [pad128(rows), cols/16] (uint8, contiguous), the copies inside the library
    call, pipelined over `chunk_rows`-row chunks.  gamma, mod_table, global_scale and
    row_frame are CUDA tensors; `workspace` is a CUDA uint8 tensor of at least
    host_workspace_bytes(chunk_rows, cols, rows, row_frame is None) bytes.  The host
    outputs may be read once `stream` (default: the current stream) is synchronised."""
    import torch

    if not isinstance(x_host, torch.Tensor) or x_host.is_cuda or x_host.dtype != torch.bfloat16:
        raise ValueError("x_host must be a host bf16 tensor")
    if x_host.dim() != 2 or not x_host.is_contiguous():
        raise ValueError("x_host must be contiguous [rows, cols]")
    rows, cols = x_host.shape
    _cuda_tensor("workspace", workspace, torch.uint8)
    dev = workspace.device
    for name, t, shape in (("codes_host", codes_host, (rows, cols // 2)),
                           ("scales_host", scales_host, (padded_rows(rows), cols // 16))):
        if (not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.uint8 or tuple(t.shape) != shape
                or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous host uint8 tensor {shape}")
    _contiguous("gamma", gamma, torch.bfloat16, (cols,), dev)
    _cuda_tensor("mod_table", mod_table, torch.bfloat16, dev)
    if mod_table.dim() != 3 or mod_table.shape[1:] != (2, cols) or not mod_table.is_contiguous():
        raise ValueError("mod_table must be contiguous [frames, 2, cols]")
    rf_ptr = None
    if row_frame is not None:
        _contiguous("row_frame", row_frame, torch.int32, (rows,), dev)
        rf_ptr = row_frame.data_ptr()
        rows_per_frame = 0
    elif rows_per_frame is None:
        raise ValueError("give row_frame or rows_per_frame")
    gsf = _gsf(global_scale, dev)
    with torch.cuda.device(dev):
        rc = library().h3q_rmsnorm_adaln_nvfp4_host(
            x_host.data_ptr(), rows, cols, gamma.data_ptr(), mod_table.data_ptr(), mod_table.shape[0], rf_ptr,
            int(rows_per_frame), float(eps), gsf.data_ptr(), codes_host.data_ptr(), scales_host.data_ptr(),
            workspace.data_ptr(), workspace.numel(), int(chunk_rows), _stream(stream, dev))
    _check("h3q_rmsnorm_adaln_nvfp4_host", rc)
    return codes_host, scales_host


def h3q_gemm_swiglu_nvfp4(a_codes, a_scales, b_codes, b_scales, alpha, global_scale, codes=None, scales=None,
                          y=None, acc=None, stream=None):
    """The FFN-up projection as a block-scaled NVFP4 GEMM with the SwiGLU + NVFP4 epilogue.

    ``a_codes`` uint8 [m, k/2] and ``a_scales`` uint8 [pad128(m), k/16] (128x4 layout) are
    the NVFP4 activation; ``b_codes`` [n, k/2] and ``b_scales`` [n, k/16] the NVFP4 weight,
    row 2j the value and row 2j+1 the gate of output j.  ``alpha`` and ``global_scale`` are
    device fp32 scalars.  Outputs: codes [m, n/4], scales [pad128(m), n/32]; optional ``y``
    (bf16 [m, n/2]) and ``acc`` (fp32 [m, n], the accumulator before alpha).
    Returns (codes, scales).
    """
    import torch

    _cuda_tensor("a_codes", a_codes, torch.uint8)
    dev = a_codes.device
    if a_codes.dim() != 2 or not a_codes.is_contiguous():
        raise ValueError("a_codes must be contiguous [m, k/2]")
    m, k = a_codes.shape[0], 2 * a_codes.shape[1]
    _cuda_tensor("b_codes", b_codes, torch.uint8, dev)
    if b_codes.dim() != 2 or b_codes.shape[1] != k // 2 or not b_codes.is_contiguous():
        raise ValueError("b_codes must be contiguous [n, k/2]")
    n = b_codes.shape[0]
    f = n // 2
    for name, t, rows in (("a_scales", a_scales, padded_rows(m)), ("b_scales", b_scales, padded_rows(n))):
        _cuda_tensor(name, t, torch.uint8, dev)
        if not t.is_contiguous() or t.numel() != rows * (k // 16):
            raise ValueError(f"{name} must be contiguous with {rows} x {k // 16} bytes")
    _gsf(alpha, dev)
    gsf = _gsf(global_scale, dev)
    codes, scales = _outputs(dev, m, f, codes, scales)
    y_ptr = acc_ptr = None
    if y is not None:
        _contiguous("y", y, torch.bfloat16, (m, f), dev)
        y_ptr = y.data_ptr()
    if acc is not None:
        _contiguous("acc", acc, torch.float32, (m, n), dev)
        acc_ptr = acc.data_ptr()
    with torch.cuda.device(dev):
        rc = library().h3q_gemm_swiglu_nvfp4(
            a_codes.data_ptr(), a_scales.data_ptr(), m, k, b_codes.data_ptr(), b_scales.data_ptr(), n,
            alpha.data_ptr(), gsf.data_ptr(), codes.data_ptr(), scales.data_ptr(), y_ptr, acc_ptr,
            _stream(stream, dev))
    _check("h3q_gemm_swiglu_nvfp4", rc)
    return codes, scales


def h3q_kernel_error_flag() -> int:
    """Reads and clears the flag a kernel sets when one of its bounded waits ran out
    (synchronises the device); 0 when none did."""
    flag = ctypes.c_int(0)
    _check("h3q_kernel_error_flag", library().h3q_kernel_error_flag(ctypes.byref(flag)))
    return flag.value
