"""CPU oracle for the fused NVFP4 activation producers (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  The library never does: the CUDA path fails loudly when its
extension is missing and has no CPU fallback.

The arithmetic lives in ``h3q_oracle.c`` (plain C, binary32, one rounding per
operation, built with ``-ffp-contract=off``).  This module compiles it with
gcc on first use and wraps it for numpy arrays.  bf16 tensors travel as
``uint16`` arrays of their bit patterns.

Functions here mirror the four library calls on host arrays:

* :func:`quantize_rows`  -- standalone NVFP4 quantize (attention output)
* :func:`adaln_rows`     -- RMSNorm (fp32 statistics) + AdaLN modulation -> NVFP4
* :func:`swiglu_rows`    -- silu(gate) * up -> NVFP4
* :func:`dequantize_rows`-- codes + block scales -> fp32
* :func:`nvfp4_gemm`, :func:`swiglu_epilogue_rows` -- the block-scaled NVFP4 GEMM
  (exact sum, rounded once) and its SwiGLU + NVFP4 epilogue

plus :func:`swizzle_scales` (logical [rows, cols/16] scales to the 128x4
layout with zeroed padding rows) and the element-wise conversions the pin
tests check.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "h3q_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (host compiler)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if force or not fresh:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float

_SIGNATURES = {
    "orc_bf16_bits": ([_F], ctypes.c_uint16),
    "orc_bf16_value": ([ctypes.c_uint16], _F),
    "orc_e4m3_value": ([ctypes.c_uint8], _F),
    "orc_e4m3_encode": ([_F], ctypes.c_uint8),
    "orc_e2m1_value": ([ctypes.c_uint8], _F),
    "orc_e2m1_encode": ([_F], ctypes.c_uint8),
    "orc_exp": ([_F], _F),
    "orc_exp_constants": ([_P], None),
    "orc_swiglu_value": ([_F, _F], _F),
    "orc_quantize_block": ([_P, _F, _P, _P], None),
    "orc_global_scale": ([_F], _F),
    "orc_amax_bf16": ([_P, _I64], _F),
    "orc_row_rstd_f32": ([_P, _I64, _F], _F),
    "orc_sumsq_bf16": ([_P, _I64, ctypes.c_int], _F),
    "orc_sumsq_f32": ([_P, _I64, ctypes.c_int], _F),
    "orc_head_rstd": ([_P, _I64, _F], _F),
    "orc_nvfp4_gemm_rows": ([_P, _P, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _P], None),
    "orc_swiglu_epilogue_rows": ([_P, _I64, _I64, _F, _F, _P, _P, _P, _P], None),
    "orc_qkv_epilogue_rows": ([_P, _I64, _P, _I64, _I64, _I64, ctypes.c_int, _P, _P, _I64, ctypes.c_int, _F,
                               _P], None),
    "orc_swiglu_packed_rows": ([_P, _I64, _P, _I64, _I64, _F, _P, _P, _P, _P], None),
    "orc_residual_adaln_rows": ([_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _P, _P, _F, _F, _P, _P, _P, _P, _P], None),
    "orc_global_scale_from_amax": ([_F], _F),
    "orc_scale_offset": ([_I64, _I64, _I64], _I64),
    "orc_padded_rows": ([_I64], _I64),
    "orc_scale_offsets_rows": ([_P, _I64, _I64, _P], None),
    "orc_swizzle_scales": ([_P, _I64, _I64, _P], None),
    "orc_quantize_rows": ([_P, _I64, _I64, _I64, _F, _P, _P, _P], None),
    "orc_row_rstd": ([_P, _I64, _F], _F),
    "orc_adaln_rows": ([_P, _I64, _I64, _I64, _P, _P, _P, _F, _F, _P, _P, _P, _P, _P], None),
    "orc_swiglu_rows": ([_P, _I64, _P, _I64, _I64, _I64, _F, _P, _P, _P, _P], None),
    "orc_dequantize_rows": ([_P, _P, _I64, _I64, _F, _P], None),
    "orc_bf16_bits_array": ([_P, _I64, _P], None),
    "orc_e4m3_encode_array": ([_P, _I64, _P], None),
    "orc_e2m1_encode_array": ([_P, _I64, _P], None),
    "orc_exp_array": ([_P, _I64, _P], None),
    "orc_swiglu_value_array": ([_P, _P, _I64, _P], None),
}


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            handle = ctypes.CDLL(build())
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 data must be passed as uint16 bit patterns, got {a.dtype}")
    return a


def _check_cols(cols: int) -> None:
    if cols <= 0 or cols % 64:
        raise ValueError(f"cols must be a positive multiple of 64, got {cols}")


def _split(n: int, threads: int):
    threads = max(1, min(threads, n))
    step = (n + threads - 1) // threads
    return [(s, min(n, s + step)) for s in range(0, n, step)]


# --------------------------------------------------------------------------- #
# element-wise conversions (used by the pins)                                  #
# --------------------------------------------------------------------------- #

def bf16_bits(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_bits_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_value(bits: np.ndarray) -> np.ndarray:
    bits = _u16(bits)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e2m1_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def exp_c(z: np.ndarray) -> np.ndarray:
    z = np.ascontiguousarray(z, dtype=np.float32)
    out = np.empty(z.shape, np.float32)
    lib().orc_exp_array(_ptr(z), z.size, _ptr(out))
    return out


def exp_constants() -> dict:
    buf = np.zeros(11, np.float32)
    lib().orc_exp_constants(_ptr(buf))
    names = ["L2E", "C1", "C2"] + [f"P{n}" for n in range(8)]
    return dict(zip(names, buf.tolist()))


def swiglu_value(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(gate, dtype=np.float32)
    u = np.ascontiguousarray(up, dtype=np.float32)
    assert g.shape == u.shape
    out = np.empty(g.shape, np.float32)
    lib().orc_swiglu_value_array(_ptr(g), _ptr(u), g.size, _ptr(out))
    return out


def quantize_block(y, gsf: float):
    """(scale byte, 8 packed code bytes) of one 16-element block of fp32 values."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    assert y.shape == (16,)
    sf = np.zeros(1, np.uint8)
    packed = np.zeros(8, np.uint8)
    lib().orc_quantize_block(_ptr(y), float(gsf), _ptr(sf), _ptr(packed))
    return int(sf[0]), packed


def global_scale(amax: float) -> float:
    """fl(448 * 6 / amax): the static per-tensor scale for a tensor amax."""
    if not amax > 0:
        raise ValueError("global amax must be positive")
    return float(lib().orc_global_scale(float(amax)))


def amax_bf16(bits: np.ndarray) -> float:
    """max |v| over bf16 values given as uint16 bit patterns (exact; 0 when empty)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return float(lib().orc_amax_bf16(_ptr(b), b.size))


def global_scale_from_amax(amax: float) -> float:
    """fl(2688 / amax) with amax = 0 giving 1 and +inf clamped to the largest float."""
    return float(lib().orc_global_scale_from_amax(float(amax)))


# --------------------------------------------------------------------------- #
# layout                                                                        #
# --------------------------------------------------------------------------- #

def padded_rows(rows: int) -> int:
    return int(lib().orc_padded_rows(rows))


def scale_offset(row: int, group: int, cols: int) -> int:
    return int(lib().orc_scale_offset(row, group, cols))


def scale_offsets(rows: np.ndarray, cols: int) -> np.ndarray:
    """[len(rows), cols/16] int64 swizzled offsets of the scales of the given rows."""
    rows = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    out = np.empty((rows.size, cols // 16), np.int64)
    lib().orc_scale_offsets_rows(_ptr(rows), rows.size, cols, _ptr(out))
    return out


def swizzle_scales(sf_logical: np.ndarray, rows: int, cols: int) -> np.ndarray:
    _check_cols(cols)
    sf = np.ascontiguousarray(sf_logical, dtype=np.uint8)
    assert sf.shape == (rows, cols // 16)
    out = np.empty(padded_rows(rows) * (cols // 16), np.uint8)
    lib().orc_swizzle_scales(_ptr(sf), rows, cols, _ptr(out))
    return out


# --------------------------------------------------------------------------- #
# row producers                                                                 #
# --------------------------------------------------------------------------- #

def quantize_rows(x_bits: np.ndarray, gsf: float, threads: int = 1):
    """Standalone quantize of bf16 rows [n, cols] -> (codes [n, cols/2], sf [n, cols/16])."""
    x = _u16(x_bits)
    n, cols = x.shape
    _check_cols(cols)
    codes = np.empty((n, cols // 2), np.uint8)
    sf = np.empty((n, cols // 16), np.uint8)

    def work(span):
        a, b = span
        scratch = np.empty(cols, np.float32)
        lib().orc_quantize_rows(_ptr(x[a:b]), b - a, cols, cols, float(gsf), _ptr(scratch),
                                _ptr(codes[a:b]), _ptr(sf[a:b]))

    _run(work, n, threads)
    return codes, sf


def sumsq_bf16(bits: np.ndarray, lanes: int = 128) -> float:
    """The canonical sum of squares of bf16 values (bit patterns): 128 lanes for a
    row, hd/8 for a head of hd values."""
    x = _u16(bits).ravel()
    _check_lanes(x.size, lanes)
    return float(lib().orc_sumsq_bf16(_ptr(x), x.size, int(lanes)))


def sumsq_f32(values: np.ndarray, lanes: int = 128) -> float:
    """The canonical sum of squares of binary32 values (same order as sumsq_bf16)."""
    v = np.ascontiguousarray(values, dtype=np.float32).ravel()
    _check_lanes(v.size, lanes)
    return float(lib().orc_sumsq_f32(_ptr(v), v.size, int(lanes)))


def _check_lanes(n: int, lanes: int) -> None:
    if n % 8 or not (lanes == 128 or lanes in (2, 4, 8, 16, 32)):
        raise ValueError(f"the canonical order takes n % 8 == 0 and 128 or 2..32 (a power of two) "
                         f"lanes, got n={n}, lanes={lanes}")
    if lanes != 128 and n != 8 * lanes:
        raise ValueError("a head has one chunk per lane: n must be 8 * lanes")


def head_rstd(values: np.ndarray, eps: float) -> float:
    """rstd of one head of the QKV epilogue: hd binary32 values, hd/8 lanes."""
    v = np.ascontiguousarray(values, dtype=np.float32).ravel()
    _check_lanes(v.size, v.size // 8)
    return float(lib().orc_head_rstd(_ptr(v), v.size, float(eps)))


def row_rstd(x_row_bits: np.ndarray, eps: float) -> float:
    x = _u16(x_row_bits)
    _check_cols(x.size)
    return float(lib().orc_row_rstd(_ptr(x), x.size, float(eps)))


def adaln_rows(x_bits, gamma_bits, table_bits, frames, eps: float, gsf: float | None,
               want_y: bool = False, threads: int = 1):
    """RMSNorm + AdaLN -> NVFP4 of bf16 rows [n, cols].

    ``table_bits`` is [T, 2, cols] (index 0 shift, 1 scale); ``frames[i]`` is
    the frame of row i.  With ``gsf=None`` only rstd (and y) are produced.
    Returns (codes, sf, rstd, y) with y (bf16 bits) or None.
    """
    x = _u16(x_bits)
    n, cols = x.shape
    _check_cols(cols)
    gamma = _u16(gamma_bits).reshape(cols)
    table = _u16(table_bits)
    assert table.ndim == 3 and table.shape[1:] == (2, cols)
    frames = np.ascontiguousarray(frames, dtype=np.int64).reshape(n)
    if n and (frames.min() < 0 or frames.max() >= table.shape[0]):
        raise ValueError("frame index outside [0, frames)")
    quant = gsf is not None
    codes = np.empty((n, cols // 2), np.uint8) if quant else None
    sf = np.empty((n, cols // 16), np.uint8) if quant else None
    rstd = np.empty(n, np.float32)
    y = np.empty((n, cols), np.uint16) if want_y else None

    def work(span):
        a, b = span
        scratch = np.empty(cols, np.float32)
        lib().orc_adaln_rows(_ptr(x[a:b]), b - a, cols, cols, _ptr(gamma), _ptr(table),
                             _ptr(frames[a:b]), float(eps), float(gsf if quant else 1.0),
                             _ptr(scratch), _ptr(codes[a:b]) if quant else None,
                             _ptr(sf[a:b]) if quant else None, _ptr(rstd[a:b]),
                             _ptr(y[a:b]) if want_y else None)

    _run(work, n, threads)
    return codes, sf, rstd, y


def row_rstd_f32(row: np.ndarray, eps: float) -> float:
    """rstd of one fp32 row in the canonical order (squares of fp32 values)."""
    r = np.ascontiguousarray(row, dtype=np.float32).ravel()
    _check_cols(r.size)
    return float(lib().orc_row_rstd_f32(_ptr(r), r.size, float(eps)))


def residual_adaln_rows(h, o_bits, bias_bits, gate_bits, gamma_bits, table_bits, frames, eps: float,
                        gsf: float | None, want_y: bool = False, threads: int = 1):
    """Residual fold + RMSNorm + AdaLN -> NVFP4.

    ``h`` fp32 [n, cols] (not modified; the folded residual is returned), ``o``
    bf16 bits [n, cols], ``bias`` bf16 bits [cols] or None, ``gate`` bf16 bits
    [T, cols], ``table`` [T, 2, cols]; ``frames[i]`` indexes both tables.
    Returns (h_out, codes, sf, rstd, y)."""
    h_out = np.array(h, dtype=np.float32, copy=True, order="C")
    o = _u16(o_bits)
    n, cols = o.shape
    _check_cols(cols)
    assert h_out.shape == (n, cols)
    bias = None if bias_bits is None else _u16(bias_bits).reshape(cols)
    gate = _u16(gate_bits)
    assert gate.ndim == 2 and gate.shape[1] == cols
    gamma = _u16(gamma_bits).reshape(cols)
    table = _u16(table_bits)
    assert table.ndim == 3 and table.shape[1:] == (2, cols) and table.shape[0] == gate.shape[0]
    frames = np.ascontiguousarray(frames, dtype=np.int64).reshape(n)
    if n and (frames.min() < 0 or frames.max() >= table.shape[0]):
        raise ValueError("frame index outside [0, frames)")
    quant = gsf is not None
    codes = np.empty((n, cols // 2), np.uint8) if quant else None
    sf = np.empty((n, cols // 16), np.uint8) if quant else None
    rstd = np.empty(n, np.float32)
    y = np.empty((n, cols), np.uint16) if want_y else None

    def work(span):
        a, b = span
        scratch = np.empty(cols, np.float32)
        lib().orc_residual_adaln_rows(
            _ptr(h_out[a:b]), b - a, cols, cols, _ptr(o[a:b]), cols,
            _ptr(bias) if bias is not None else None, _ptr(gate), _ptr(gamma), _ptr(table),
            _ptr(frames[a:b]), float(eps), float(gsf if quant else 1.0), _ptr(scratch),
            _ptr(codes[a:b]) if quant else None, _ptr(sf[a:b]) if quant else None,
            _ptr(rstd[a:b]), _ptr(y[a:b]) if want_y else None)

    _run(work, n, threads)
    return h_out, codes, sf, rstd, y


def swiglu_rows(gate_bits, up_bits, gsf: float | None, want_y: bool = False, threads: int = 1):
    """silu(gate) * up -> NVFP4 of bf16 rows [n, cols]. Returns (codes, sf, y)."""
    g = _u16(gate_bits)
    u = _u16(up_bits)
    assert g.shape == u.shape
    n, cols = g.shape
    _check_cols(cols)
    quant = gsf is not None
    codes = np.empty((n, cols // 2), np.uint8) if quant else None
    sf = np.empty((n, cols // 16), np.uint8) if quant else None
    y = np.empty((n, cols), np.uint16) if want_y else None

    def work(span):
        a, b = span
        scratch = np.empty(cols, np.float32)
        lib().orc_swiglu_rows(_ptr(g[a:b]), cols, _ptr(u[a:b]), cols, b - a, cols,
                              float(gsf if quant else 1.0), _ptr(scratch),
                              _ptr(codes[a:b]) if quant else None,
                              _ptr(sf[a:b]) if quant else None,
                              _ptr(y[a:b]) if want_y else None)

    _run(work, n, threads)
    return codes, sf, y


def swiglu_packed_rows(o_bits, bias_bits, gsf: float | None, want_y: bool = False, threads: int = 1):
    """SwiGLU of a value-first packed projection o [n, 2F] (value, then gate) plus
    its bias [2F] (or None) -> NVFP4 of the [n, F] output. Returns (codes, sf, y)."""
    o = _u16(o_bits)
    n, two_f = o.shape
    f = two_f // 2
    _check_cols(f)
    bias = None if bias_bits is None else _u16(bias_bits).reshape(two_f)
    quant = gsf is not None
    codes = np.empty((n, f // 2), np.uint8) if quant else None
    sf = np.empty((n, f // 16), np.uint8) if quant else None
    y = np.empty((n, f), np.uint16) if want_y else None

    def work(span):
        a, b = span
        scratch = np.empty(f, np.float32)
        lib().orc_swiglu_packed_rows(_ptr(o[a:b]), two_f, _ptr(bias) if bias is not None else None,
                                     b - a, f, float(gsf if quant else 1.0), _ptr(scratch),
                                     _ptr(codes[a:b]) if quant else None,
                                     _ptr(sf[a:b]) if quant else None, _ptr(y[a:b]) if want_y else None)

    _run(work, n, threads)
    return codes, sf, y


def qkv_epilogue_rows(x_bits, bias_bits, heads: int, cos_bits, sin_bits, eps: float, is_v: bool,
                      threads: int = 1, interleaved: bool = False) -> np.ndarray:
    """QKV epilogue of one projected tensor x [n, heads * HD] (bf16 bits) with its bias
    [heads * HD]: v gets the bias only; q and k the bias, the per-head RMSNorm and the
    RoPE on the first ROT values of each head (cos, sin bf16 [n, ROT]): rotate-half
    pairs (i, i + ROT/2), or with `interleaved` the pairs (2j, 2j + 1).
    Returns bf16 bits [n, heads, HD]."""
    x = _u16(x_bits)
    n, d = x.shape
    hd = d // heads
    # the canonical order takes hd/8 lanes, a power of two up to 32
    assert hd * heads == d and hd in (16, 32, 64, 128, 256)
    bias = _u16(bias_bits).reshape(d)
    # ROT is the tables' width; no tables is ROT = 0: the norm without a rotation
    cos = _u16(cos_bits) if cos_bits is not None else np.zeros((n, 0), np.uint16)
    sin = _u16(sin_bits) if sin_bits is not None else np.zeros((n, 0), np.uint16)
    rot = cos.shape[1]
    assert cos.shape == (n, rot) and sin.shape == (n, rot) and rot <= hd and rot % 2 == 0
    out = np.empty((n, heads, hd), np.uint16)

    def work(span):
        a, b = span
        lib().orc_qkv_epilogue_rows(_ptr(x[a:b]), d, _ptr(bias), b - a, heads, hd, int(is_v),
                                    _ptr(cos[a:b]), _ptr(sin[a:b]), rot, int(interleaved), float(eps),
                                    _ptr(out[a:b]))

    _run(work, n, threads)
    return out


def nvfp4_gemm(a_codes: np.ndarray, a_sf: np.ndarray, b_codes: np.ndarray, b_sf: np.ndarray,
               threads: int = 1) -> np.ndarray:
    """acc [m, n] = fl(exact sum over k of a * b) of NVFP4 A [m, k] (codes [m, k/2],
    logical scales [m, k/16]) and B [n, k] (codes [n, k/2], scales [n, k/16])."""
    a = np.ascontiguousarray(a_codes, dtype=np.uint8)
    b = np.ascontiguousarray(b_codes, dtype=np.uint8)
    sfa = np.ascontiguousarray(a_sf, dtype=np.uint8)
    sfb = np.ascontiguousarray(b_sf, dtype=np.uint8)
    m, half = a.shape
    n = b.shape[0]
    k = 2 * half
    if k % 16 or k > 2**19:
        raise ValueError("k must be a multiple of 16, at most 2^19")
    assert b.shape == (n, half) and sfa.shape == (m, k // 16) and sfb.shape == (n, k // 16)
    if any(((sf & 0x80) != 0).any() or (sf == 0x7F).any() for sf in (sfa, sfb)):
        raise ValueError("scale bytes must be E4M3 codes 0x00..0x7E")
    acc = np.empty((m, n), np.float32)

    def work(span):
        i0, i1 = span
        au = np.empty((i1 - i0) * k, np.int64)
        bu = np.empty(k, np.int64)
        lib().orc_nvfp4_gemm_rows(_ptr(a), _ptr(sfa), i0, i1, k, _ptr(b), _ptr(sfb), n, _ptr(au),
                                  _ptr(bu), _ptr(acc[i0:i1]))

    _run(work, m, threads)
    return acc


def swiglu_epilogue_rows(acc: np.ndarray, alpha: float, gsf: float | None, want_y: bool = False,
                         threads: int = 1):
    """The GEMM's SwiGLU + NVFP4 epilogue on acc [m, n] (column 2j the value, 2j+1
    the gate of output j): returns (codes [m, n/4], logical scales [m, n/32], y bf16
    bits [m, n/2] or None)."""
    acc = np.ascontiguousarray(acc, dtype=np.float32)
    m, n = acc.shape
    f = n // 2
    _check_cols(f)
    quant = gsf is not None
    codes = np.empty((m, f // 2), np.uint8) if quant else None
    sf = np.empty((m, f // 16), np.uint8) if quant else None
    y = np.empty((m, f), np.uint16) if want_y else None

    def work(span):
        a, b = span
        scratch = np.empty(f, np.float32)
        lib().orc_swiglu_epilogue_rows(_ptr(acc[a:b]), b - a, n, float(alpha),
                                       float(gsf if quant else 1.0), _ptr(scratch),
                                       _ptr(codes[a:b]) if quant else None,
                                       _ptr(sf[a:b]) if quant else None, _ptr(y[a:b]) if want_y else None)

    _run(work, m, threads)
    return codes, sf, y


def dequantize_rows(codes: np.ndarray, sf_logical: np.ndarray, gsf: float,
                    threads: int = 1) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf_logical, dtype=np.uint8)
    n, half = codes.shape
    cols = 2 * half
    _check_cols(cols)
    assert sf.shape == (n, cols // 16)
    out = np.empty((n, cols), np.float32)

    def work(span):
        a, b = span
        lib().orc_dequantize_rows(_ptr(codes[a:b]), _ptr(sf[a:b]), b - a, cols, float(gsf),
                                  _ptr(out[a:b]))

    _run(work, n, threads)
    return out


def _run(work, n: int, threads: int) -> None:
    if n == 0:
        return
    spans = _split(n, threads)
    if len(spans) == 1:
        work(spans[0])
        return
    # ctypes releases the GIL during the C call, so row spans run in parallel.
    with ThreadPoolExecutor(len(spans)) as pool:
        list(pool.map(work, spans))
