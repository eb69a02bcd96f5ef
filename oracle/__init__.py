"""CPU oracle for the FP8 weight-only linear layer (numpy front end).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg, never by the library.  The arithmetic lives in
fp8w_oracle.c (plain C, fp64 for the linear layer); this module only moves
numpy arrays across ctypes.

Each function follows page "kadirnar/kernel-agent fp8-weights", section
"The contract", unless its docstring names another passage.
"""
import ctypes
import os

import numpy as np

from . import build as _build

ACT_BF16 = 1
ACT_F16 = 2

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        c = ctypes
        P = c.c_void_p
        lib.oracle_e4m3_decode.restype = c.c_double
        lib.oracle_e4m3_decode.argtypes = [c.c_uint8]
        lib.oracle_e4m3_encode.restype = c.c_uint8
        lib.oracle_e4m3_encode.argtypes = [c.c_float]
        lib.oracle_row_scale.restype = c.c_float
        lib.oracle_row_scale.argtypes = [P, c.c_int64]
        lib.oracle_quantize.restype = None
        lib.oracle_quantize.argtypes = [P, c.c_int64, c.c_int64, P, P]
        lib.oracle_dequantize.restype = None
        lib.oracle_dequantize.argtypes = [P, P, c.c_int64, c.c_int64, P]
        lib.oracle_round_bf16.restype = c.c_uint16
        lib.oracle_round_bf16.argtypes = [c.c_double]
        lib.oracle_round_f16.restype = c.c_uint16
        lib.oracle_round_f16.argtypes = [c.c_double]
        lib.oracle_bf16_value.restype = c.c_double
        lib.oracle_bf16_value.argtypes = [c.c_uint16]
        lib.oracle_f16_value.restype = c.c_double
        lib.oracle_f16_value.argtypes = [c.c_uint16]
        lib.oracle_linear.restype = c.c_int
        lib.oracle_linear.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, P,
                                      c.c_int64, P, P, c.c_int]
        lib.oracle_quantize_grouped.restype = None
        lib.oracle_quantize_grouped.argtypes = [P, c.c_int64, c.c_int64, c.c_int64, P, P]
        lib.oracle_linear_grouped.restype = c.c_int
        lib.oracle_linear_grouped.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, c.c_int64, P,
                                              c.c_int64, P, P, c.c_int]
        lib.oracle_e8m0_decode.restype = c.c_double
        lib.oracle_e8m0_decode.argtypes = [c.c_uint8]
        lib.oracle_mx_scale.restype = c.c_uint8
        lib.oracle_mx_scale.argtypes = [P, c.c_int64]
        lib.oracle_quantize_mx.restype = None
        lib.oracle_quantize_mx.argtypes = [P, c.c_int64, c.c_int64, P, P]
        lib.oracle_linear_mx.restype = c.c_int
        lib.oracle_linear_mx.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, P,
                                         c.c_int64, P, P, c.c_int]
        lib.oracle_dequantize_grouped.restype = None
        lib.oracle_dequantize_grouped.argtypes = [P, P, c.c_int64, c.c_int64, c.c_int64, P]
        lib.oracle_dequantize_mx.restype = None
        lib.oracle_dequantize_mx.argtypes = [P, P, c.c_int64, c.c_int64, P]
        lib.oracle_linear_w8a8.restype = c.c_int
        lib.oracle_linear_w8a8.argtypes = [P, P, c.c_int, c.c_int64, c.c_int64, P, P, P, c.c_int64, P, P]
        lib.oracle_fp8_error.restype = None
        lib.oracle_fp8_error.argtypes = [P, c.c_int64, c.c_int64, P, P, P]
        lib.oracle_e4m3_encode_many.restype = None
        lib.oracle_e4m3_encode_many.argtypes = [P, c.c_int64, P]
        lib.oracle_round_bf16_many.restype = None
        lib.oracle_round_bf16_many.argtypes = [P, c.c_int64, P]
        lib.oracle_round_f16_many.restype = None
        lib.oracle_round_f16_many.argtypes = [P, c.c_int64, P]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e4m3_decode(code: int) -> float:
    """Value of one OCP e4m3 byte (NaN for 0x7F/0xFF)."""
    return _load().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_decode_table() -> np.ndarray:
    """fp64 values of all 256 codes, index = code."""
    lib = _load()
    return np.array([lib.oracle_e4m3_decode(b) for b in range(256)], dtype=np.float64)


def e4m3_encode(v) -> np.ndarray:
    """Round-to-nearest-even, saturating e4m3 encode of fp32 values."""
    v = _c(np.atleast_1d(v), np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_many(_ptr(v), v.size, _ptr(out))
    return out


def row_scale(row) -> np.float32:
    row = _c(row, np.float32)
    return np.float32(_load().oracle_row_scale(_ptr(row), row.size))


def quantize(w):
    """W[N,K] fp32 -> (codes uint8 [N,K], scales fp32 [N])."""
    w = _c(w, np.float32)
    n, k = w.shape
    codes = np.empty((n, k), dtype=np.uint8)
    scales = np.empty(n, dtype=np.float32)
    _load().oracle_quantize(_ptr(w), n, k, _ptr(codes), _ptr(scales))
    return codes, scales


def widen_16(bits, act: int) -> np.ndarray:
    """fp32 values of bf16 (act=1) or fp16 (act=2) bit patterns: exact, as
    every bf16 and fp16 value is an fp32 value (page "B04 Precision &
    Quantization", section 2, the bf16 and fp16 rows)."""
    return act_values(bits, act).astype(np.float32)


def quantize_16(w_bits, act: int):
    """Weights stored as bf16 (act=1) or fp16 (act=2) bits: widened to fp32,
    then the per-channel rule."""
    return quantize(widen_16(w_bits, act))


def dequantize(codes, scales) -> np.ndarray:
    """fp64 W' = scale[n] * e4m3val(codes[n,k])."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    n, k = codes.shape
    out = np.empty((n, k), dtype=np.float64)
    _load().oracle_dequantize(_ptr(codes), _ptr(scales), n, k, _ptr(out))
    return out


def round_bf16(v) -> np.ndarray:
    """fp64 -> bf16 bits (uint16), one RNE rounding."""
    v = _c(np.atleast_1d(v), np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round_bf16_many(_ptr(v), v.size, _ptr(out))
    return out


def round_f16(v) -> np.ndarray:
    """fp64 -> fp16 bits (uint16), one RNE rounding."""
    v = _c(np.atleast_1d(v), np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round_f16_many(_ptr(v), v.size, _ptr(out))
    return out


def act_values(bits, act: int) -> np.ndarray:
    """fp64 values of bf16 (act=1) or fp16 (act=2) bit patterns."""
    lib = _load()
    f = lib.oracle_f16_value if act == ACT_F16 else lib.oracle_bf16_value
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([f(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


def linear(x_bits, act: int, codes, scales, bias=None, threads: int = 1,
           want_acc: bool = False):
    """y[M,N] = round_act(scale[n] * sum_k x[m,k] e4m3val(q[n,k]) + bias[n]).

    x_bits: uint16 [M,K] bf16/fp16 bit patterns.  Returns y bits (uint16
    [M,N]) and, with want_acc, also the unrounded fp64 value.
    """
    x_bits = _c(x_bits, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    m, k = x_bits.shape
    n, k2 = codes.shape
    if k != k2 or scales.shape != (n,) or (bias is not None and bias.shape != (n,)):
        raise ValueError("oracle.linear: shape mismatch")
    y = np.empty((m, n), dtype=np.uint16)
    acc = np.empty((m, n), dtype=np.float64) if want_acc else None
    rc = _load().oracle_linear(_ptr(x_bits), act, m, k, _ptr(codes), _ptr(scales),
                               _ptr(bias), n, _ptr(y), _ptr(acc), int(threads))
    if rc != 0:
        raise RuntimeError("oracle.linear: thread start failed")
    return (y, acc) if want_acc else y


def quantize_grouped(w, group: int):
    """W[N,K] fp32 -> (codes uint8 [N,K], scales fp32 [N, K/group]): one
    scale per run of `group` weights of a row, each by the per-row rule."""
    w = _c(w, np.float32)
    n, k = w.shape
    if group < 1 or k % group:
        raise ValueError("oracle.quantize_grouped: k must be a multiple of group")
    codes = np.empty((n, k), dtype=np.uint8)
    scales = np.empty((n, k // group), dtype=np.float32)
    _load().oracle_quantize_grouped(_ptr(w), n, k, group, _ptr(codes), _ptr(scales))
    return codes, scales


def linear_grouped(x_bits, act: int, codes, scales, group: int, bias=None, threads: int = 1,
                   want_acc: bool = False):
    """y[M,N] = round_act(sum_j scale[n,j] * sum_{k in group j} x[m,k] e4m3val(q[n,k]) + bias[n])."""
    x_bits = _c(x_bits, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    m, k = x_bits.shape
    n, k2 = codes.shape
    if k != k2 or k % group or scales.shape != (n, k // group) or (bias is not None and bias.shape != (n,)):
        raise ValueError("oracle.linear_grouped: shape mismatch")
    y = np.empty((m, n), dtype=np.uint16)
    acc = np.empty((m, n), dtype=np.float64) if want_acc else None
    rc = _load().oracle_linear_grouped(_ptr(x_bits), act, m, k, _ptr(codes), _ptr(scales), group,
                                       _ptr(bias), n, _ptr(y), _ptr(acc), int(threads))
    if rc != 0:
        raise RuntimeError("oracle.linear_grouped: thread start failed")
    return (y, acc) if want_acc else y


MX_BLOCK = 32


def e8m0_decode(b: int) -> float:
    """Value of one E8M0 byte: 2^(b - 127), NaN for 0xFF (page "11.
    Inference with NVFP4/MXFP8", section "MXFP8-Style FP8")."""
    return _load().oracle_e8m0_decode(int(b) & 0xFF)


def mx_scale(block) -> int:
    """E8M0 byte of one block of weights: the smallest 2^e >= amax/448."""
    block = _c(block, np.float32)
    return int(_load().oracle_mx_scale(_ptr(block), block.size))


def quantize_mx(w):
    """W[N,K] fp32 -> (codes uint8 [N,K], E8M0 scales uint8 [N, K/32])."""
    w = _c(w, np.float32)
    n, k = w.shape
    if k % MX_BLOCK:
        raise ValueError("oracle.quantize_mx: k must be a multiple of 32")
    codes = np.empty((n, k), dtype=np.uint8)
    scales = np.empty((n, k // MX_BLOCK), dtype=np.uint8)
    _load().oracle_quantize_mx(_ptr(w), n, k, _ptr(codes), _ptr(scales))
    return codes, scales


def linear_mx(x_bits, act: int, codes, scales, bias=None, threads: int = 1, want_acc: bool = False):
    """The per-group linear layer, g = 32, with scale[n, j] = e8m0val(scales[n, j])."""
    x_bits = _c(x_bits, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    bias = None if bias is None else _c(bias, np.float32)
    m, k = x_bits.shape
    n, k2 = codes.shape
    if k != k2 or k % MX_BLOCK or scales.shape != (n, k // MX_BLOCK) or (bias is not None and bias.shape != (n,)):
        raise ValueError("oracle.linear_mx: shape mismatch")
    y = np.empty((m, n), dtype=np.uint16)
    acc = np.empty((m, n), dtype=np.float64) if want_acc else None
    rc = _load().oracle_linear_mx(_ptr(x_bits), act, m, k, _ptr(codes), _ptr(scales),
                                  _ptr(bias), n, _ptr(y), _ptr(acc), int(threads))
    if rc != 0:
        raise RuntimeError("oracle.linear_mx: allocation or thread start failed")
    return (y, acc) if want_acc else y


def dequantize_grouped(codes, scales, group: int) -> np.ndarray:
    """fp64 W'[n, k] = scales[n, k // group] * e4m3val(codes[n, k])."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    n, k = codes.shape
    if k % group or scales.shape != (n, k // group):
        raise ValueError("oracle.dequantize_grouped: shape mismatch")
    out = np.empty((n, k), dtype=np.float64)
    _load().oracle_dequantize_grouped(_ptr(codes), _ptr(scales), n, k, group, _ptr(out))
    return out


def dequantize_mx(codes, scales) -> np.ndarray:
    """fp64 W'[n, k] = e8m0val(scales[n, k // 32]) * e4m3val(codes[n, k])."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    n, k = codes.shape
    if k % MX_BLOCK or scales.shape != (n, k // MX_BLOCK):
        raise ValueError("oracle.dequantize_mx: shape mismatch")
    out = np.empty((n, k), dtype=np.float64)
    _load().oracle_dequantize_mx(_ptr(codes), _ptr(scales), n, k, _ptr(out))
    return out


def quantize_act(x_bits, act: int):
    """W8A8 activation quantisation (page "tensormux Write an FP8 kernel",
    per-token scales): each row of the bf16/fp16 activations, widened
    exactly to fp32, by the per-row rule -> (codes uint8 [M, K], scales fp32 [M])."""
    return quantize_16(x_bits, act)


def linear_w8a8(qx, sx, act: int, qw, sw, bias=None, want_acc: bool = False):
    """y[M,N] = round_act(sx[m] * sw[n] * sum_k e4m3val(qx[m,k]) e4m3val(qw[n,k]) + bias[n]), fp64."""
    qx = _c(qx, np.uint8)
    sx = _c(sx, np.float32)
    qw = _c(qw, np.uint8)
    sw = _c(sw, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    m, k = qx.shape
    n, k2 = qw.shape
    if k != k2 or sx.shape != (m,) or sw.shape != (n,) or (bias is not None and bias.shape != (n,)):
        raise ValueError("oracle.linear_w8a8: shape mismatch")
    y = np.empty((m, n), dtype=np.uint16)
    acc = np.empty((m, n), dtype=np.float64) if want_acc else None
    _load().oracle_linear_w8a8(_ptr(qx), _ptr(sx), act, m, k, _ptr(qw), _ptr(sw), _ptr(bias), n, _ptr(y),
                               _ptr(acc))
    return (y, acc) if want_acc else y


def fp8_error(w, codes, scales) -> dict:
    """Weight report: rel_l2, worst_channel_rel_l2, underflow, crest (the
    readings are in the C source; the pages name the fields only)."""
    w = _c(w, np.float32)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    n, k = w.shape
    out = np.zeros(4, dtype=np.float64)
    _load().oracle_fp8_error(_ptr(w), n, k, _ptr(codes), _ptr(scales), _ptr(out))
    return {"rel_l2": out[0], "worst_channel_rel_l2": out[1],
            "underflow": out[2], "crest": out[3]}


def host_cores() -> int:
    """Cores this process may run on (for the CPU baseline's thread count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1
