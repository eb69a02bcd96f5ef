"""fp8_weight_only_gb300 -- Python binding of libfp8w (include/fp8w.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  There
is no CPU fallback: if libfp8w.so is missing or a call fails, an exception is
raised.

    codes, scales = quantize(w)                 # w: [N, K] fp32 CUDA tensor
    y = linear(x, codes, scales, bias)          # x: [M, K] bf16/fp16 CUDA tensor
    codes, e8 = quantize_mx(w)                  # one E8M0 scale byte per 32 along K
    y = linear(x, codes, e8, bias)              # bf16 x for M > 1
    qx, sx = quantize_act(x)                    # W8A8: per-token e4m3 activations
    y = linear_w8a8(qx, sx, codes, scales, bias, out_dtype=torch.bfloat16)
"""
import ctypes
import os

from .fp8w_file import Fp8wFileError, load as load_fp8w, save as save_fp8w  # noqa: F401  (the .fp8w file)

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8w.so")

FP8W_BF16 = 1
FP8W_F16 = 2
FP8W_F32 = 3
KERNEL_AUTO, KERNEL_GEMV, KERNEL_SKINNY, KERNEL_PREFILL = 0, 1, 2, 3

SYMBOLS = ("fp8w_quantize", "fp8w_linear", "fp8w_linear_ex",
           "fp8w_status_string", "fp8w_last_cuda_error", "fp8w_device_error", "fp8w_abi_version",
           "fp8w_linear_noalloc", "fp8w_dequantize", "fp8w_quantize_grouped", "fp8w_linear_grouped",
           "fp8w_quantize_mx", "fp8w_linear_mx", "fp8w_quantize_ex", "fp8w_dequantize_grouped",
           "fp8w_dequantize_mx", "fp8w_quantize_act", "fp8w_linear_w8a8")
ABI_VERSION = 12
FLAG_WEIGHTS_READY = 1


class Fp8wError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(msg)
        self.status = status


class LinearConfig(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("cluster", ctypes.c_int), ("tiles", ctypes.c_int),
                ("flags", ctypes.c_int), ("reserved", ctypes.c_int * 4)]


_lib = None


def lib():
    """The loaded libfp8w (ctypes.CDLL); raises if it was never built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise Fp8wError(-1, "libfp8w.so is not built (run __graft_entry__.build() or "
                                "python fp8_weight_only_gb300/build.py)")
        L = ctypes.CDLL(LIB_PATH)
        c, P = ctypes, ctypes.c_void_p
        L.fp8w_quantize.restype = c.c_int
        L.fp8w_quantize.argtypes = [P, c.c_int64, c.c_int64, P, P, P]
        L.fp8w_quantize_grouped.restype = c.c_int
        L.fp8w_quantize_grouped.argtypes = [P, c.c_int64, c.c_int64, c.c_int, P, P, P]
        L.fp8w_linear_grouped.restype = c.c_int
        L.fp8w_linear_grouped.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, c.c_int, P, c.c_int64, P, P]
        L.fp8w_quantize_ex.restype = c.c_int
        L.fp8w_quantize_ex.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, P]
        L.fp8w_quantize_mx.restype = c.c_int
        L.fp8w_quantize_mx.argtypes = [P, c.c_int64, c.c_int64, P, P, P]
        L.fp8w_linear_mx.restype = c.c_int
        L.fp8w_linear_mx.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, P, c.c_int64, P, P]
        L.fp8w_dequantize_grouped.restype = c.c_int
        L.fp8w_dequantize_grouped.argtypes = [P, P, c.c_int, c.c_int64, c.c_int64, c.c_int, P, P]
        L.fp8w_dequantize_mx.restype = c.c_int
        L.fp8w_dequantize_mx.argtypes = [P, P, c.c_int64, c.c_int64, c.c_int, P, P]
        L.fp8w_dequantize.restype = c.c_int
        L.fp8w_dequantize.argtypes = [P, P, c.c_int64, c.c_int64, c.c_int, P, P]
        L.fp8w_linear.restype = c.c_int
        L.fp8w_linear.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, P, c.c_int64, P, P]
        L.fp8w_linear_ex.restype = c.c_int
        L.fp8w_linear_ex.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, P, c.c_int64, P,
                                     c.POINTER(LinearConfig), P]
        L.fp8w_linear_noalloc.restype = c.c_int
        L.fp8w_linear_noalloc.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, P, c.c_int64, P, P]
        L.fp8w_quantize_act.restype = c.c_int
        L.fp8w_quantize_act.argtypes = [P, c.c_int, c.c_int64, c.c_int64, P, P, P]
        L.fp8w_linear_w8a8.restype = c.c_int
        L.fp8w_linear_w8a8.argtypes = [P, P, c.c_int64, c.c_int64, P, P, P, c.c_int64, P, c.c_int, c.c_int, P]
        L.fp8w_status_string.restype = c.c_char_p
        L.fp8w_status_string.argtypes = [c.c_int]
        L.fp8w_last_cuda_error.restype = c.c_char_p
        L.fp8w_last_cuda_error.argtypes = []
        L.fp8w_device_error.restype = c.c_int
        L.fp8w_device_error.argtypes = []
        L.fp8w_abi_version.restype = c.c_int
        L.fp8w_abi_version.argtypes = []
        _lib = L
    return _lib


def _check(status):
    if status != 0:
        L = lib()
        msg = L.fp8w_status_string(status).decode()
        if status == 5:
            msg += ": " + L.fp8w_last_cuda_error().decode()
        raise Fp8wError(status, msg)


def _stream(t):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _act(dtype):
    import torch
    if dtype == torch.bfloat16:
        return FP8W_BF16
    if dtype == torch.float16:
        return FP8W_F16
    raise TypeError("activations must be bfloat16 or float16, got %s" % dtype)


def quantize(w, codes=None, scales=None, group=None):
    """W[N, K] (CUDA, contiguous; fp32, or bf16/fp16 widened exactly) ->
    (codes uint8 [N, K], scales fp32 [N]), or with group (32, 64 or 128; fp32
    weights) scales fp32 [N, K / group], one per run of `group` weights of a row."""
    import torch
    wdt = {torch.float32: FP8W_F32, torch.bfloat16: FP8W_BF16, torch.float16: FP8W_F16}.get(w.dtype)
    if wdt is None or not w.is_cuda or w.dim() != 2 or not w.is_contiguous():
        raise TypeError("w must be a contiguous 2-D float32, bfloat16 or float16 CUDA tensor")
    if wdt != FP8W_F32 and group is not None:
        raise TypeError("per-group quantisation takes float32 weights")
    n, k = w.shape
    if codes is None:
        codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    if scales is None:
        shape = (n,) if group is None else (n, k // group)
        scales = torch.empty(shape, dtype=torch.float32, device=w.device)
    if group is None:
        _check(lib().fp8w_quantize_ex(_ptr(w), wdt, n, k, _ptr(codes), _ptr(scales), _stream(w)))
    else:
        _check(lib().fp8w_quantize_grouped(_ptr(w), n, k, int(group), _ptr(codes), _ptr(scales), _stream(w)))
    return codes, scales


def quantize_mx(w, codes=None, scales=None):
    """W[N, K] fp32 (CUDA, contiguous, K % 32 == 0) -> (codes uint8 [N, K],
    scales uint8 [N, K / 32]): the MX-style form, one E8M0 byte (2^(b - 127))
    per 32 weights along K."""
    import torch
    if w.dtype != torch.float32 or not w.is_cuda or w.dim() != 2 or not w.is_contiguous():
        raise TypeError("w must be a contiguous 2-D float32 CUDA tensor")
    n, k = w.shape
    if codes is None:
        codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((n, k // 32), dtype=torch.uint8, device=w.device)
    _check(lib().fp8w_quantize_mx(_ptr(w), n, k, _ptr(codes), _ptr(scales), _stream(w)))
    return codes, scales


def dequantize(codes, scales, dtype=None, out=None):
    """W'[N, K] = e4m3(codes) * scales[:, None], rounded once to `dtype`
    (torch.float32, bfloat16 or float16; default bfloat16).  scales may also
    be per-group fp32 [N, K / group] or E8M0 uint8 [N, K / 32]."""
    import torch
    if dtype is None:
        dtype = out.dtype if out is not None else torch.bfloat16
    kind = {torch.float32: FP8W_F32, torch.bfloat16: FP8W_BF16, torch.float16: FP8W_F16}.get(dtype)
    if kind is None:
        raise TypeError("dequantize: dtype must be float32, bfloat16 or float16, got %s" % dtype)
    mx = scales.dim() == 2 and scales.dtype == torch.uint8
    for name, t, dt in (("codes", codes, torch.uint8), ("scales", scales, torch.uint8 if mx else torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError("%s must be a contiguous %s CUDA tensor" % (name, dt))
    n, k = codes.shape
    if out is None:
        out = torch.empty((n, k), dtype=dtype, device=codes.device)
    elif out.shape != (n, k) or out.dtype != dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [N, K] tensor of the requested dtype")
    if scales.dim() == 2:
        if scales.shape[0] != n or scales.shape[1] == 0 or k % scales.shape[1] or (mx and scales.shape[1] * 32 != k):
            raise ValueError("shape mismatch for per-group scales")
        if mx:
            _check(lib().fp8w_dequantize_mx(_ptr(codes), _ptr(scales), n, k, kind, _ptr(out), _stream(codes)))
        else:
            _check(lib().fp8w_dequantize_grouped(_ptr(codes), _ptr(scales), k // scales.shape[1], n, k, kind,
                                                 _ptr(out), _stream(codes)))
        return out
    _check(lib().fp8w_dequantize(_ptr(codes), _ptr(scales), n, k, kind, _ptr(out), _stream(codes)))
    return out


def linear(x, codes, scales, bias=None, out=None, kernel=KERNEL_AUTO, cluster=0, tiles=0,
           weights_ready=False):
    """y[M, N] = round(scale[n] * sum_k x[m, k] * e4m3(codes[n, k]) + bias[n]).

    kernel, and for the tensor-core kernel cluster (CTAs per thread-block
    cluster) with tiles (128-channel tiles a cluster shares), override the
    automatic launch choice, for tests and tuning (0, 0 = from the shape).
    weights_ready: every write to codes and scales has completed before this
    call (FP8W_FLAG_WEIGHTS_READY): the kernels stream the codes without
    waiting for the preceding kernel in the stream.  Per-row scales only."""
    import torch
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous 2-D CUDA tensor")
    # E8M0 scale bytes [N, K / 32] (the MX-style form) or fp32 scales
    mx = scales.dim() == 2 and scales.dtype == torch.uint8
    for name, t, dt in (("codes", codes, torch.uint8), ("scales", scales, torch.uint8 if mx else torch.float32),
                        ("bias", bias, torch.float32)):
        if t is not None and (t.dtype != dt or not t.is_cuda or not t.is_contiguous()):
            raise TypeError("%s must be a contiguous %s CUDA tensor" % (name, dt))
    m, k = x.shape
    n = codes.shape[0]
    if scales.dim() == 2:
        # per-group scales [N, K / group] (fp32), or E8M0 bytes [N, K / 32]
        if codes.dim() != 2 or codes.shape[1] != k or scales.shape[0] != n or k % scales.shape[1] or \
                (mx and scales.shape[1] * 32 != k) or (bias is not None and bias.numel() != n):
            raise ValueError("shape mismatch for per-group scales")
        if out is None:
            out = torch.empty((m, n), dtype=x.dtype, device=x.device)
        elif out.shape != (m, n) or out.dtype != x.dtype or not out.is_contiguous():
            raise ValueError("out must be a contiguous [M, N] tensor of x's dtype")
        if mx:
            _check(lib().fp8w_linear_mx(_ptr(x), _act(x.dtype), m, k, _ptr(codes), _ptr(scales), _ptr(bias), n,
                                        _ptr(out), _stream(x)))
        else:
            _check(lib().fp8w_linear_grouped(_ptr(x), _act(x.dtype), m, k, _ptr(codes), _ptr(scales),
                                             k // scales.shape[1], _ptr(bias), n, _ptr(out), _stream(x)))
        return out
    if codes.dim() != 2 or codes.shape[1] != k or scales.numel() != n or \
            (bias is not None and bias.numel() != n):
        raise ValueError("shape mismatch: x %s, codes %s, scales %s, bias %s" % (
            tuple(x.shape), tuple(codes.shape), tuple(scales.shape),
            None if bias is None else tuple(bias.shape)))
    if out is None:
        out = torch.empty((m, n), dtype=x.dtype, device=x.device)
    elif out.shape != (m, n) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] tensor of x's dtype")
    act = _act(x.dtype)
    L = lib()
    stream = _stream(x)
    if kernel == KERNEL_AUTO and cluster == 0 and not weights_ready:
        st = L.fp8w_linear(_ptr(x), act, m, k, _ptr(codes), _ptr(scales), _ptr(bias), n, _ptr(out), stream)
    else:
        cfg = LinearConfig(kernel, cluster, tiles, FLAG_WEIGHTS_READY if weights_ready else 0)
        st = L.fp8w_linear_ex(_ptr(x), act, m, k, _ptr(codes), _ptr(scales), _ptr(bias), n,
                              _ptr(out), ctypes.byref(cfg), stream)
    _check(st)
    return out


def quantize_act(x, codes=None, scales=None):
    """W8A8 activation quantisation: x[M, K] bf16/fp16 (CUDA, contiguous) ->
    (codes uint8 [M, K], scales fp32 [M]), the per-row rule on every token."""
    import torch
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous 2-D CUDA tensor")
    m, k = x.shape
    if codes is None:
        codes = torch.empty((m, k), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((m,), dtype=torch.float32, device=x.device)
    _check(lib().fp8w_quantize_act(_ptr(x), _act(x.dtype), m, k, _ptr(codes), _ptr(scales), _stream(x)))
    return codes, scales


def linear_w8a8(x_codes, x_scales, codes, scales, bias=None, out=None, out_dtype=None, weights_ready=False):
    """W8A8: y[M, N] = round(x_scales[m] * scales[n] * sum_k e4m3(x_codes[m, k]) e4m3(codes[n, k]) + bias[n]),
    out_dtype torch.bfloat16 (default) or torch.float16."""
    import torch
    for name, t, dt in (("x_codes", x_codes, torch.uint8), ("x_scales", x_scales, torch.float32),
                        ("codes", codes, torch.uint8), ("scales", scales, torch.float32),
                        ("bias", bias, torch.float32)):
        if t is not None and (t.dtype != dt or not t.is_cuda or not t.is_contiguous()):
            raise TypeError("%s must be a contiguous %s CUDA tensor" % (name, dt))
    m, k = x_codes.shape
    n = codes.shape[0]
    if codes.dim() != 2 or codes.shape[1] != k or x_scales.numel() != m or scales.numel() != n or \
            (bias is not None and bias.numel() != n):
        raise ValueError("shape mismatch for W8A8")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=codes.device)
    elif out.shape != (m, n) or out.dtype != out_dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] tensor of out_dtype")
    _check(lib().fp8w_linear_w8a8(_ptr(x_codes), _ptr(x_scales), m, k, _ptr(codes), _ptr(scales), _ptr(bias), n,
                                  _ptr(out), _act(out_dtype), FLAG_WEIGHTS_READY if weights_ready else 0,
                                  _stream(codes)))
    return out


def device_error():
    """Nonzero if a kernel gave up a bounded wait since the last call (syncs)."""
    return lib().fp8w_device_error()
