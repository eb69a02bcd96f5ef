"""The C-ABI library loads and exports every symbol include/fp8w.h declares,
and rejects bad arguments on the host before any CUDA call (no GPU needed:
every case below fails a host-side check first)."""
import ctypes
import os
import re

import pytest

import fp8_weight_only_gb300 as fw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "fp8w.h")).read()
    return sorted(set(re.findall(r"FP8W_API\s+[\w\s\*]+?\b(fp8w_\w+)\s*\(", txt)))


def test_header_declares_the_binding_symbols():
    assert _declared() == sorted(fw.SYMBOLS)


def test_library_exports_every_declared_symbol():
    L = fw.lib()
    for name in _declared():
        assert hasattr(L, name), name
    assert L.fp8w_abi_version() == fw.ABI_VERSION


def test_status_strings():
    L = fw.lib()
    for s in range(7):
        assert L.fp8w_status_string(s)
    assert L.fp8w_status_string(99) == b"unknown status"


A16 = ctypes.c_void_p(0x100000)        # 16-byte aligned fake device addresses
B16 = ctypes.c_void_p(0x200000)
C16 = ctypes.c_void_p(0x300000)
D16 = ctypes.c_void_p(0x400000)


# Every case below is refused on the host, before any launch: the pointers
# are fake device addresses.
def _lin(x=A16, act=1, m=1, k=64, codes=B16, scales=C16, bias=None, n=8, y=D16, cfg=None):
    L = fw.lib()
    if cfg is None:
        return L.fp8w_linear(x, act, m, k, codes, scales, bias, n, y, None)
    return L.fp8w_linear_ex(x, act, m, k, codes, scales, bias, n, y, ctypes.byref(cfg), None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1), (dict(codes=None), 1), (dict(scales=None), 1), (dict(y=None), 1),
    (dict(act=0), 4), (dict(act=3), 4),
    (dict(m=0), 2), (dict(n=0), 2), (dict(k=0), 2), (dict(k=8), 2), (dict(k=40), 2),
    (dict(k=65536 + 16), 2), (dict(m=-1), 2), (dict(n=2 ** 31), 2),
    (dict(x=ctypes.c_void_p(0x100008)), 3), (dict(codes=ctypes.c_void_p(0x200004)), 3),
    (dict(scales=ctypes.c_void_p(0x300002)), 3), (dict(bias=ctypes.c_void_p(0x500001)), 3),
    (dict(y=ctypes.c_void_p(0x400001)), 3),
])
def test_linear_rejects_bad_arguments(kw, status):
    assert _lin(**kw) == status


def _cfg(kernel=fw.KERNEL_SKINNY, cluster=0, tiles=0, flags=0, reserved=0):
    c = fw.LinearConfig(kernel, cluster, tiles, flags)
    c.reserved[2] = reserved
    return c


@pytest.mark.parametrize("cfg", [
    _cfg(fw.KERNEL_GEMV),                      # gemv needs m == 1 (m = 2 below)
    _cfg(7), _cfg(-1),                         # unknown kernel
    _cfg(cluster=-3, tiles=1), _cfg(cluster=2, tiles=-1),
    _cfg(cluster=2), _cfg(tiles=3),            # cluster and tiles come together
    _cfg(cluster=17, tiles=1),                 # beyond the largest cluster size
    _cfg(cluster=4, tiles=1),                  # more ranks than k-blocks (k = 256: two)
    _cfg(fw.KERNEL_PREFILL, 2, 1),             # only the tensor-core kernel takes a shape
    _cfg(flags=2), _cfg(reserved=1),           # unknown flag, reserved field
])
def test_linear_rejects_bad_config(cfg):
    assert _lin(m=2, k=256, cfg=cfg) == 6


def test_gemv_rejects_a_cluster_shape():
    assert _lin(m=1, k=256, cfg=_cfg(fw.KERNEL_GEMV, 2, 1)) == 6


def test_tensor_core_kernel_beyond_32_tokens_shares_one_tile_at_most():
    # 64-token launches hold one accumulator per MMA warp
    assert _lin(m=40, k=1024, cfg=_cfg(cluster=2, tiles=3)) == 6


def test_gemv_rejects_rows_longer_than_it_stages():
    # x of a GEMV row lives in shared memory: k <= 32768
    assert _lin(m=1, k=32768 + 16, cfg=fw.LinearConfig(fw.KERNEL_GEMV)) == 6


@pytest.mark.parametrize("args,status", [
    ((None, 4, 64, B16, C16), 1), ((A16, 4, 64, None, C16), 1), ((A16, 4, 64, B16, None), 1),
    ((A16, 0, 64, B16, C16), 2), ((A16, 4, 24, B16, C16), 2), ((A16, 4, 0, B16, C16), 2),
    ((ctypes.c_void_p(0x100004), 4, 64, B16, C16), 3),
    ((A16, 4, 64, ctypes.c_void_p(0x200008), C16), 3),
    ((A16, 4, 64, B16, ctypes.c_void_p(0x300001)), 3),
])
def test_quantize_rejects_bad_arguments(args, status):
    assert fw.lib().fp8w_quantize(*args, None) == status


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fw, "_lib", None)
    monkeypatch.setattr(fw, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(fw.Fp8wError):
        fw.lib()


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1), (dict(y=None), 1), (dict(act=3), 4), (dict(m=0), 2), (dict(k=40), 2),
    (dict(codes=ctypes.c_void_p(0x200004)), 3),
])
def test_noalloc_entry_rejects_bad_arguments_on_the_host(kw, status):
    a = dict(x=A16, act=1, m=2, k=64, codes=B16, scales=C16, bias=None, n=8, y=D16)
    a.update(kw)
    L = fw.lib()
    assert L.fp8w_linear_noalloc(a["x"], a["act"], a["m"], a["k"], a["codes"], a["scales"], a["bias"],
                                 a["n"], a["y"], None) == status


@pytest.mark.parametrize("args,status", [
    ((None, C16, 4, 64, 1, D16), 1), ((B16, None, 4, 64, 1, D16), 1), ((B16, C16, 4, 64, 1, None), 1),
    ((B16, C16, 0, 64, 1, D16), 2), ((B16, C16, 4, 24, 1, D16), 2), ((B16, C16, 4, 65536 + 16, 1, D16), 2),
    ((B16, C16, 4, 64, 0, D16), 4), ((B16, C16, 4, 64, 7, D16), 4),
    ((ctypes.c_void_p(0x200004), C16, 4, 64, 1, D16), 3), ((B16, ctypes.c_void_p(0x300002), 4, 64, 1, D16), 3),
    ((B16, C16, 4, 64, 3, ctypes.c_void_p(0x400008)), 3),
])
def test_dequantize_rejects_bad_arguments(args, status):
    assert fw.lib().fp8w_dequantize(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, 4, 128, 32, B16, C16), 1), ((A16, 4, 128, 32, None, C16), 1),
    ((A16, 4, 128, 48, B16, C16), 2), ((A16, 4, 128, 256, B16, C16), 2), ((A16, 4, 96, 64, B16, C16), 2),
    ((A16, 0, 128, 32, B16, C16), 2), ((ctypes.c_void_p(0x100004), 4, 128, 32, B16, C16), 3),
])
def test_quantize_grouped_rejects_bad_arguments(args, status):
    assert fw.lib().fp8w_quantize_grouped(*args, None) == status


def _lin_g(m=1, k=512, group=32, scales=C16):
    return fw.lib().fp8w_linear_grouped(A16, 1, m, k, B16, scales, group, None, 8, D16, None)


@pytest.mark.parametrize("kw,status", [
    (dict(group=16), 2), (dict(group=96), 2),
    (dict(k=512 + 16, group=32), 2),     # k % group != 0
    (dict(k=1024 + 64, group=128), 2),
    (dict(m=0), 2), (dict(k=65536 + 128, group=128), 2),   # beyond FP8W_MAX_K
    (dict(scales=ctypes.c_void_p(0x300004)), 3),   # scales: 16-byte aligned (the GEMV bulk-copies them)
    (dict(m=40, scales=ctypes.c_void_p(0x300008)), 3),
])
def test_linear_grouped_rejects_bad_arguments(kw, status):
    # every case is refused on the host (any m is accepted now: the GEMV at
    # m == 1, the tensor-core kernels' per-group form otherwise)
    assert _lin_g(**kw) == status


@pytest.mark.parametrize("args,status", [
    ((None, 4, 128, B16, C16), 1), ((A16, 4, 128, None, C16), 1), ((A16, 4, 128, B16, None), 1),
    ((A16, 4, 48, B16, C16), 2), ((A16, 0, 128, B16, C16), 2), ((A16, 4, 65536 + 32, B16, C16), 2),
    ((ctypes.c_void_p(0x100004), 4, 128, B16, C16), 3), ((A16, 4, 128, ctypes.c_void_p(0x200008), C16), 3),
])
def test_quantize_mx_rejects_bad_arguments(args, status):
    assert fw.lib().fp8w_quantize_mx(*args, None) == status


def test_quantize_mx_takes_scale_bytes_at_any_alignment():
    # a host check only: a misaligned scale pointer passes, a bad k still fails
    assert fw.lib().fp8w_quantize_mx(A16, 4, 48, B16, ctypes.c_void_p(0x300001), None) == 2


@pytest.mark.parametrize("kw,status", [
    (dict(scales=None), 1), (dict(x=None), 1),
    (dict(k=256 + 64), 2), (dict(k=1024 + 16), 2),   # k % 128 != 0
    (dict(k=65536 + 128), 2),                  # beyond FP8W_MAX_K
    (dict(act=3), 4),
    (dict(scales=ctypes.c_void_p(0x300008)), 3),   # scale bytes: 16-byte aligned
    (dict(m=2, act=2, scales=ctypes.c_void_p(0x300001)), 3),   # fp16 beyond one token: the per-group form
])
def test_linear_mx_rejects_bad_arguments(kw, status):
    a = dict(x=A16, act=1, m=1, k=1024, codes=B16, scales=C16, bias=None, n=8, y=D16)
    a.update(kw)
    assert fw.lib().fp8w_linear_mx(a["x"], a["act"], a["m"], a["k"], a["codes"], a["scales"], a["bias"],
                                   a["n"], a["y"], None) == status


@pytest.mark.parametrize("args,status", [
    ((None, 1, 4, 64, B16, C16), 1), ((A16, 1, 4, 64, None, C16), 1), ((A16, 2, 4, 64, B16, None), 1),
    ((A16, 0, 4, 64, B16, C16), 4), ((A16, 5, 4, 64, B16, C16), 4),
    ((A16, 1, 0, 64, B16, C16), 2), ((A16, 2, 4, 24, B16, C16), 2), ((A16, 1, 4, 65536 + 16, B16, C16), 2),
    ((ctypes.c_void_p(0x100008), 1, 4, 64, B16, C16), 3), ((A16, 2, 4, 64, ctypes.c_void_p(0x200004), C16), 3),
    ((A16, 3, 4, 24, B16, C16), 2),              # FP8W_F32: fp8w_quantize's checks
])
def test_quantize_ex_rejects_bad_arguments(args, status):
    assert fw.lib().fp8w_quantize_ex(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, C16, 32, 4, 64, 1, D16), 1), ((B16, None, 32, 4, 64, 1, D16), 1), ((B16, C16, 32, 4, 64, 1, None), 1),
    ((B16, C16, 48, 4, 96, 1, D16), 2), ((B16, C16, 128, 4, 192, 1, D16), 2), ((B16, C16, 32, 0, 64, 1, D16), 2),
    ((B16, C16, 32, 4, 64, 7, D16), 4),
    ((ctypes.c_void_p(0x200004), C16, 32, 4, 64, 1, D16), 3), ((B16, ctypes.c_void_p(0x300002), 32, 4, 64, 1, D16), 3),
    ((B16, C16, 32, 4, 64, 3, ctypes.c_void_p(0x400008)), 3),
])
def test_dequantize_grouped_rejects_bad_arguments(args, status):
    assert fw.lib().fp8w_dequantize_grouped(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, C16, 4, 64, 1, D16), 1), ((B16, None, 4, 64, 1, D16), 1),
    ((B16, C16, 4, 48, 1, D16), 2), ((B16, C16, 4, 64, 0, D16), 4),
    ((ctypes.c_void_p(0x200004), C16, 4, 64, 1, D16), 3),
    ((B16, ctypes.c_void_p(0x300001), 4, 48, 1, D16), 2),   # scale bytes: any alignment, the shape still checked
])
def test_dequantize_mx_rejects_bad_arguments(args, status):
    assert fw.lib().fp8w_dequantize_mx(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((A16, 0, 2, 64, B16, C16), 4),            # fp32 activations: bf16 or fp16 only
    ((A16, 3, 2, 64, B16, C16), 4),
    ((None, 1, 2, 64, B16, C16), 1), ((A16, 1, 2, 64, None, C16), 1), ((A16, 2, 2, 64, B16, None), 1),
    ((A16, 1, 0, 64, B16, C16), 2), ((A16, 1, 2, 24, B16, C16), 2), ((A16, 2, 2, 65536 + 16, B16, C16), 2),
    ((ctypes.c_void_p(0x100008), 1, 2, 64, B16, C16), 3),
    ((A16, 1, 2, 64, ctypes.c_void_p(0x200004), C16), 3),
    ((A16, 1, 2, 64, B16, ctypes.c_void_p(0x300002)), 3),
])
def test_quantize_act_rejects_bad_arguments(args, status):
    assert fw.lib().fp8w_quantize_act(*args, None) == status


E16 = ctypes.c_void_p(0x500000)


def _w8a8(xc=A16, xs=B16, m=2, k=64, wc=C16, ws=D16, bias=None, n=8, y=E16, out=1, flags=0):
    return fw.lib().fp8w_linear_w8a8(xc, xs, m, k, wc, ws, bias, n, y, out, flags, None)


@pytest.mark.parametrize("kw,status", [
    (dict(xc=None), 1), (dict(xs=None), 1), (dict(wc=None), 1), (dict(ws=None), 1), (dict(y=None), 1),
    (dict(out=0), 4), (dict(out=3), 4),
    (dict(m=0), 2), (dict(n=0), 2), (dict(k=8), 2), (dict(k=40), 2), (dict(k=65536 + 16), 2),
    (dict(m=-1), 2), (dict(n=2 ** 31), 2),
    (dict(xc=ctypes.c_void_p(0x100008)), 3), (dict(wc=ctypes.c_void_p(0x300004)), 3),
    (dict(xs=ctypes.c_void_p(0x200002)), 3), (dict(ws=ctypes.c_void_p(0x400001)), 3),
    (dict(bias=ctypes.c_void_p(0x600002)), 3), (dict(y=ctypes.c_void_p(0x500001)), 3),
    (dict(flags=2), 6), (dict(flags=-1), 6),
])
def test_linear_w8a8_rejects_bad_arguments(kw, status):
    assert _w8a8(**kw) == status
