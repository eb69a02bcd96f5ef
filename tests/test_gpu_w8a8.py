"""GPU parity of the W8A8 path (page "tensormux Write an FP8 kernel":
per-token activation scales, per-channel weight scales, both amax / 448,
e4m3 x e4m3 GEMM, accumulator times both scales) against the oracle.

Activation codes and scales must be bit-exact; outputs within the stated
tolerance (rel_l2 <= 2e-3, per-row cosine >= 0.9999) of the oracle's fp64
sum rounded once, and bit-identical where the sum is exact in fp32.  Output
buffers are poisoned and surrounded by canaries.
"""
import numpy as np
import pytest

import oracle
import synthetic
from tests.parity import assert_parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import fp8_weight_only_gb300 as fw  # noqa: E402

DEV = torch.device("cuda:0")
CANARY = 64
POISON16 = 0x7FC1


def oracle_w8a8(qx, sx, act, qw, sw, bias):
    """The oracle over channel blocks on all host cores (each block is one
    oracle call; ctypes releases the interpreter lock), same sums."""
    import concurrent.futures as cf
    n = qw.shape[0]
    parts = max(1, min(oracle.host_cores(), n // 256))
    if parts == 1:
        return oracle.linear_w8a8(qx, sx, act, qw, sw, bias)
    edges = [n * i // parts for i in range(parts + 1)]
    with cf.ThreadPoolExecutor(parts) as ex:
        outs = list(ex.map(lambda i: oracle.linear_w8a8(
            qx, sx, act, qw[edges[i]:edges[i + 1]], sw[edges[i]:edges[i + 1]],
            None if bias is None else bias[edges[i]:edges[i + 1]]), range(parts)))
    return np.concatenate(outs, axis=1)


def _dt(act):
    return torch.bfloat16 if act == oracle.ACT_BF16 else torch.float16


def _x_bits(seed, m, k, act):
    return synthetic.act_normal_bf16(seed, m, k) if act == oracle.ACT_BF16 else synthetic.act_uniform_f16(seed, m, k)


def gpu_quantize_act(x_bits, act):
    m, k = x_bits.shape
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(DEV).view(_dt(act))
    cbuf = torch.full((m * k + 2 * CANARY,), 0xA5, dtype=torch.uint8, device=DEV)
    sbuf = torch.full((m + 2 * CANARY,), -7.0, dtype=torch.float32, device=DEV)
    codes = cbuf[CANARY:CANARY + m * k].view(m, k)
    scales = sbuf[CANARY:CANARY + m]
    fw.quantize_act(x, codes, scales)
    torch.cuda.synchronize()
    assert bool((cbuf[:CANARY] == 0xA5).all()) and bool((cbuf[CANARY + m * k:] == 0xA5).all())
    assert bool((sbuf[:CANARY] == -7.0).all()) and bool((sbuf[CANARY + m:] == -7.0).all())
    return codes, scales


def gpu_w8a8(qx, sx, qw, sw, bias, act, weights_ready=False):
    """qx, sx, qw, sw: device tensors or numpy arrays; returns y bits [m, n]."""
    def dev(a):
        return a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    qx, sx, qw, sw = dev(qx), dev(sx), dev(qw), dev(sw)
    b = None if bias is None else dev(bias)
    m, n = qx.shape[0], qw.shape[0]
    ybuf = torch.empty(m * n + 2 * CANARY, dtype=_dt(act), device=DEV)
    ybuf.view(torch.int16).fill_(int(np.uint16(POISON16).view(np.int16)))
    y = ybuf[CANARY:CANARY + m * n].view(m, n)
    fw.linear_w8a8(qx, sx, qw, sw, b, out=y, weights_ready=weights_ready)
    torch.cuda.synchronize()
    p = int(np.uint16(POISON16).view(np.int16))
    assert bool((ybuf[:CANARY].view(torch.int16) == p).all()), "canary before output overwritten"
    assert bool((ybuf[CANARY + m * n:].view(torch.int16) == p).all()), "canary after output overwritten"
    assert fw.device_error() == 0
    return y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(m, n)


# ----------------------------------------------------- activation codes --

@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("m,k", [(1, 16), (3, 1040), (32, 4096), (130, 256), (17, 14336)])
def test_activation_codes_and_scales_bit_exact(m, k, act):
    xb = _x_bits(100 + m, m, k, act)
    xb[0, :3] = 0   # exact zeros keep their codes
    codes, scales = gpu_quantize_act(xb, act)
    rc, rs = oracle.quantize_act(xb, act)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_activation_zero_row_takes_scale_one():
    xb = _x_bits(7, 4, 64, oracle.ACT_BF16)
    xb[2] = 0
    codes, scales = gpu_quantize_act(xb, oracle.ACT_BF16)
    assert scales.cpu().numpy()[2] == 1.0 and int(codes[2].abs().sum()) == 0


# ---------------------------------------------------------------- linear --

def _case(seed, m, n, k, act, with_bias=True):
    xb = _x_bits(seed, m, k, act)
    w = synthetic.weight_normal(seed + 1, n, k, 0.02)
    bias = synthetic.bias_normal(seed + 2, n) if with_bias else None
    qx, sx = oracle.quantize_act(xb, act)
    qw, sw = oracle.quantize(w)
    return qx, sx, qw, sw, bias


# (m, n, k): one token tile and few channel tiles (cluster split over k),
# ragged n and k, every token-tile width (16, 32, 64, 128, 256) with a
# ragged tail, and persistent CTAs with several tiles each
W8A8_SHAPES = [(1, 1, 16), (1, 200, 1040), (3, 1000, 144), (16, 128, 4096), (17, 300, 1040), (32, 1024, 4096),
               (33, 640, 272), (64, 129, 528), (65, 700, 384), (128, 2048, 256), (200, 1500, 160),
               (520, 5000, 144), (300, 20000, 128)]


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("m,n,k", W8A8_SHAPES)
def test_w8a8_parity(m, n, k, act):
    qx, sx, qw, sw, bias = _case(2000 + m + n, m, n, k, act)
    y = gpu_w8a8(qx, sx, qw, sw, bias, act)
    ref = oracle_w8a8(qx, sx, act, qw, sw, bias)
    assert_parity(y, ref, act, "w8a8 %dx%dx%d" % (m, n, k))


@pytest.mark.parametrize("m,n,k", [(8, 1000, 4096), (130, 600, 512)])
def test_w8a8_weights_ready_flag_same_result(m, n, k):
    qx, sx, qw, sw, bias = _case(31 + m, m, n, k, oracle.ACT_BF16)
    a = gpu_w8a8(qx, sx, qw, sw, bias, oracle.ACT_BF16)
    b = gpu_w8a8(qx, sx, qw, sw, bias, oracle.ACT_BF16, weights_ready=True)
    assert np.array_equal(a, b)


def test_w8a8_bias_none_equals_zero_bias_and_is_deterministic():
    qx, sx, qw, sw, _ = _case(41, 24, 900, 1024, oracle.ACT_BF16)
    a = gpu_w8a8(qx, sx, qw, sw, None, oracle.ACT_BF16)
    b = gpu_w8a8(qx, sx, qw, sw, np.zeros(900, np.float32), oracle.ACT_BF16)
    c = gpu_w8a8(qx, sx, qw, sw, None, oracle.ACT_BF16)
    assert np.array_equal(a, b) and np.array_equal(a, c)


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("m,n,k", [(1, 300, 1040), (9, 130, 4096), (100, 257, 528), (300, 1200, 256)])
def test_w8a8_exact_cases_bit_identical(m, n, k, act):
    """Codes whose values are small multiples of 1/4 (and one 448 a row, so
    the scales are powers of two): every partial sum is exact in fp32 in any
    order, so the output must equal the oracle's bit for bit."""
    rng = np.random.default_rng(61 + m)
    t = oracle.e4m3_decode_table()
    small = [b for b in range(0x7F) if t[b] in (0.0, 0.25, 0.5, 1.0, 1.5, 2.0)]
    qw = rng.choice(small, size=(n, k)).astype(np.uint8) | (rng.integers(0, 2, (n, k)) * 0x80).astype(np.uint8)
    qx = rng.choice(small, size=(m, k)).astype(np.uint8) | (rng.integers(0, 2, (m, k)) * 0x80).astype(np.uint8)
    qw[:, 3] = 0x7E
    qx[:, 5] = 0x7E
    sw = (2.0 ** rng.integers(-12, -4, n)).astype(np.float32)
    sx = (2.0 ** rng.integers(-8, 0, m)).astype(np.float32)
    bias = (rng.integers(-64, 64, n) * 2.0 ** -6).astype(np.float32)
    y = gpu_w8a8(qx, sx, qw, sw, bias, act)
    ref = oracle.linear_w8a8(qx, sx, act, qw, sw, bias)
    assert np.array_equal(y, ref)


def test_w8a8_end_to_end_from_activations():
    """quantize_act on the device feeds linear_w8a8 directly."""
    act = oracle.ACT_BF16
    m, n, k = 12, 2000, 1024
    xb = _x_bits(77, m, k, act)
    w = synthetic.weight_normal(78, n, k, 0.02)
    bias = synthetic.bias_normal(79, n)
    wd = torch.from_numpy(w).to(DEV)
    qw, sw = fw.quantize(wd)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    qx, sx = fw.quantize_act(x)
    y = fw.linear_w8a8(qx, sx, qw, sw, torch.from_numpy(bias).to(DEV))
    torch.cuda.synchronize()
    rqx, rsx = oracle.quantize_act(xb, act)
    rqw, rsw = oracle.quantize(w)
    ref = oracle.linear_w8a8(rqx, rsx, act, rqw, rsw, bias)
    assert_parity(y.view(torch.int16).cpu().numpy().view(np.uint16), ref, act, "w8a8 end to end")


@pytest.mark.parametrize("m", synthetic.DECODE_STACK_M)
def test_w8a8_full_gate_every_channel(m):
    """The decode-stack gate weight [14336 x 4096] at M = 1, 8 and 32, every
    output compared (the oracle on all host cores)."""
    c = synthetic.case("decode_stack", m, "gate")
    act = oracle.ACT_BF16
    qx, sx = oracle.quantize_act(c["x"], act)
    qw, sw = oracle.quantize(c["w"])
    y = gpu_w8a8(qx, sx, qw, sw, c["bias"], act, weights_ready=True)
    ref = oracle_w8a8(qx, sx, act, qw, sw, c["bias"])
    assert_parity(y, ref, act, "w8a8 gate m=%d" % m)


def test_w8a8_host_checks():
    L = fw.lib()
    import ctypes
    P = ctypes.c_void_p
    buf = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    p = P(buf.data_ptr())
    s = P(torch.cuda.current_stream().cuda_stream)
    assert L.fp8w_linear_w8a8(None, p, 1, 16, p, p, None, 1, p, fw.FP8W_BF16, 0, s) == 1
    assert L.fp8w_linear_w8a8(p, p, 1, 16, p, p, None, 1, p, fw.FP8W_F32, 0, s) == 4
    assert L.fp8w_linear_w8a8(p, p, 1, 24, p, p, None, 1, p, fw.FP8W_BF16, 0, s) == 2
    assert L.fp8w_linear_w8a8(p, p, 0, 16, p, p, None, 1, p, fw.FP8W_BF16, 0, s) == 2
    assert L.fp8w_linear_w8a8(P(buf.data_ptr() + 8), p, 1, 16, p, p, None, 1, p, fw.FP8W_BF16, 0, s) == 3
    assert L.fp8w_linear_w8a8(p, p, 1, 16, p, p, None, 1, p, fw.FP8W_BF16, 2, s) == 6
    assert L.fp8w_quantize_act(p, fw.FP8W_F32, 1, 16, p, p, s) == 4
