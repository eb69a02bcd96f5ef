"""GPU parity of the per-group forms beyond one token: fp32 scales per run of
g = 32, 64 or 128 codes of a row, and E8M0 bytes with fp16 activations, on
the tensor-core kernels, against the oracle's per-group linear layer
(y = round(sum_j scale[n, j] * sum_{k in group j} x[m, k] e4m3(q[n, k]) + bias[n])).

Shapes span whole tiles, clusters that split a tile, ragged n, k that is a
multiple of the group but not of the 128-code unit, token counts across the
16/32-token launches and their 32-row slabs, and the prefill GEMM beyond 64
tokens.  Output buffers are poisoned and guarded by canaries.
"""
import numpy as np
import pytest

import oracle
import synthetic
from tests.parity import assert_parity, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import fp8_weight_only_gb300 as fw  # noqa: E402

DEV = torch.device("cuda:0")
CANARY = 64
POISON16 = 0x7FC1


def _dt(act):
    return torch.bfloat16 if act == oracle.ACT_BF16 else torch.float16


def _run(x_bits, act, codes, scales, bias):
    """fw.linear through the C ABI into a poisoned, canary-guarded buffer."""
    m, k = x_bits.shape
    n = codes.shape[0]
    dt = _dt(act)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV).view(dt)
    buf = torch.empty(m * n + 2 * CANARY, dtype=dt, device=DEV)
    buf.view(torch.int16).fill_(int(np.uint16(POISON16).view(np.int16)))
    y = buf[CANARY:CANARY + m * n].view(m, n)
    b = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias)).to(DEV)
    fw.linear(x, torch.from_numpy(np.ascontiguousarray(codes)).to(DEV),
              torch.from_numpy(np.ascontiguousarray(scales)).to(DEV), b, out=y)
    torch.cuda.synchronize()
    guard = buf.view(torch.int16).cpu().numpy()
    v = int(np.uint16(POISON16).view(np.int16))
    assert (guard[:CANARY] == v).all() and (guard[CANARY + m * n:] == v).all(), "canary overwritten"
    assert fw.device_error() == 0
    return y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(m, n)


def _grouped_case(seed, m, n, k, group, act):
    c = synthetic.random_case(seed, m, n, k, act=act, with_bias=(n % 2 == 1))
    w = c["w"].copy()
    w[:, ::97] *= 40.0                     # outliers that per-group scales contain
    codes, scales = oracle.quantize_grouped(w, group)
    return c, codes, scales


GROUPED_SHAPES = [  # (m, n, k, group)
    (2, 300, 4096, 32), (8, 4096, 4096, 128), (8, 4096, 4096, 32), (16, 1000, 1024, 64),
    (17, 257, 1056, 32),      # k % 128 == 32: the last unit's later groups lie past k
    (32, 14336, 4096, 128),   # whole tiles, one a CTA
    (32, 640, 14336, 64),     # a cluster splits each tile
    (5, 130, 4160, 64), (31, 129, 256, 128), (9, 64, 128, 32),
    (33, 300, 1056, 32),      # two 32-row slabs
    (1, 300, 1056, 32),       # one token, k % (4 g) != 0: the tensor-core kernel, not the GEMV
    (64, 1000, 4096, 128),
    (70, 260, 512, 64), (129, 300, 2048, 32), (300, 1000, 4096, 128), (513, 257, 1024, 64),  # beyond 64 tokens
]


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("m,n,k,group", GROUPED_SHAPES)
def test_linear_grouped_parity_beyond_one_token(m, n, k, group, act):
    c, codes, scales = _grouped_case(1300 + m + n + k + group + act, m, n, k, group, act)
    got = _run(c["x"], act, codes, scales, c["bias"])
    ref = oracle.linear_grouped(c["x"], act, codes, scales, group, c["bias"], threads=oracle.host_cores())
    assert_parity(got, ref, act, (m, n, k, group))


@pytest.mark.parametrize("m", [8, 32])
def test_linear_grouped_gate_every_output(m):
    """The 14336 x 4096 gate matrix, g = 128, every output against the oracle."""
    n, k, group = 14336, 4096, 128
    c, codes, scales = _grouped_case(71 + m, m, n, k, group, oracle.ACT_BF16)
    got = _run(c["x"], oracle.ACT_BF16, codes, scales, c["bias"])
    ref = oracle.linear_grouped(c["x"], oracle.ACT_BF16, codes, scales, group, c["bias"],
                                threads=oracle.host_cores())
    assert_parity(got, ref, oracle.ACT_BF16, ("gate", m))


@pytest.mark.parametrize("group", [64, 128])
def test_linear_grouped_prefill_gate_repeatable(group):
    """The prefill GEMM's per-group form on the whole 14336 x 4096 gate matrix
    (130 tokens: two token tiles, every SM walking several weight tiles):
    three launches give the same bits, and every output is within the
    tolerance of the oracle."""
    m, n, k = 130, 14336, 4096
    c, codes, scales = _grouped_case(97 + group, m, n, k, group, oracle.ACT_BF16)
    runs = [_run(c["x"], oracle.ACT_BF16, codes, scales, c["bias"]) for _ in range(3)]
    assert np.array_equal(runs[0], runs[1]) and np.array_equal(runs[0], runs[2])
    ref = oracle.linear_grouped(c["x"], oracle.ACT_BF16, codes, scales, group, c["bias"],
                                threads=oracle.host_cores())
    assert_parity(runs[0], ref, oracle.ACT_BF16, ("gate prefill", group))


def test_linear_grouped_one_group_scale_equals_the_row_scale():
    """Every group of a row with the row's scale: the per-group product equals
    the per-channel one within the tolerance (the scale is applied per group
    instead of once, so the fp32 sums are rounded in another order)."""
    m, n, k = 16, 1000, 4096
    c = synthetic.random_case(19, m, n, k, act=oracle.ACT_BF16, with_bias=True)
    codes, scales = oracle.quantize(c["w"])
    gs = np.repeat(scales[:, None], k // 64, axis=1).astype(np.float32)
    yg = _run(c["x"], oracle.ACT_BF16, codes, gs, c["bias"])
    y1 = _run(c["x"], oracle.ACT_BF16, codes, scales, c["bias"])
    cmp = compare(yg, y1, oracle.ACT_BF16)
    assert cmp["rel_l2"] <= 1e-3 and cmp["bit_equal"] >= 0.9, cmp


def test_linear_grouped_power_of_two_scales_are_exact_per_group():
    """Codes whose group sums are exact in fp32 (few small integers) with
    power-of-two group scales: every product and partial sum is exact, so the
    result equals the oracle's bit for bit."""
    m, n, k, group = 24, 384, 1024, 32
    rng = np.random.default_rng(5)
    # codes of the integers -4..4 (e4m3 codes of small integers are exact)
    ints = rng.integers(-4, 5, size=(n, k))
    enc = {v: int(oracle.e4m3_encode(np.float32(v))[0]) for v in range(-4, 5)}
    codes = np.vectorize(enc.get)(ints).astype(np.uint8)
    scales = (2.0 ** rng.integers(-6, 4, size=(n, k // group))).astype(np.float32)
    xi = rng.integers(-3, 4, size=(m, k)).astype(np.float32)
    x_bits = (xi.view(np.uint32) >> 16).astype(np.uint16)
    bias = rng.integers(-8, 9, size=n).astype(np.float32)
    got = _run(x_bits, oracle.ACT_BF16, codes, scales, bias)
    ref = oracle.linear_grouped(x_bits, oracle.ACT_BF16, codes, scales, group, bias, threads=oracle.host_cores())
    assert np.array_equal(got, ref)


MX_F16_SHAPES = [(2, 300, 4096), (8, 4096, 4096), (17, 257, 640), (32, 14336, 1024), (48, 1000, 1024),
                 (64, 640, 14336), (100, 300, 1024)]


@pytest.mark.parametrize("m,n,k", MX_F16_SHAPES)
def test_linear_mx_fp16_beyond_one_token(m, n, k):
    """E8M0 scales with fp16 activations: the per-group form with each byte
    decoded to its fp32 power of two."""
    c = synthetic.random_case(500 + m + n + k, m, n, k, act=oracle.ACT_F16, with_bias=(n % 2 == 1))
    w = c["w"].copy()
    w[:, ::97] *= 40.0
    codes, e8 = oracle.quantize_mx(w)
    got = _run(c["x"], oracle.ACT_F16, codes, e8, c["bias"])
    ref = oracle.linear_mx(c["x"], oracle.ACT_F16, codes, e8, c["bias"], threads=oracle.host_cores())
    assert_parity(got, ref, oracle.ACT_F16, (m, n, k, "mx f16"))


def test_linear_mx_fp16_equals_grouped_on_decoded_scales():
    """The bytes decode to exact fp32 powers of two, so the E8M0 form and the
    fp32 per-group form at g = 32 run the same arithmetic: bit-equal, the
    2^-127 and 2^127 ends and the NaN byte included (its row NaN)."""
    m, n, k = 12, 700, 2048
    c = synthetic.random_case(6, m, n, k, act=oracle.ACT_F16, with_bias=True)
    codes, e8 = oracle.quantize_mx(c["w"])
    e8[3, :4] = [0, 1, 254, 253]
    e8[5, 7] = 255
    dec = np.vectorize(oracle.e8m0_decode)(e8).astype(np.float32)
    y_mx = _run(c["x"], oracle.ACT_F16, codes, e8, c["bias"])
    y_g = _run(c["x"], oracle.ACT_F16, codes, dec, c["bias"])
    assert np.array_equal(y_mx, y_g)
    nan = (y_mx & 0x7FFF) > 0x7C00
    assert nan[:, 5].all()
