"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Codes and scales must be bit-exact; outputs within the stated tolerance
(rel_l2 <= 2e-3, per-row cosine >= 0.9999), and bit-identical where the
result is exact in fp32 regardless of summation order.  Output buffers are
poisoned before every call and surrounded by canary bytes, so a skipped or
out-of-bounds write fails.
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
CANARY = 64          # elements of canary on each side of an output
POISON16 = 0x7FC1    # a NaN pattern in bf16 (and a NaN in fp16)


def _dt(act):
    return torch.bfloat16 if act == oracle.ACT_BF16 else torch.float16


def _guarded(n_elems, dtype, fill):
    """A device buffer with canaries around a poisoned payload."""
    buf = torch.empty(n_elems + 2 * CANARY, dtype=dtype, device=DEV)
    buf.view(torch.uint8 if dtype == torch.uint8 else torch.int16)
    if dtype == torch.uint8:
        buf.fill_(0xA5)
    else:
        buf.view(torch.int16).fill_(np.int16(np.uint16(fill).view(np.int16)))
    return buf, buf[CANARY:CANARY + n_elems]


def _check_canaries(buf, n_elems, fill):
    head = buf[:CANARY]
    tail = buf[CANARY + n_elems:]
    if buf.dtype == torch.uint8:
        assert bool((head == 0xA5).all()) and bool((tail == 0xA5).all()), "canary overwritten"
    else:
        v = np.int16(np.uint16(fill).view(np.int16))
        assert bool((head.view(torch.int16) == int(v)).all()), "canary before output overwritten"
        assert bool((tail.view(torch.int16) == int(v)).all()), "canary after output overwritten"


def gpu_quantize(w_np):
    n, k = w_np.shape
    w = torch.from_numpy(w_np).to(DEV)
    cbuf, codes = _guarded(n * k, torch.uint8, 0)
    codes = codes.view(n, k)
    sbuf = torch.full((n + 2 * CANARY,), -7.0, dtype=torch.float32, device=DEV)
    scales = sbuf[CANARY:CANARY + n]
    fw.quantize(w, codes, scales)
    torch.cuda.synchronize()
    _check_canaries(cbuf, n * k, 0)
    assert bool((sbuf[:CANARY] == -7.0).all()) and bool((sbuf[CANARY + n:] == -7.0).all())
    return codes.cpu().numpy(), scales.cpu().numpy()


def gpu_linear(x_bits, act, codes, scales, bias, kernel=fw.KERNEL_AUTO, cluster=0, tiles=0, weights_ready=False):
    m, k = x_bits.shape
    n = codes.shape[0]
    dt = _dt(act)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV).view(dt)
    c = torch.from_numpy(np.ascontiguousarray(codes)).to(DEV)
    s = torch.from_numpy(np.ascontiguousarray(scales)).to(DEV)
    b = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias)).to(DEV)
    ybuf, y = _guarded(m * n, dt, POISON16)
    fw.linear(x, c, s, b, out=y.view(m, n), kernel=kernel, cluster=cluster, tiles=tiles, weights_ready=weights_ready)
    torch.cuda.synchronize()
    _check_canaries(ybuf, m * n, POISON16)
    assert fw.device_error() == 0
    return y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(m, n)


# --------------------------------------------------------------- quantise --

@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("n,k", [(1, 16), (33, 1040), (300, 4096), (7, 14336), (5, 65536)])
def test_quantize_16_bit_weights_bit_exact(n, k, act):
    """bf16 / fp16 weights: codes and scales equal the fp32 quantiser's on
    the exactly widened matrix."""
    rng = np.random.default_rng(n + k + act)
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    w[:, ::113] *= 300.0
    if n > 2:
        w[1] = 0.0                                        # zero row: scale 1.0
        w[2] *= 1e-4                                      # fp16 subnormals
    bits = synthetic.to_f16_bits(w) if act == oracle.ACT_F16 else synthetic.to_bf16_bits(w)
    wd = torch.from_numpy(bits.view(np.int16)).to(DEV).view(_dt(act))
    codes, scales = fw.quantize(wd)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_16(bits, act)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("shape,seed,kind", [
    ((1, 16), 1, "normal"), ((3, 48), 2, "normal"), ((129, 1040), 3, "t"),
    ((1024, 1024), 4, "normal"), ((300, 4096), 5, "t"), ((77, 14336), 6, "normal"),
    ((5, 16384), 7, "t"), ((3, 20000 // 16 * 16), 8, "normal"), ((2, 65536), 9, "t"),
])
def test_quantize_bit_exact(shape, seed, kind):
    rng = np.random.default_rng(seed)
    n, k = shape
    if kind == "t":
        w = (rng.standard_t(3, size=shape) * 0.02).astype(np.float32)
    else:
        w = (rng.standard_normal(shape) * 10.0 ** rng.uniform(-8, 3, size=(n, 1))).astype(np.float32)
    w[0, : min(k, 7)] = 0.0
    if n > 2:
        w[1] = 0.0                         # all-zero row -> scale 1
        w[2, 3] = np.float32(1e-45)        # underflowing amax -> scale 1
        w[2, 4] = np.float32(-1e-45)
    codes, scales = gpu_quantize(w)
    rc, rs = oracle.quantize(w)
    assert np.array_equal(scales.view(np.uint32), rs.view(np.uint32))
    bad = np.nonzero(codes != rc)
    assert bad[0].size == 0, (bad[0][:5], bad[1][:5], codes[bad][:5], rc[bad][:5], w[bad][:5])


def test_quantize_configs_bit_exact():
    for name in ("tiny_gemv", "outlier_gemv", "fp16_template"):
        w = synthetic.case(name)["w"]
        codes, scales = gpu_quantize(w)
        rc, rs = oracle.quantize(w)
        assert np.array_equal(scales.view(np.uint32), rs.view(np.uint32)), name
        assert np.array_equal(codes, rc), name


@pytest.mark.parametrize("matrix", [s[0] for s in synthetic.DECODE_STACK])
def test_quantize_decode_stack_bit_exact(matrix):
    w = synthetic.case("decode_stack", 1, matrix)["w"]
    codes, scales = gpu_quantize(w)
    rc, rs = oracle.quantize(w)
    assert np.array_equal(scales.view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(codes, rc)


def test_quantize_every_reachable_fp32_bit_exact():
    """Rows [448, v...] have scale exactly 1, so their codes are e4m3(v): this
    sweeps every fp32 pattern in [2^-12, 448] of both signs, plus a strided
    sample of everything smaller (subnormals included), through the kernel's
    hardware conversion, against the oracle's encoder."""
    lo = np.float32(2.0 ** -12).view(np.uint32)
    hi = np.float32(448.0).view(np.uint32)
    dense = np.arange(lo, hi + 1, dtype=np.uint32)
    sparse = np.arange(0, lo, 4099, dtype=np.uint32)
    pos = np.concatenate([dense, sparse])
    vals = np.concatenate([pos, pos | np.uint32(0x80000000)]).view(np.float32)
    k = 4096
    per_row = k - 1
    rows = -(-vals.size // per_row)
    pad = np.zeros(rows * per_row, dtype=np.float32)
    pad[: vals.size] = vals
    w = np.empty((rows, k), dtype=np.float32)
    w[:, 0] = 448.0
    w[:, 1:] = pad.reshape(rows, per_row)
    del pad
    wd = torch.from_numpy(w).to(DEV)
    codes, scales = fw.quantize(wd)
    torch.cuda.synchronize()
    assert bool((scales == 1.0).all())
    got = codes[:, 1:].reshape(-1)[: vals.size].cpu().numpy()
    want = oracle.e4m3_encode(vals)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (vals[bad[:8]], got[bad[:8]], want[bad[:8]])


# ----------------------------------------------------------------- linear --

def _case(seed, m, n, k, act, with_bias=True, std=0.02):
    c = synthetic.random_case(seed, m, n, k, act=act, std=std, with_bias=with_bias)
    codes, scales = oracle.quantize(c["w"])
    return c, codes, scales


SHAPES = [  # (m, n, k): several tiles and ragged tails in n and k
    (1, 1, 16), (1, 33, 48), (1, 300, 1040), (1, 1024, 1024), (1, 257, 4096), (1, 130, 14336),
    (1, 64, 20000 // 16 * 16), (1, 40, 65536),
    (2, 300, 1040), (3, 129, 4096), (4, 1024, 1024), (7, 257, 2064), (8, 640, 4096),
    (16, 300, 1040), (17, 300, 1040), (22, 4096, 1024), (31, 129, 256), (32, 1000, 4096),
    (33, 300, 1040), (70, 260, 528), (2, 128, 16), (5, 513, 14336), (64, 1000, 4096), (129, 300, 2064),
]


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("m,n,k", SHAPES)
def test_linear_parity(m, n, k, act):
    c, codes, scales = _case(1000 * m + n + k + act, m, n, k, act, with_bias=(n % 2 == 0))
    y = gpu_linear(c["x"], act, codes, scales, c["bias"])
    ref = oracle.linear(c["x"], act, codes, scales, c["bias"])
    assert_parity(y, ref, act, (m, n, k))


@pytest.mark.parametrize("n,k", [
    (128, 128),      # one unit
    (1000, 256),     # 8 tiles x 2 k-blocks
    (2432, 1024),    # 19 tiles x 8 k-blocks = 152 units
    (1100, 4096),    # 9 tiles x 32
    (300, 14336),    # 3 tiles x 112 k-blocks
    (20000, 272),    # 157 tiles x 3 (ragged k): more tiles than SMs
    (14336, 4096),   # the gate weight: 112 tiles x 32
])
@pytest.mark.parametrize("m", [1, 2, 9, 32, 48, 64])
def test_tensor_core_shapes(m, n, k):
    """The tensor-core kernel in its automatic launch shape and in forced
    cluster shapes of every kind: whole tiles (one CTA a cluster, one or
    several tiles each), a tile split over a cluster, clusters of 2..8 ranks
    sharing 2..5 tiles (ranges that start and end inside tiles, a rank inside
    one tile, the last cluster with fewer tiles), ragged N and K; every
    output against the oracle."""
    c, codes, scales = _case(77 + m + n + k, m, n, k, oracle.ACT_BF16)
    ref = oracle.linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], threads=oracle.host_cores())
    nkb = -(-k // 128)
    shapes = [(0, 0), (1, 1), (1, 3), (2, 1), (8, 1), (2, 3), (3, 2), (4, 3), (5, 2), (7, 5), (4, 1)]
    for cl, tpc in shapes:
        if cl > nkb or (m > 32 and cl > 1 and tpc > 1):
            continue
        y = gpu_linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], kernel=fw.KERNEL_SKINNY,
                       cluster=cl, tiles=tpc)
        assert_parity(y, ref, oracle.ACT_BF16, (m, n, k, cl, tpc))


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("n,k", [
    (1, 512),        # one row: one CTA
    (151, 512),      # fewer rows than SMs
    (153, 1024),     # one CTA with two rows, the rest one
    (1000, 2048),    # odd and even row counts per CTA
    (4097, 4096),    # 27 rows a CTA: ragged last slot and row pair
    (700, 14336),    # long rows: one row per item, rows split over warps
    (96, 32768),     # the longest rows the GEMV takes
])
def test_gemv_shapes(n, k, act):
    """The M = 1 kernel across slot sizes, row pairs and warp groups, with
    odd row counts per CTA and both activation types."""
    c, codes, scales = _case(300 + n + k + act, 1, n, k, act, with_bias=(n % 2 == 1))
    ref = oracle.linear(c["x"], act, codes, scales, c["bias"], threads=oracle.host_cores())
    y = gpu_linear(c["x"], act, codes, scales, c["bias"], kernel=fw.KERNEL_GEMV)
    assert_parity(y, ref, act, (1, n, k))


@pytest.mark.parametrize("kind", ["huge", "tiny", "subnormal", "spread", "zero", "one_big"])
def test_gemv_activation_range(kind):
    """The GEMV's result must not depend on where x's values sit in bf16's
    range: huge, tiny, subnormal, widely spread, all zero, one outlier."""
    n, k = 500, 4096
    rng = np.random.default_rng(11)
    # weights 2^20 larger keep y a normal number when x is tiny
    c, codes, scales = _case(41, 1, n, k, oracle.ACT_BF16, with_bias=False,
                             std=0.02 * (2.0 ** 20 if kind in ("tiny", "subnormal") else 1.0))
    xf = rng.standard_normal((1, k))
    if kind == "huge":
        # the fp32 sum is in code units (|code| <= 448): it holds x up to ~2^110
        xf *= 2.0 ** 100
    elif kind == "tiny":
        xf *= 2.0 ** -120
    elif kind == "subnormal":
        xf *= 2.0 ** -128          # bf16 subnormals and the smallest normals
    elif kind == "spread":
        xf *= 2.0 ** rng.integers(-40, 40, size=(1, k))
    elif kind == "zero":
        xf[:] = 0.0
    elif kind == "one_big":
        xf[0, 17] = 3.0e4
    x = synthetic.to_bf16_bits(xf.astype(np.float32))
    y = gpu_linear(x, oracle.ACT_BF16, codes, scales, None, kernel=fw.KERNEL_GEMV)
    ref = oracle.linear(x, oracle.ACT_BF16, codes, scales, None)
    if kind == "zero":
        assert not y.any() or np.all((y & 0x7FFF) == 0)
    else:
        assert_parity(y, ref, oracle.ACT_BF16, kind)


def test_calls_on_two_streams_at_once_are_independent():
    """The library keeps no state between calls: calls of different shapes
    enqueued on two streams at the same time, over and over, give the same
    bits as the same calls one at a time."""
    shapes = [(8, 1100, 4096), (32, 14336, 4096), (3, 300, 14336), (16, 20000, 272)]
    runs = []
    for i, (m, n, k) in enumerate(shapes):
        c, codes, scales = _case(500 + i, m, n, k, oracle.ACT_BF16)
        x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
        cd, sd, bd = (torch.from_numpy(v).to(DEV) for v in (codes, scales, c["bias"]))
        ref = oracle.linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], threads=oracle.host_cores())
        runs.append((x, cd, sd, bd, ref))
    serial = [fw.linear(x, cd, sd, bd) for x, cd, sd, bd, _ in runs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(device=DEV), torch.cuda.Stream(device=DEV)]
    outs = [[torch.empty_like(y) for y in serial] for _ in range(8)]
    for rep in range(8):
        for i, (x, cd, sd, bd, _) in enumerate(runs):
            with torch.cuda.stream(streams[(i + rep) % 2]):
                fw.linear(x, cd, sd, bd, out=outs[rep][i])
    torch.cuda.synchronize()
    for i, (_, _, _, _, ref) in enumerate(runs):
        assert_parity(serial[i].view(torch.int16).cpu().numpy().view(np.uint16), ref, oracle.ACT_BF16, shapes[i])
        for rep in range(8):
            assert torch.equal(outs[rep][i].view(torch.int16), serial[i].view(torch.int16)), (rep, shapes[i])
    assert fw.device_error() == 0


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("kernel,m", [(fw.KERNEL_GEMV, 1), (fw.KERNEL_SKINNY, 1), (fw.KERNEL_SKINNY, 5),
                                      (fw.KERNEL_SKINNY, 32), (fw.KERNEL_SKINNY, 64), (fw.KERNEL_PREFILL, 2),
                                      (fw.KERNEL_PREFILL, 65), (fw.KERNEL_PREFILL, 200), (fw.KERNEL_PREFILL, 300)])
def test_exact_cases_bit_identical(kernel, m, act):
    """Power-of-two scales, small-integer activations and weights whose codes
    lie in [1/8, 8] (plus the 448 that fixes the scale): every product and
    partial sum is a multiple of 2^-6 below 2^14, so the fp32 accumulation is
    exact in any order and the output must equal the oracle bit for bit."""
    rng = np.random.default_rng(5 + m + act)
    n, k = 300, 512
    t = oracle.e4m3_decode_table()
    mid = np.nonzero(np.isfinite(t) & (np.abs(t) >= 0.125) & (np.abs(t) <= 8.0))[0]
    p = 2.0 ** (np.arange(n) % 9 - 4)
    w = (t[rng.choice(mid, size=(n, k))] * p[:, None]).astype(np.float32)
    w[np.arange(n), np.arange(n) % k] = (448.0 * p).astype(np.float32)
    codes, scales = oracle.quantize(w)
    assert np.array_equal(scales, p.astype(np.float32))
    xi = rng.integers(-3, 4, size=(m, k)).astype(np.float32)
    to_bits = synthetic.to_f16_bits if act == oracle.ACT_F16 else synthetic.to_bf16_bits
    x = to_bits(xi)
    bias = (rng.integers(-2, 3, size=n) * p).astype(np.float32)
    y = gpu_linear(x, act, codes, scales, bias, kernel=kernel)
    ref = oracle.linear(x, act, codes, scales, bias)
    assert np.array_equal(y, ref)


@pytest.mark.parametrize("m,n,k", [(8, 14300, 1024), (32, 13700, 512), (8, 14600, 512), (16, 14336, 272)])
def test_whole_tile_launches(m, n, k):
    """Whole-tile launches (108 to 115 tiles of 128 rows, one a CTA) with a
    ragged last tile or a ragged k."""
    c, codes, scales = _case(900 + m + n + k, m, n, k, oracle.ACT_BF16)
    y = gpu_linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"])
    ref = oracle.linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], threads=oracle.host_cores())
    assert_parity(y, ref, oracle.ACT_BF16, (m, n, k))


# ------------------------------------------------------- prefill GEMM (K4) --

PREFILL_SHAPES = [  # (m, n, k): 128- and 256-token tiles, ragged m, n and k (k % 128 == 16, 64, 112)
    (65, 300, 1040), (100, 129, 4096), (128, 1000, 512), (129, 257, 2064), (200, 640, 4096),
    (256, 130, 1008), (300, 1024, 1024), (513, 300, 256), (777, 64, 2000),
    (100, 50, 16), (70, 200, 64), (300, 33, 48), (66, 1, 16),   # k below one code stage, one row
]


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("m,n,k", PREFILL_SHAPES)
def test_prefill_parity(m, n, k, act):
    c, codes, scales = _case(7000 + m + n + k + act, m, n, k, act, with_bias=(m % 2 == 1))
    y = gpu_linear(c["x"], act, codes, scales, c["bias"])          # m > 64: the prefill GEMM
    ref = oracle.linear(c["x"], act, codes, scales, c["bias"], threads=oracle.host_cores())
    assert_parity(y, ref, act, (m, n, k))


@pytest.mark.parametrize("m", [512, 2048])
def test_prefill_full_gate_every_output(m):
    """The gate weight [14336 x 4096] at prefill sizes, in the launch shape a
    caller gets: every output against the oracle."""
    base = synthetic.case("decode_stack", 1, "gate")
    rng = np.random.default_rng(m)
    x = synthetic.to_bf16_bits(rng.standard_normal((m, 4096)).astype(np.float32))
    case = dict(base, m=m, x=x)
    _full_parity(case)


@pytest.mark.parametrize("m", [1, 2, 17])
def test_prefill_kernel_at_few_tokens(m):
    """The prefill GEMM chosen explicitly for a handful of tokens (a mostly
    empty 128-token tile)."""
    c, codes, scales = _case(61 + m, m, 300, 1040, oracle.ACT_BF16)
    y = gpu_linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], kernel=fw.KERNEL_PREFILL)
    assert_parity(y, oracle.linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"]), oracle.ACT_BF16, m)


def test_prefill_captures_in_a_graph():
    """No path needs a workspace, so a prefill call can be captured in a CUDA
    graph with nothing allocated for it."""
    c, codes, scales = _case(47, 100, 300, 1024, oracle.ACT_BF16)
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
    cd, sd, bd = (torch.from_numpy(v).to(DEV) for v in (codes, scales, c["bias"]))
    y = torch.empty((100, 300), dtype=torch.bfloat16, device=DEV)
    fw.linear(x, cd, sd, bd, out=torch.empty_like(y))     # eager first launch (function attributes)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(device=DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fw.linear(x, cd, sd, bd, out=y)
    g.replay()
    torch.cuda.synchronize()
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_parity(got, oracle.linear(c["x"], 1, codes, scales, c["bias"], threads=oracle.host_cores()), 1, "graph")


def test_prefill_agrees_with_the_skinny_kernel():
    c, codes, scales = _case(41, 200, 1000, 4096, oracle.ACT_BF16)
    yp = gpu_linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], kernel=fw.KERNEL_PREFILL)
    ys = gpu_linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], kernel=fw.KERNEL_SKINNY)
    cmp = compare(yp, ys, oracle.ACT_BF16)
    assert cmp["rel_l2"] <= 2e-3 and cmp["min_cosine"] >= 0.9999 and cmp["bit_equal"] >= 0.9, cmp


def test_prefill_without_workspace_through_the_no_alloc_entry():
    c, codes, scales = _case(43, 150, 300, 1024, oracle.ACT_BF16)
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
    y = torch.empty((150, 300), dtype=torch.bfloat16, device=DEV)
    cd, sd, bd = (torch.from_numpy(v).to(DEV) for v in (codes, scales, c["bias"]))
    st = fw.lib().fp8w_linear_noalloc(x.data_ptr(), 1, 150, 1024, cd.data_ptr(), sd.data_ptr(), bd.data_ptr(), 300,
                                      y.data_ptr(), None)
    assert st == 0
    torch.cuda.synchronize()
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_parity(got, oracle.linear(c["x"], 1, codes, scales, c["bias"], threads=oracle.host_cores()), 1, "noalloc")


def test_one_hot_reads_every_code():
    """x = e_j reads column j of the quantised weight: y[n] = RN(scale[n] * e4m3(q[n, j])),
    with scale a power of two so the product is exact; column j holds all 254
    finite codes down the rows."""
    t = oracle.e4m3_decode_table()
    fin = [b for b in range(256) if np.isfinite(t[b])]
    n, k = 256, 64
    w = np.zeros((n, k), dtype=np.float32)
    w[:, 0] = 448.0
    w[: len(fin), 5] = t[fin]
    codes, scales = oracle.quantize(w)
    assert np.all(scales == 1.0)
    for act in (oracle.ACT_BF16, oracle.ACT_F16):
        to_bits = synthetic.to_f16_bits if act == oracle.ACT_F16 else synthetic.to_bf16_bits
        for m, kern in ((1, fw.KERNEL_GEMV), (1, fw.KERNEL_SKINNY), (3, fw.KERNEL_SKINNY), (70, fw.KERNEL_PREFILL)):
            xf = np.zeros((m, k), dtype=np.float32)
            xf[:, 5] = 1.0
            y = gpu_linear(to_bits(xf), act, codes, scales, None, kernel=kern)
            ref = oracle.linear(to_bits(xf), act, codes, scales, None)
            assert np.array_equal(y, ref), (act, m, kern)


def test_bias_none_equals_zero_bias_and_runs_are_deterministic():
    c, codes, scales = _case(99, 8, 700, 4096, oracle.ACT_BF16)
    for m in (1, 8):
        x = c["x"][:m]
        a = gpu_linear(x, oracle.ACT_BF16, codes, scales, None)
        b = gpu_linear(x, oracle.ACT_BF16, codes, scales, np.zeros(700, np.float32))
        d = gpu_linear(x, oracle.ACT_BF16, codes, scales, None)
        assert np.array_equal(a, b) and np.array_equal(a, d)


def test_cuda_graph_capture_replays_identically():
    c, codes, scales = _case(7, 8, 1000, 4096, oracle.ACT_BF16)
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
    cd = torch.from_numpy(codes).to(DEV)
    sd = torch.from_numpy(scales).to(DEV)
    bd = torch.from_numpy(c["bias"]).to(DEV)
    y1 = torch.empty((1, 1000), dtype=torch.bfloat16, device=DEV)
    y8 = torch.empty((8, 1000), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fw.linear(x[:1], cd, sd, bd, out=y1)
        fw.linear(x, cd, sd, bd, out=y8)
    torch.cuda.synchronize()
    ref1, ref8 = y1.clone(), y8.clone()
    y1.zero_()
    y8.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fw.linear(x[:1], cd, sd, bd, out=y1)
        fw.linear(x, cd, sd, bd, out=y8)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1, ref1) and torch.equal(y8, ref8)


# ---------------------------------------------------- full-size workloads --

def _full_parity(case, kernel=fw.KERNEL_AUTO, weights_ready=False):
    """Every output of a full-size case against the oracle (on all host
    cores), codes and scales bit-exact, in the launch shape the bench uses."""
    act = case["act"]
    codes, scales = gpu_quantize(case["w"])
    rc, rs = oracle.quantize(case["w"])
    assert np.array_equal(codes, rc) and np.array_equal(scales.view(np.uint32), rs.view(np.uint32))
    y = gpu_linear(case["x"], act, codes, scales, case["bias"], kernel=kernel, weights_ready=weights_ready)
    ref = oracle.linear(case["x"], act, rc, rs, case["bias"], threads=oracle.host_cores())
    return assert_parity(y, ref, act, (case["m"], case["n"], case["k"]))


@pytest.mark.parametrize("name", ["tiny_gemv", "outlier_gemv", "fp16_template"])
def test_config_parity_full(name):
    case = synthetic.case(name)
    act = case["act"]
    codes, scales = oracle.quantize(case["w"])
    y = gpu_linear(case["x"], act, codes, scales, case["bias"])
    ref = oracle.linear(case["x"], act, codes, scales, case["bias"], threads=oracle.host_cores())
    assert_parity(y, ref, act, name)
    if name == "outlier_gemv":
        yb = gpu_linear(case["x"], act, codes, scales, np.zeros(case["n"], np.float32))
        assert np.array_equal(y, yb)


@pytest.mark.parametrize("m", (1,) + synthetic.SKINNY_M)
def test_skinny_sweep_every_output(m):
    _full_parity(synthetic.case("skinny_sweep", m))


@pytest.mark.parametrize("m", synthetic.DECODE_STACK_M)
@pytest.mark.parametrize("matrix", [s[0] for s in synthetic.DECODE_STACK])
def test_decode_stack_every_output(matrix, m):
    """The bench's calls: weights ready, as the timed step passes them."""
    _full_parity(synthetic.case("decode_stack", m, matrix), weights_ready=True)


def test_m1_tensor_core_path_matches_gemv_tolerance():
    case = synthetic.case("decode_stack", 1, "gate")
    codes, scales = oracle.quantize(case["w"])
    yg = gpu_linear(case["x"], 1, codes, scales, case["bias"], kernel=fw.KERNEL_GEMV)
    yt = gpu_linear(case["x"], 1, codes, scales, case["bias"], kernel=fw.KERNEL_SKINNY)
    c = compare(yt, yg, 1)
    assert c["rel_l2"] <= 2e-3 and c["min_cosine"] >= 0.9999, c


@pytest.mark.parametrize("m,matrix", [(1, "gate"), (32, "gate"), (8, "down"), (1, "down"), (32, "k")])
def test_full_size_outputs_within_the_quantisation_bound(m, matrix):
    """At the bench's sizes and launch configuration, with GPU-quantised
    weights, every sampled output lies within the e4m3 bound of the
    UNQUANTISED product x . W^T + b: half an e4m3 step a weight (2^-4 of |w|,
    or 2^-10 * scale below the normal range), widened by the fp32
    accumulation (k * 2^-22 of sum |x w|, generous for any summation order)
    and the one rounding to bf16 (2^-8 of |y|).  That worst case is loose at
    large k, so the aggregate is also held to the statistical level of
    independent, centred e4m3 rounding errors: rel_l2 about 0.0255 (a
    doubled scale gives 1.0, a permuted channel 1.4).  A check against the
    mathematics rather than the oracle."""
    case = synthetic.case("decode_stack", m, matrix)
    codes, scales = gpu_quantize(case["w"])
    y = gpu_linear(case["x"], case["act"], codes, scales, case["bias"])
    n, k = case["n"], case["k"]
    cols = np.random.default_rng(m + n).choice(n, size=256, replace=False)
    x = oracle.act_values(case["x"], case["act"])
    w = case["w"][cols].astype(np.float64)
    y_true = x @ w.T + case["bias"][cols].astype(np.float64)
    yv = oracle.act_values(y[:, cols], case["act"])
    ax, aw = np.abs(x), np.abs(w)
    quant = ax @ (2.0 ** -4 * aw * (1 + 2.0 ** -20)).T + ax.sum(1)[:, None] * 2.0 ** -10 * scales[cols].astype(np.float64)
    accum = k * 2.0 ** -22 * (ax @ (aw * (1 + 2.0 ** -4)).T)
    bound = (quant + accum) * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(y_true) + 1e-30
    err = np.abs(yv - y_true)
    assert np.all(err <= bound), float(np.max(err / bound))
    rel = np.linalg.norm(yv - y_true) / np.linalg.norm(y_true)
    assert 0.015 <= rel <= 0.04, rel


# ------------------------------------------------------ fused decode stack --

FUSED = {"qkv": ("q", "k", "v"), "gate_up": ("gate", "up")}


@pytest.mark.parametrize("group", list(FUSED))
def test_fused_weights_quantise_as_their_parts(group):
    """q/k/v (and gate/up) fused into one weight of concatenated rows: the
    quantiser is row-wise, so the fused codes and scales are the parts'
    codes and scales, bit for bit."""
    ws = [synthetic.case("decode_stack", 1, name)["w"] for name in FUSED[group]]
    fused_codes, fused_scales = gpu_quantize(np.concatenate(ws))
    parts = [gpu_quantize(w) for w in ws]
    assert np.array_equal(fused_codes, np.concatenate([p[0] for p in parts]))
    assert np.array_equal(fused_scales, np.concatenate([p[1] for p in parts]))


@pytest.mark.parametrize("m", synthetic.DECODE_STACK_M)
@pytest.mark.parametrize("group", list(FUSED))
def test_fused_linear_matches_its_parts(group, m):
    """One call over the fused weight and the parts' calls on the same x.
    At M = 1 every row's sum runs in the same order in both launches, so the
    outputs are bit-identical; at M = 8 and 32 the tensor-core kernel shares
    the fused tiles differently (gate/up: 224 tiles, clusters of ranks that
    share tiles), so both are held to the oracle on every channel."""
    cases = [synthetic.case("decode_stack", m, name) for name in FUSED[group]]
    x = cases[0]["x"]
    q = [oracle.quantize(c["w"]) for c in cases]
    codes = np.concatenate([c for c, _ in q])
    scales = np.concatenate([s for _, s in q])
    bias = np.concatenate([c["bias"] for c in cases])
    y = gpu_linear(x, oracle.ACT_BF16, codes, scales, bias)
    parts = np.concatenate([gpu_linear(x, oracle.ACT_BF16, cq, sq, c["bias"]) for (cq, sq), c in zip(q, cases)],
                           axis=1)
    if m == 1:
        assert np.array_equal(y, parts)
    ref = oracle.linear(x, oracle.ACT_BF16, codes, scales, bias, threads=oracle.host_cores())
    assert_parity(y, ref, oracle.ACT_BF16, (group, m))
    assert_parity(parts, ref, oracle.ACT_BF16, (group, m, "parts"))


# ------------------------------------------------------------ dequantise --

def _oracle_dequant_bits(codes, scales, dtype):
    """The oracle's exact product rounded once to dtype, as raw bits."""
    w = oracle.dequantize(codes, scales)
    if dtype == torch.float32:
        return w.astype(np.float32).view(np.uint32)
    return (oracle.round_bf16(w) if dtype == torch.bfloat16 else oracle.round_f16(w)).reshape(w.shape)


def _gpu_dequant_bits(codes, scales, dtype):
    c = torch.from_numpy(np.ascontiguousarray(codes)).to(DEV)
    s = torch.from_numpy(np.ascontiguousarray(scales)).to(DEV)
    n, k = codes.shape
    esize = 4 if dtype == torch.float32 else 2
    buf = torch.full(((n * k + 2 * CANARY) * esize,), 0xA5, dtype=torch.uint8, device=DEV)
    out = buf[CANARY * esize:(CANARY + n * k) * esize].view(dtype).view(n, k)
    fw.dequantize(c, s, dtype=dtype, out=out)
    torch.cuda.synchronize()
    assert bool((buf[:CANARY * esize] == 0xA5).all()) and bool((buf[(CANARY + n * k) * esize:] == 0xA5).all())
    raw = out.view(torch.int32 if esize == 4 else torch.int16).cpu().numpy()
    return raw.view(np.uint32 if esize == 4 else np.uint16)


DQ_TYPES = [torch.float32, torch.bfloat16, torch.float16]


@pytest.mark.parametrize("dtype", DQ_TYPES)
@pytest.mark.parametrize("n,k", [(1, 16), (37, 1040), (300, 4096), (1024, 14336)])
def test_dequantize_bit_exact(n, k, dtype):
    rng = np.random.default_rng(n + k)
    codes = rng.integers(0, 256, size=(n, k), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A               # NaN codes are tested apart
    # scales over a wide range, fp16 outputs kept within fp16's range
    hi_exp = 6 if dtype == torch.float16 else 60
    scales = (2.0 ** rng.uniform(-30, hi_exp, size=n) * rng.uniform(1, 2, size=n)).astype(np.float32)
    got = _gpu_dequant_bits(codes, scales, dtype)
    want = _oracle_dequant_bits(codes, scales, dtype)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], want[tuple(bad[0])])


def _tie_cases(bits_fn, lo_range, hi_range, mask, tie, seed, rounds=20):
    """(code, scale) pairs whose fp32 product lies exactly on a rounding
    midpoint of the 16-bit type while the exact product does not: the case
    where rounding the fp32 product again would round twice."""
    t = oracle.e4m3_decode_table()
    pos = np.array([b for b in range(1, 127) if np.isfinite(t[b])], dtype=np.uint8)
    rng = np.random.default_rng(seed)
    found_c, found_s = [], []
    for _ in range(rounds):
        s = rng.uniform(lo_range, hi_range, size=200_000).astype(np.float32)
        c = rng.choice(pos, size=s.size)
        p = t[c] * s.astype(np.float64)
        hi = p.astype(np.float32)
        sel = ((bits_fn(hi) & mask) == tie) & (hi.astype(np.float64) != p)
        found_c.append(c[sel])
        found_s.append(s[sel])
    c = np.concatenate(found_c)
    s = np.concatenate(found_s)
    sign = (np.arange(c.size) % 2 * 0x80).astype(np.uint8)   # half of them negative
    return np.repeat((c | sign)[:, None], 16, axis=1), s


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_dequantize_rounds_once_at_exact_midpoints(dtype):
    if dtype == torch.bfloat16:
        codes, scales = _tie_cases(lambda h: h.view(np.uint32), 1e-4, 1e-1, 0xFFFF, 0x8000, 21, rounds=60)
    else:
        # fp16 normal range: the 13 low mantissa bits of the fp32 midpoint are 1000000000000
        codes, scales = _tie_cases(lambda h: h.view(np.uint32), 1e-2, 10.0, 0x1FFF, 0x1000, 22)
        keep = np.abs(oracle.dequantize(codes[:, :1], scales)[:, 0]) >= 2.0 ** -14
        codes, scales = codes[keep], scales[keep]
    assert codes.shape[0] >= 50
    got = _gpu_dequant_bits(codes, scales, dtype)
    want = _oracle_dequant_bits(codes, scales, dtype)
    assert np.array_equal(got, want)
    # the cases matter: rounding the fp32 product again differs from the exact rounding in some
    hi = (oracle.dequantize(codes, scales)).astype(np.float32).astype(np.float64)
    twice = (oracle.round_bf16(hi) if dtype == torch.bfloat16 else oracle.round_f16(hi)).reshape(hi.shape)
    assert np.count_nonzero(twice != want) > 0


@pytest.mark.parametrize("dtype", DQ_TYPES)
def test_dequantize_nan_codes_give_nan(dtype):
    codes = np.tile(np.array([0x7F, 0xFF, 0x00, 0x80], np.uint8), (2, 4))
    got = _gpu_dequant_bits(codes, np.float32([0.5, 3.0]), dtype)
    vals = torch.from_numpy(got.view(np.int32 if dtype == torch.float32 else np.int16)).view(dtype).float().numpy()
    assert np.isnan(vals[:, 0::4]).all() and np.isnan(vals[:, 1::4]).all()
    assert (vals[:, 2::4] == 0).all() and (vals[:, 3::4] == 0).all()


@pytest.mark.parametrize("dtype", DQ_TYPES)
@pytest.mark.parametrize("form", ["g32", "g64", "g128", "mx"])
@pytest.mark.parametrize("n,k", [(3, 128), (77, 1024), (300, 4096)])
def test_dequantize_grouped_and_mx_bit_exact(n, k, form, dtype):
    rng = np.random.default_rng(n + k + len(form))
    codes = rng.integers(0, 256, size=(n, k), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A
    if form == "mx":
        lo, hi = (100, 140) if dtype == torch.float16 else (1, 250)
        scales = rng.integers(lo, hi, size=(n, k // 32), dtype=np.uint8)
        if dtype != torch.float16:
            scales[0, :2] = [0, 254]                      # 2^-127 and 2^127 (products overflow to inf)
        want_w = oracle.dequantize_mx(codes, scales)
    else:
        g = int(form[1:])
        hi_exp = 6 if dtype == torch.float16 else 60
        scales = (2.0 ** rng.uniform(-30, hi_exp, size=(n, k // g)) * rng.uniform(1, 2, size=(n, k // g))).astype(np.float32)
        want_w = oracle.dequantize_grouped(codes, scales, g)
    got = _gpu_dequant_bits(codes, scales, dtype)
    if dtype == torch.float32:
        with np.errstate(over="ignore"):                   # products beyond fp32 round to inf, as intended
            want = want_w.astype(np.float32).view(np.uint32)
    else:
        want = (oracle.round_bf16(want_w) if dtype == torch.bfloat16 else oracle.round_f16(want_w)).reshape(want_w.shape)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], want[tuple(bad[0])])


def test_dequantize_mx_of_quantize_mx_is_the_oracle_weight():
    case = synthetic.case("decode_stack", 1, "k")
    w = torch.from_numpy(case["w"]).to(DEV)
    codes, e8 = fw.quantize_mx(w)
    c, s = codes.cpu().numpy(), e8.cpu().numpy()
    got = _gpu_dequant_bits(c, s, torch.float32)
    assert np.array_equal(got, oracle.dequantize_mx(c, s).astype(np.float32).view(np.uint32))


def test_dequantize_of_quantize_is_the_oracle_fallback_weight():
    case = synthetic.case("decode_stack", 1, "k")
    codes, scales = gpu_quantize(case["w"])
    got = _gpu_dequant_bits(codes, scales, torch.float32)
    assert np.array_equal(got, oracle.dequantize(codes, scales).astype(np.float32).view(np.uint32))


# ------------------------------------------------------ per-group scales --

@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("n,k,kind", [(1, 128, "normal"), (300, 4096, "t"), (77, 14336, "normal"),
                                      (5, 1152, "zeros")])
def test_quantize_grouped_bit_exact(n, k, kind, group):
    if k % group:
        pytest.skip("k not a multiple of the group")
    if kind == "t":
        w = synthetic.weight_outlier(31 + n, n, k)
    else:
        w = synthetic.weight_normal(37 + n, n, k, 0.02)
    if kind == "zeros":
        w[:, :group] = 0.0                               # a whole zero group: scale 1.0
        w[1, group: 2 * group] = 1e-45                    # an underflowing group
    wd = torch.from_numpy(w).to(DEV)
    codes, scales = fw.quantize(wd, group=group)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_grouped(w, group)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("n,k,group", [(1, 512, 32), (300, 4096, 32), (1000, 4096, 128), (257, 14336, 64),
                                       (4097, 4096, 128), (153, 1024, 64), (64, 32768, 128)])
def test_linear_grouped_parity(n, k, group, act):
    c = synthetic.random_case(900 + n + k + group + act, 1, n, k, act=act, with_bias=(n % 2 == 1))
    w = c["w"].copy()
    w[:, ::97] *= 40.0                                    # outliers that per-group scales contain
    codes, scales = oracle.quantize_grouped(w, group)
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(_dt(act))
    cd = torch.from_numpy(codes).to(DEV)
    sd = torch.from_numpy(scales).to(DEV)
    bd = None if c["bias"] is None else torch.from_numpy(c["bias"]).to(DEV)
    buf, y = _guarded(n, _dt(act), POISON16)
    fw.linear(x, cd, sd, bd, out=y.view(1, n))
    torch.cuda.synchronize()
    _check_canaries(buf, n, POISON16)
    assert fw.device_error() == 0
    got = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(1, n)
    ref = oracle.linear_grouped(c["x"], act, codes, scales, group, c["bias"], threads=oracle.host_cores())
    assert_parity(got, ref, act, (n, k, group))


def _mx_weight(seed, n, k, kind):
    if kind == "t":
        w = synthetic.weight_outlier(seed, n, k)
    else:
        w = synthetic.weight_normal(seed, n, k, 0.02)
    if kind == "range":
        # blocks spread over the whole fp32 exponent range: clamped (2^-127),
        # subnormal and near-FLT_MAX amaxes, and exact 448 * 2^e boundaries
        rng = np.random.default_rng(seed)
        ex = rng.integers(-149, 128, size=(n, k // 32)).astype(np.float64)
        w = (w.reshape(n, k // 32, 32) / 0.1 * 2.0 ** ex[:, :, None]).astype(np.float32).reshape(n, k)
        w[np.isinf(w)] = np.float32(3e38)
        w[0, 0:32] = 0.0
        if k >= 96:
            w[0, 32] = np.float32(448.0 * 2.0 ** -20)
            w[0, 64] = np.nextafter(np.float32(448.0 * 2.0 ** 5), np.float32(np.inf))
    if kind == "inf":
        w[n // 2, 40 % k] = np.inf
        w[0, 3] = -np.inf
    return w


@pytest.mark.parametrize("kind", ["normal", "t", "range", "inf"])
@pytest.mark.parametrize("n,k", [(1, 32), (7, 96), (300, 4096), (257, 14336), (33, 1056)])
def test_quantize_mx_bit_exact(n, k, kind):
    w = _mx_weight(41 + n + k, n, k, kind)
    codes, scales = fw.quantize_mx(torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_mx(w)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantize_mx_scale_byte_at_every_boundary():
    """One block per amax 448 * 2^e and its two fp32 neighbours, e over the
    whole range, plus tiny and huge amaxes: every byte as the oracle's."""
    amax = []
    for e in range(-140, 120):
        v = np.float32(448.0 * 2.0 ** e)
        if v == 0 or not np.isfinite(v):
            continue
        amax += [np.nextafter(v, np.float32(0)), v, np.nextafter(v, np.float32(np.inf))]
    amax += [np.float32(1e-45), np.float32(1e-40), np.finfo(np.float32).max, np.float32(0)]
    w = np.zeros((len(amax), 32), np.float32)
    for i, a in enumerate(amax):
        w[i, :] = a / np.float32(3)
        w[i, i % 32] = -a
    codes, scales = fw.quantize_mx(torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_mx(w)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
@pytest.mark.parametrize("n,k", [(1, 512), (300, 4096), (1000, 4096), (257, 14336), (4097, 4096), (153, 1024),
                                 (64, 32768), (14336, 4096)])
def test_linear_mx_parity(n, k, act):
    c = synthetic.random_case(700 + n + k + act, 1, n, k, act=act, with_bias=(n % 2 == 1))
    w = c["w"].copy()
    w[:, ::97] *= 40.0                                    # outliers that the blocks of 32 contain
    codes, scales = oracle.quantize_mx(w)
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(_dt(act))
    cd = torch.from_numpy(codes).to(DEV)
    sd = torch.from_numpy(scales).to(DEV)
    bd = None if c["bias"] is None else torch.from_numpy(c["bias"]).to(DEV)
    buf, y = _guarded(n, _dt(act), POISON16)
    fw.linear(x, cd, sd, bd, out=y.view(1, n))
    torch.cuda.synchronize()
    _check_canaries(buf, n, POISON16)
    assert fw.device_error() == 0
    got = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(1, n)
    ref = oracle.linear_mx(c["x"], act, codes, scales, c["bias"], threads=oracle.host_cores())
    assert_parity(got, ref, act, (n, k, "mx"))


def test_linear_mx_equals_the_grouped_linear_on_decoded_scales():
    """The E8M0 bytes decode to exact fp32 powers of two: the MX GEMV and the
    fp32 per-group GEMV at g = 32 do the same arithmetic, bit for bit,
    including the 2^-127 and 2^127 ends and the NaN byte."""
    n, k = 700, 4096
    c = synthetic.random_case(5, 1, n, k, act=oracle.ACT_BF16, with_bias=True)
    codes, scales = oracle.quantize_mx(c["w"])
    scales[3, :4] = [0, 1, 254, 253]
    scales[5, 7] = 255
    dec = np.vectorize(oracle.e8m0_decode)(scales).astype(np.float32)
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
    cd = torch.from_numpy(codes).to(DEV)
    bd = torch.from_numpy(c["bias"]).to(DEV)
    y_mx = fw.linear(x, cd, torch.from_numpy(scales).to(DEV), bd)
    y_g = fw.linear(x, cd, torch.from_numpy(dec).to(DEV), bd)
    torch.cuda.synchronize()
    a = y_mx.view(torch.int16).cpu().numpy()
    b = y_g.view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b)
    assert (int(a[0, 5]) & 0x7FFF) > 0x7F80              # the NaN byte's row is NaN
    assert np.count_nonzero((a[0] & 0x7FFF) > 0x7F80) == 1 + int(((a[0, 3] & 0x7FFF) > 0x7F80))


MX_TC_SHAPES = [  # (m, n, k): the tensor-core form (whole tiles, cluster splits, stream-K) and, beyond 64
    (1, 300, 384), (2, 300, 4096), (8, 4096, 4096), (9, 1024, 4096), (32, 14336, 4096), (17, 257, 640),
    (8, 20480, 1024), (48, 1000, 1024), (64, 640, 14336), (70, 257, 640), (129, 130, 256),   # tokens, the prefill GEMM
    (200, 1000, 4096), (513, 300, 1024), (90, 64, 128), (65, 300, 384),
]


def _mx_case(seed, m, n, k):
    c = synthetic.random_case(seed, m, n, k, act=oracle.ACT_BF16, with_bias=(n % 2 == 1))
    w = c["w"].copy()
    w[:, ::97] *= 40.0
    codes, scales = oracle.quantize_mx(w)
    return c, codes, scales


def _gpu_mx(c, codes, scales):
    m, k = c["x"].shape
    n = codes.shape[0]
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
    bd = None if c["bias"] is None else torch.from_numpy(c["bias"]).to(DEV)
    buf, y = _guarded(m * n, torch.bfloat16, POISON16)
    fw.linear(x, torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV), bd, out=y.view(m, n))
    torch.cuda.synchronize()
    _check_canaries(buf, m * n, POISON16)
    assert fw.device_error() == 0
    return y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(m, n)


@pytest.mark.parametrize("m,n,k", MX_TC_SHAPES)
def test_linear_mx_tensor_core_parity(m, n, k):
    c, codes, scales = _mx_case(300 + m + n + k, m, n, k)
    got = _gpu_mx(c, codes, scales)
    ref = oracle.linear_mx(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], threads=oracle.host_cores())
    assert_parity(got, ref, oracle.ACT_BF16, (m, n, k, "mx"))


@pytest.mark.parametrize("m,n,k,lo,hi", [
    (8, 4096, 4096, 100, 134),      # one multiply
    (32, 14336, 1024, 100, 134),
    (8, 1000, 4096, 120, 141),      # rows with bytes 135..254: two multiplies in their warps
    (48, 300, 1024, 130, 150),
    (100, 640, 1024, 100, 134),     # the prefill GEMM, one and two multiplies
    (300, 1000, 512, 120, 141),
])
def test_linear_mx_with_equal_blocks_is_the_per_channel_linear(m, n, k, lo, hi):
    """Every block of a row with the same byte b: the MX result equals the
    per-channel result with scale 2^(b - 127) bit for bit (a power of two
    commutes with every rounding of the fp32 sums)."""
    rng = np.random.default_rng(m + n + k + lo)
    c = synthetic.random_case(31 + m + n, m, n, k, act=oracle.ACT_BF16, with_bias=True)
    codes = rng.integers(0, 0x7E, size=(n, k), dtype=np.uint8) | rng.integers(0, 2, size=(n, k), dtype=np.uint8) << 7
    b = rng.integers(lo, hi + 1, size=n).astype(np.uint8)
    e8 = np.repeat(b[:, None], k // 32, axis=1)
    per_row = np.float32(2.0) ** (b.astype(np.int32) - 127).astype(np.float32)
    y_mx = _gpu_mx(c, codes, e8)
    kern = fw.KERNEL_PREFILL if m > 64 else fw.KERNEL_SKINNY
    y_pc = gpu_linear(c["x"], oracle.ACT_BF16, codes, per_row, c["bias"], kernel=kern)
    assert np.array_equal(y_mx, y_pc)


def test_linear_mx_tensor_core_nan_byte_poisons_its_row_only():
    m, n, k = 8, 640, 1024
    c, codes, scales = _mx_case(77, m, n, k)
    scales[5, 3] = 255
    got = _gpu_mx(c, codes, scales)
    nan = (got & 0x7FFF) > 0x7F80
    assert nan[:, 5].all() and nan.sum() == m
    ref = oracle.linear_mx(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], threads=oracle.host_cores())
    keep = np.ones(n, bool)
    keep[5] = False
    assert_parity(got[:, keep], ref[:, keep], oracle.ACT_BF16, "nan row")


def test_linear_grouped_with_one_scale_per_group_equal_to_per_channel():
    """Group scales all equal to the row's scale: the grouped GEMV must give
    the per-channel GEMV's output (the same sums, scaled per chunk instead of
    once: equal within the tolerance, and bit-equal for most outputs)."""
    c, codes, scales = _case(17, 1, 500, 4096, oracle.ACT_BF16)
    gs = np.repeat(scales[:, None], 4096 // 128, axis=1).astype(np.float32)
    y1 = gpu_linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"])
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
    yg = fw.linear(x, torch.from_numpy(codes).to(DEV), torch.from_numpy(gs).to(DEV),
                   torch.from_numpy(c["bias"]).to(DEV))
    torch.cuda.synchronize()
    yg = yg.view(torch.int16).cpu().numpy().view(np.uint16)
    cmp = compare(yg, y1, oracle.ACT_BF16)
    assert cmp["rel_l2"] <= 1e-3 and cmp["bit_equal"] >= 0.95, cmp


# ------------------------------------------------------ weights-ready flag --

@pytest.mark.parametrize("m,n,k", [(1, 4096, 4096), (1, 300, 14336), (8, 3000, 1024), (40, 640, 2048),
                                   (96, 1000, 512)])
def test_weights_ready_flag_gives_the_same_bits(m, n, k):
    """FP8W_FLAG_WEIGHTS_READY only moves the code stream ahead of the
    dependency wait: GEMV, tensor-core kernel and prefill GEMM give the same
    bits with and without it, also right after the kernel that quantised the
    weights (the flag's precondition then holds after a synchronisation)."""
    c = synthetic.random_case(5100 + m, m, n, k)
    w = torch.from_numpy(c["w"]).to(DEV)
    codes, scales = fw.quantize(w)
    torch.cuda.synchronize()
    bias = torch.from_numpy(c["bias"]).to(DEV)
    x = torch.from_numpy(c["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
    a = fw.linear(x, codes, scales, bias)
    b = fw.linear(x, codes, scales, bias, weights_ready=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert fw.device_error() == 0
