"""fp8w_linear_noalloc, the entry point for callers that cannot allocate
device memory while they run, against fp8w_linear and the oracle, through
the C ABI.  No path of the library uses scratch memory, so the two entry
points must agree bit for bit.

Named to be collected last: it must pass in a fresh process and after every
other test has run.  Each case makes two calls in a row with different
inputs, so the second one would expose any state the first left behind.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synthetic
from tests.parity import COSINE_MIN, REL_L2_MAX, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import fp8_weight_only_gb300 as fw  # noqa: E402

DEV = torch.device("cuda:0")

# (m, n, k, act): a tile split over a cluster, whole tiles, the GEMV path,
# 40 rows (one 64-token launch), fp16, and
# the gate weight (clusters sharing tiles)
CASES = [(8, 1024, 4096, oracle.ACT_BF16), (32, 4096, 1024, oracle.ACT_BF16), (1, 2048, 1024, oracle.ACT_BF16),
         (40, 640, 2048, oracle.ACT_BF16), (22, 4096, 1024, oracle.ACT_F16), (8, 14336, 4096, oracle.ACT_BF16)]


def _inputs(seed, m, n, k, act):
    c = synthetic.random_case(seed, m, n, k, act=act)
    w = torch.from_numpy(c["w"]).to(DEV)
    codes, scales = fw.quantize(w)
    bias = torch.from_numpy(c["bias"]).to(DEV)
    dt = torch.bfloat16 if act == oracle.ACT_BF16 else torch.float16
    x = torch.from_numpy(np.ascontiguousarray(c["x"]).view(np.int16)).to(DEV).view(dt)
    return x, codes, scales, bias, c


def _noalloc(x, codes, scales, bias):
    m, k = x.shape
    n = codes.shape[0]
    y = torch.full((m, n), float("nan"), dtype=x.dtype, device=DEV)
    act = oracle.ACT_BF16 if x.dtype == torch.bfloat16 else oracle.ACT_F16
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    st = fw.lib().fp8w_linear_noalloc(ctypes.c_void_p(x.data_ptr()), act, m, k, ctypes.c_void_p(codes.data_ptr()),
                                      ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(bias.data_ptr()), n,
                                      ctypes.c_void_p(y.data_ptr()), stream)
    assert st == 0, fw.lib().fp8w_status_string(st)
    return y


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("m,n,k,act", CASES)
def test_noalloc_matches_fp8w_linear_and_the_oracle_twice(m, n, k, act):
    for call, seed in enumerate((7001 + m, 7002 + m)):
        x, codes, scales, bias, c = _inputs(seed, m, n, k, act)
        y = _noalloc(x, codes, scales, bias)
        ref = fw.linear(x, codes, scales, bias)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(y), _bits(ref)), call
        rc, rs = oracle.quantize(c["w"])
        want = oracle.linear(c["x"], act, rc, rs, c["bias"], threads=oracle.host_cores())
        cmp = compare(_bits(y), want, act)
        assert cmp["finite"], (call, cmp)
        assert cmp["rel_l2"] <= REL_L2_MAX and cmp["min_cosine"] >= COSINE_MIN, (call, cmp)
    assert fw.device_error() == 0
