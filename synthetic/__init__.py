"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and lays them out; it holds none of
the layer's arithmetic (no quantisation, no rounding of results, no dot
products).  Activations are drawn in fp32 and converted to bf16 / fp16 by
the library conversions of torch (bf16) and numpy (fp16).

Workloads (weights are [N, K] = nn.Linear [out, in], row-major):
  tiny_gemv       M=1,  K=1024,  N=1024,  x bf16 N(0,1), W N(0,0.02), bias N(0,0.01)
  outlier_gemv    M=1,  K=4096,  N=4096,  x bf16 N(0,1), W 0.02*t(df=3) with
                  round(1% of N) rows x50, no bias
  skinny_sweep    M in {2,4,8,16,32}, K=4096, N=14336, x bf16 N(0,1),
                  W N(0,0.02), bias N(0,0.01)
  fp16_template   M=22, K=1024, N=4096, x fp16 U(-1,1), W N(0,0.05), bias N(0,0.01)
  decode_stack    an 8B-style block (hidden 4096, 32 q / 8 kv heads of 128,
                  intermediate 14336): q 4096x4096, k 1024x4096, v 1024x4096,
                  o 4096x4096, gate 14336x4096, up 14336x4096, down 4096x14336,
                  W N(0,0.02), bias N(0,0.01), x bf16 N(0,1) at M in {1,8,32}
"""
import numpy as np

ACT_BF16 = 1
ACT_F16 = 2

# (name, N, K) of the decode-stack block, in the order the block runs them.
DECODE_STACK = (
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 14336, 4096),
    ("up", 14336, 4096),
    ("down", 4096, 14336),
)
DECODE_STACK_M = (1, 8, 32)
SKINNY_M = (2, 4, 8, 16, 32)


def to_bf16_bits(a32: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16) via torch's RNE conversion."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def to_f16_bits(a32: np.ndarray) -> np.ndarray:
    """fp32 array -> fp16 bit patterns (uint16) via numpy's RNE conversion."""
    return np.ascontiguousarray(a32, dtype=np.float32).astype(np.float16).view(np.uint16)


def weight_normal(seed: int, n: int, k: int, std: float) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, k), dtype=np.float32) * np.float32(std)).astype(np.float32)


def weight_outlier(seed: int, n: int, k: int) -> np.ndarray:
    """0.02 * Student-t(df=3), with round(0.01*N) seeded rows scaled by 50."""
    rng = np.random.default_rng(seed)
    w = (rng.standard_t(3, size=(n, k)) * 0.02).astype(np.float32)
    rows = rng.permutation(n)[: int(round(0.01 * n))]
    w[rows] *= np.float32(50.0)
    return w


def bias_normal(seed: int, n: int, std: float = 0.01) -> np.ndarray:
    rng = np.random.default_rng(seed + 7919)
    return (rng.standard_normal(n, dtype=np.float32) * np.float32(std)).astype(np.float32)


def act_normal_bf16(seed: int, m: int, k: int) -> np.ndarray:
    rng = np.random.default_rng(seed + 104729)
    return to_bf16_bits(rng.standard_normal((m, k), dtype=np.float32))


def act_uniform_f16(seed: int, m: int, k: int) -> np.ndarray:
    rng = np.random.default_rng(seed + 104729)
    return to_f16_bits(rng.uniform(-1.0, 1.0, size=(m, k)).astype(np.float32))


def case(name: str, m: int = None, matrix: str = None):
    """Inputs of one workload: dict(x bits, act, W fp32, bias or None, M, N, K)."""
    if name == "tiny_gemv":
        m, n, k, seed = 1, 1024, 1024, 1001
        return dict(x=act_normal_bf16(seed, m, k), act=ACT_BF16,
                    w=weight_normal(seed, n, k, 0.02), bias=bias_normal(seed, n),
                    m=m, n=n, k=k)
    if name == "outlier_gemv":
        m, n, k, seed = 1, 4096, 4096, 1002
        return dict(x=act_normal_bf16(seed, m, k), act=ACT_BF16,
                    w=weight_outlier(seed, n, k), bias=None, m=m, n=n, k=k)
    if name == "skinny_sweep":
        m = 32 if m is None else m
        n, k, seed = 14336, 4096, 1003
        return dict(x=act_normal_bf16(seed + m, m, k), act=ACT_BF16,
                    w=weight_normal(seed, n, k, 0.02), bias=bias_normal(seed, n),
                    m=m, n=n, k=k)
    if name == "fp16_template":
        m, n, k, seed = 22, 4096, 1024, 1004
        return dict(x=act_uniform_f16(seed, m, k), act=ACT_F16,
                    w=weight_normal(seed, n, k, 0.05), bias=bias_normal(seed, n),
                    m=m, n=n, k=k)
    if name == "decode_stack":
        m = 1 if m is None else m
        idx = [s[0] for s in DECODE_STACK].index(matrix)
        _, n, k = DECODE_STACK[idx]
        seed = 1005 + 10 * idx
        return dict(x=act_normal_bf16(seed + 1000 * m, m, k), act=ACT_BF16,
                    w=weight_normal(seed, n, k, 0.02), bias=bias_normal(seed, n),
                    m=m, n=n, k=k)
    raise KeyError(name)


def random_case(seed: int, m: int, n: int, k: int, act: int = ACT_BF16,
                std: float = 0.02, with_bias: bool = True):
    """A generic seeded case of any shape (for ragged and edge shapes)."""
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((n, k), dtype=np.float32) * np.float32(std)).astype(np.float32)
    xf = rng.standard_normal((m, k), dtype=np.float32)
    x = to_f16_bits(xf) if act == ACT_F16 else to_bf16_bits(xf)
    bias = (rng.standard_normal(n, dtype=np.float32) * np.float32(0.01)).astype(np.float32) \
        if with_bias else None
    return dict(x=x, act=act, w=w, bias=bias, m=m, n=n, k=k)
