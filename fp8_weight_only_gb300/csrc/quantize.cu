// quantize.cu -- kernel K1: per-output-channel e4m3 quantisation.
//
// Page "kadirnar/kernel-agent fp8-weights", section "The contract": one scale
// per row of the [out, in] weight, scale = amax(|row|) / 448, codes =
// round(w / scale) in e4m3, nearest even, clamped to +-448.  The quantisation
// pass itself is page "tensormux Write an FP8 kernel", step 4 (row amax by a
// warp/block reduction, then the saturating cvt.rn.satfinite.e4m3x2.f32).
//
// One CTA per row.  The row is read from HBM once into registers (fp32,
// 16-byte streaming loads, warp-contiguous), reduced to its amax (max is
// order-independent, so the result is exact), and every element is divided
// by the scale with an IEEE fp32 division (not a multiply by 1/scale) and
// converted by the hardware's saturating RNE conversion.  Rows longer than
// the register tile take a second, L2-resident read.  HBM bytes per element:
// 4 read + 1 written.
#include "fp8w_device.cuh"
#include "fp8w_internal.h"

namespace fp8w {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ float block_max_nonneg(float v, float* red) {
    // non-negative floats order like their bit patterns
    uint32_t u = __reduce_max_sync(0xffffffffu, __float_as_uint(v));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = __uint_as_float(u);
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int i = 1; i < kQuantThreads / 32; ++i) m = fmaxf(m, red[i]);
    return m;
}

__device__ __forceinline__ float scale_from_amax(float amax) {
    float s = __fdiv_rn(amax, 448.0f);
    return s == 0.0f ? 1.0f : s;
}

__device__ __forceinline__ uint32_t encode4(float4 v, float s) {
    const uint16_t a = f32x2_to_e4m3x2(__fdiv_rn(v.x, s), __fdiv_rn(v.y, s));
    const uint16_t b = f32x2_to_e4m3x2(__fdiv_rn(v.z, s), __fdiv_rn(v.w, s));
    return static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
}

// Row held in registers: thread t owns float4 chunks t + 256*j, j < VPT.
template <int VPT>
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_reg(const float* __restrict__ w, int64_t k,
                                                                   uint8_t* __restrict__ codes,
                                                                   float* __restrict__ scales) {
    __shared__ float red[kQuantThreads / 32];
    const int64_t row = blockIdx.x;
    const int64_t nf4 = k >> 2;
    const float4* src = reinterpret_cast<const float4*>(w + row * k);
    float4 v[VPT];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(kQuantThreads) * j;
        if (c < nf4) {
            v[j] = ldg_stream_f4(reinterpret_cast<const float*>(src + c));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
        }
    }
    const float s = scale_from_amax(block_max_nonneg(amax, red));
    uint32_t* dst = reinterpret_cast<uint32_t*>(codes + row * k);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(kQuantThreads) * j;
        if (c < nf4) dst[c] = encode4(v[j], s);
    }
    if (threadIdx.x == 0) scales[row] = s;
}

// Any k: pass 1 finds the amax, pass 2 re-reads the (L2-resident) row.
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_two_pass(const float* __restrict__ w, int64_t k,
                                                                        uint8_t* __restrict__ codes,
                                                                        float* __restrict__ scales) {
    __shared__ float red[kQuantThreads / 32];
    const int64_t row = blockIdx.x;
    const int64_t nf4 = k >> 2;
    const float4* src = reinterpret_cast<const float4*>(w + row * k);
    float amax = 0.0f;
    for (int64_t c = threadIdx.x; c < nf4; c += kQuantThreads) {
        const float4 v = src[c];
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    const float s = scale_from_amax(block_max_nonneg(amax, red));
    uint32_t* dst = reinterpret_cast<uint32_t*>(codes + row * k);
    for (int64_t c = threadIdx.x; c < nf4; c += kQuantThreads) dst[c] = encode4(ldg_stream_f4(reinterpret_cast<const float*>(src + c)), s);
    if (threadIdx.x == 0) scales[row] = s;
}

// 16-bit weights (bf16 or fp16) widened exactly to fp32, then the same rule.
// One CTA per row; the second pass re-reads the row from L2.
template <bool kBf16W>
__device__ __forceinline__ void widen8(const uint4 v, float (&f)[8]) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if constexpr (kBf16W) {
            f[2 * e] = bf16_lo_to_f32(u[e]);
            f[2 * e + 1] = bf16_hi_to_f32(u[e]);
        } else {
            f[2 * e] = f16_lo_to_f32(u[e]);
            f[2 * e + 1] = f16_hi_to_f32(u[e]);
        }
    }
}

template <bool kBf16W>
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_16(const uint16_t* __restrict__ w, int64_t k,
                                                                   uint8_t* __restrict__ codes,
                                                                   float* __restrict__ scales) {
    __shared__ float red[kQuantThreads / 32];
    const int64_t row = blockIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(w + row * k);
    const int64_t n8 = k >> 3;
    float amax = 0.0f;
    for (int64_t c = threadIdx.x; c < n8; c += kQuantThreads) {
        float f[8];
        widen8<kBf16W>(src[c], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
    }
    const float s = scale_from_amax(block_max_nonneg(amax, red));
    uint2* dst = reinterpret_cast<uint2*>(codes + row * k);
    for (int64_t c = threadIdx.x; c < n8; c += kQuantThreads) {
        float f[8];
        widen8<kBf16W>(src[c], f);
        dst[c] = make_uint2(encode4(make_float4(f[0], f[1], f[2], f[3]), s),
                            encode4(make_float4(f[4], f[5], f[6], f[7]), s));
    }
    if (threadIdx.x == 0) scales[row] = s;
}

cudaError_t launch_quantize_16(const uint16_t* w, bool bf16, int64_t n, int64_t k, uint8_t* codes, float* scales,
                               cudaStream_t st) {
    if (bf16)
        quantize_rows_16<true><<<static_cast<unsigned>(n), kQuantThreads, 0, st>>>(w, k, codes, scales);
    else
        quantize_rows_16<false><<<static_cast<unsigned>(n), kQuantThreads, 0, st>>>(w, k, codes, scales);
    return cudaGetLastError();
}

template <int VPT>
static cudaError_t launch_reg(const float* w, int64_t n, int64_t k, uint8_t* codes, float* scales,
                              cudaStream_t st) {
    quantize_rows_reg<VPT><<<static_cast<unsigned>(n), kQuantThreads, 0, st>>>(w, k, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const float* w, int64_t n, int64_t k, uint8_t* codes, float* scales,
                            cudaStream_t st) {
    const int64_t nf4 = k / 4;
    const int64_t vpt = (nf4 + kQuantThreads - 1) / kQuantThreads;
    if (vpt <= 1) return launch_reg<1>(w, n, k, codes, scales, st);
    if (vpt <= 2) return launch_reg<2>(w, n, k, codes, scales, st);
    if (vpt <= 4) return launch_reg<4>(w, n, k, codes, scales, st);
    if (vpt <= 8) return launch_reg<8>(w, n, k, codes, scales, st);
    if (vpt <= 14) return launch_reg<14>(w, n, k, codes, scales, st);
    quantize_rows_two_pass<<<static_cast<unsigned>(n), kQuantThreads, 0, st>>>(w, k, codes, scales);
    return cudaGetLastError();
}

// ------------------------------------------------- per-group quantise --
// One scale per run of `group` weights of a row (page "B04 Precision &
// Quantization", section "Post-training quantization versus
// quantization-aware training", the per-group row), each group by the
// per-channel rule above.  A lane takes 4 weights; a group is GL = group / 4
// consecutive lanes of one warp, whose amax is an exact shuffle maximum.
// HBM bytes per element: 4 read + 1 written (+ 4 per group).
//
// kMx: the MX-style form (page "11. Inference with NVFP4/MXFP8", section
// "MXFP8-Style FP8"): group 32 and an E8M0 byte per group, the smallest
// power of two 2^e >= amax / 448, e clamped to [-127, 127]; an all-zero
// group takes 2^0 and an infinite amax the NaN byte 0xFF with NaN codes.

// E8M0 byte of a group's amax (non-negative, NaN already dropped by fmaxf
// unless every weight was NaN).  With amax = (1 + f) 2^E, amax / 448 =
// (1 + f) / 1.75 * 2^(E - 8), a number in (2^(E - 9), 2^(E - 8)] while
// 1 + f <= 1.75 (mantissa field <= 0x600000), else in (2^(E - 8), 2^(E - 7)):
// an integer decision on the bits, no rounding involved.
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
    const uint32_t u = __float_as_uint(amax);
    if (u == 0u || u > 0x7F800000u) return 127u;  // zero (or an all-NaN group, as a zero amax)
    if (u == 0x7F800000u) return 255u;            // infinite
    if (u < 0x00800000u) return 0u;               // subnormal: far below 448 * 2^-127
    const int e = static_cast<int>(u >> 23) - 135 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return e < -127 ? 0u : static_cast<uint32_t>(e + 127);
}

// The fp32 value of an E8M0 byte below 0xFF: 2^(b - 127) (b = 0 is the
// subnormal 2^-127).
__device__ __forceinline__ float mx_scale_value(uint32_t b) {
    return __uint_as_float(b == 0u ? 0x00400000u : b << 23);
}

template <int GL, bool kMx>
__global__ void __launch_bounds__(kQuantThreads) quantize_grouped_kernel(const float* __restrict__ w, int64_t nf4,
                                                                         int gshift, uint8_t* __restrict__ codes,
                                                                         void* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kQuantThreads;
    // a warp-uniform loop: the shuffles below need every lane; nf4 is a
    // multiple of GL, so a group is all in or all out
    for (int64_t base = blockIdx.x * static_cast<int64_t>(kQuantThreads) + (threadIdx.x & ~31); base < nf4;
         base += stride) {
        const int64_t f = base + lane;
        const bool in = f < nf4;
        const float4 v = in ? ldg_stream_f4(w + f * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
        for (int off = GL / 2; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        if constexpr (kMx) {
            const uint32_t b = mx_scale_byte(a);
            if (in) {
                reinterpret_cast<uint32_t*>(codes)[f] = b == 255u ? 0x7F7F7F7Fu : encode4(v, mx_scale_value(b));
                if ((lane & (GL - 1)) == 0) static_cast<uint8_t*>(scales)[(f * 4) >> gshift] = static_cast<uint8_t>(b);
            }
        } else {
            const float sc = scale_from_amax(a);
            if (in) {
                reinterpret_cast<uint32_t*>(codes)[f] = encode4(v, sc);
                if ((lane & (GL - 1)) == 0) static_cast<float*>(scales)[(f * 4) >> gshift] = sc;
            }
        }
    }
}

static unsigned grouped_grid(int64_t nf4, int sms) {
    int64_t blocks = (nf4 + kQuantThreads - 1) / kQuantThreads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    return static_cast<unsigned>(blocks > cap ? cap : blocks);
}

cudaError_t launch_quantize_grouped(const float* w, int64_t n, int64_t k, int group, uint8_t* codes, float* scales,
                                    cudaStream_t st) {
    int sms = 0;
    cudaError_t e = device_sm_count(sms);
    if (e != cudaSuccess) return e;
    const int64_t nf4 = n * k / 4;
    const unsigned g = grouped_grid(nf4, sms);
    const int gshift = group == 32 ? 5 : group == 64 ? 6 : 7;
    if (group == 32) quantize_grouped_kernel<8, false><<<g, kQuantThreads, 0, st>>>(w, nf4, gshift, codes, scales);
    else if (group == 64) quantize_grouped_kernel<16, false><<<g, kQuantThreads, 0, st>>>(w, nf4, gshift, codes, scales);
    else quantize_grouped_kernel<32, false><<<g, kQuantThreads, 0, st>>>(w, nf4, gshift, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_quantize_mx(const float* w, int64_t n, int64_t k, uint8_t* codes, uint8_t* scales,
                               cudaStream_t st) {
    int sms = 0;
    cudaError_t e = device_sm_count(sms);
    if (e != cudaSuccess) return e;
    const int64_t nf4 = n * k / 4;
    quantize_grouped_kernel<8, true><<<grouped_grid(nf4, sms), kQuantThreads, 0, st>>>(w, nf4, 5, codes, scales);
    return cudaGetLastError();
}

// ------------------------------------------------------------ dequantise --
// Page "kadirnar/kernel-agent fp8-weights", section "The contract" (the
// fallback: the decoded codes times the row scale): w[n, k] = e4m3(q[n, k]) *
// scale[n], rounded once to the output type.  The product of a 4-bit and a
// 24-bit significand needs up to 28 bits, so it is carried as hi = fp32
// product plus lo = its exact remainder (fmaf); a 16-bit result rounds hi
// and lets lo decide when hi lies exactly on a rounding midpoint (no other
// midpoint can lie between hi and the exact product: both are within half
// an fp32 ulp, and every 16-bit midpoint is an fp32 number).  HBM bytes per
// element: 1 read + 2 or 4 written.

constexpr int kDequantThreads = 256;

// bf16 nearest-even of the exact product c * s, hi = fp32(c * s).  The
// hardware rounds hi; only when hi sits exactly on a bf16 midpoint (its low
// 16 bits are 0x8000) does the remainder lo = c * s - hi decide.
__device__ __forceinline__ uint16_t exact_to_bf16(float hi, float c, float s) {
    const uint32_t t = __float_as_uint(hi);
    uint16_t r = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    if ((t & 0xFFFFu) == 0x8000u) {
        const float lo = fmaf(c, s, -hi);
        // on lo's side of the midpoint: away from zero when lo has hi's sign
        if (lo != 0.0f) r = static_cast<uint16_t>((t >> 16) + (((__float_as_uint(lo) ^ t) >> 31) ^ 1u));
    }
    return r;
}

// fp16 nearest-even of the exact product c * s, hi = fp32(c * s).  The
// hardware rounds hi; only when hi may sit exactly on a midpoint (its 12 low
// mantissa bits are zero, a necessary condition in fp16's normal and
// subnormal ranges) and the remainder lo = c * s - hi is not zero does the
// exact product need a look.
__device__ __forceinline__ uint16_t exact_to_f16(float hi, float c, float s) {
    const uint16_t r = __half_as_ushort(__float2half_rn(hi));
    const uint32_t t = __float_as_uint(hi);
    if ((t & 0xFFFu) != 0u || (t & 0x7FFFFFFFu) >= 0x7F800000u) return r;
    const float lo = fmaf(c, s, -hi);
    if (lo == 0.0f) return r;
    const uint16_t sign = static_cast<uint16_t>(r & 0x8000u), rm = static_cast<uint16_t>(r & 0x7FFFu);
    const float a = fabsf(hi);
    float back, other;
    uint16_t om;  // the other candidate's magnitude bits
    if (rm == 0x7C00u) {  // rounded to inf: the candidates are 65504 and inf, the midpoint 65520
        back = 65536.0f;
        om = 0x7BFFu;
        other = 65504.0f;
    } else {
        back = __half2float(__ushort_as_half(rm));
        if (back == a) return r;  // hi itself is an fp16 value
        om = static_cast<uint16_t>(a > back ? rm + 1u : rm - 1u);
        other = om == 0x7C00u ? 65536.0f : __half2float(__ushort_as_half(om));
    }
    if (a != 0.5f * (back + other)) return r;  // not a midpoint: hi's rounding is the exact one
    // on the midpoint: the exact product lies on lo's side (away from zero when lo has hi's sign)
    const bool away = (lo > 0.0f) == (hi > 0.0f);
    const uint16_t lower = back < other ? rm : om, upper = back < other ? om : rm;
    return static_cast<uint16_t>(sign | (away ? upper : lower));
}

constexpr int kDequantUnroll = 4;  // chunks a thread has in flight

// OUT: 0 fp32, 1 bf16, 2 fp16.  A chunk is C codes (8 for 16-bit outputs,
// whose 16 bytes a lane stores at once, 4 for fp32), so a warp's loads and
// stores are contiguous; k % 16 == 0, so a chunk lies in one row.  Thread t
// converts the chunks t, t + P, t + 2P, ... (P = the grid's threads),
// kDequantUnroll at a time with all their loads issued first; each of its
// kDequantUnroll sequences tracks its row as it advances (one division per
// sequence).
// SK: 0 one fp32 scale a row; 1 fp32 scales[n, k / g] per group (page "B04
// Precision & Quantization", the per-group row); 2 E8M0 bytes[n, k / 32]
// (page "11. Inference with NVFP4/MXFP8", section "MXFP8-Style FP8"), each
// 2^(b - 127), whose product with a code is exact in fp32 (the smallest,
// 2^-9 * 2^-127, is an fp32 subnormal), so lo is 0 there.  A chunk lies in
// one group (g >= 32, chunks of 8 or 4 aligned).
template <int OUT, int SK>
__global__ void __launch_bounds__(kDequantThreads) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                                      const void* __restrict__ scales, int64_t k,
                                                                      int64_t nchunk, int gshift,
                                                                      void* __restrict__ out) {
    constexpr int U = kDequantUnroll;
    constexpr int C = OUT == 0 ? 4 : 8;
    const int64_t cpr = k / C;  // chunks per row
    const int64_t P = static_cast<int64_t>(gridDim.x) * kDequantThreads;
    const int64_t step = U * P;
    const int64_t srow = step / cpr, scol = step - srow * cpr;
    const int64_t i0 = blockIdx.x * static_cast<int64_t>(kDequantThreads) + threadIdx.x;
    int64_t row[U], col[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t v = i0 + u * P;
        row[u] = v / cpr;
        col[u] = v - row[u] * cpr;
    }
    for (int64_t i = i0; i < nchunk; i += step) {
        uint32_t cw[U][C / 4];
        float sc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = i + u * P;
            if (v < nchunk) {
                if constexpr (C == 8) {
                    const uint2 c2 = __ldcs(reinterpret_cast<const uint2*>(codes) + v);
                    cw[u][0] = c2.x;
                    cw[u][C / 4 - 1] = c2.y;
                } else {
                    cw[u][0] = __ldcs(reinterpret_cast<const uint32_t*>(codes) + v);
                }
                if constexpr (SK == 0) {
                    sc[u] = static_cast<const float*>(scales)[row[u]];
                } else {
                    const int64_t gi = row[u] * (k >> gshift) + ((col[u] * C) >> gshift);
                    if constexpr (SK == 1) {
                        sc[u] = static_cast<const float*>(scales)[gi];
                    } else {
                        const uint32_t b = static_cast<const uint8_t*>(scales)[gi];
                        sc[u] = __uint_as_float(b == 0u ? 0x00400000u : b == 255u ? 0x7FFFFFFFu : b << 23);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = i + u * P;
            if (v >= nchunk) break;
            const float s = sc[u];
            uint32_t o[C];
#pragma unroll
            for (int q = 0; q < C / 4; ++q) {
                uint32_t p01, p23;
                e4m3x4_to_f16x2(cw[u][q], p01, p23);
                const float c[4] = {f16_lo_to_f32(p01), f16_hi_to_f32(p01), f16_lo_to_f32(p23), f16_hi_to_f32(p23)};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float hi = __fmul_rn(c[e], s);
                    if constexpr (OUT == 0) {
                        o[4 * q + e] = __float_as_uint(hi);
                    } else {
                        o[4 * q + e] = OUT == 1 ? exact_to_bf16(hi, c[e], s) : exact_to_f16(hi, c[e], s);
                    }
                }
            }
            uint4* dst = reinterpret_cast<uint4*>(out) + v;
            if constexpr (OUT == 0) {
                __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
            } else {
                __stcs(dst, make_uint4(o[0] | (o[1] << 16), o[2] | (o[3] << 16), o[4] | (o[5] << 16),
                                       o[6] | (o[7] << 16)));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            row[u] += srow;
            col[u] += scol;
            if (col[u] >= cpr) {
                col[u] -= cpr;
                ++row[u];
            }
        }
    }
}

template <int SK>
static cudaError_t launch_dq(const uint8_t* codes, const void* scales, int64_t n, int64_t k, int gshift,
                             int out_dtype, void* w, cudaStream_t st) {
    int sms = 0;
    cudaError_t e = device_sm_count(sms);
    if (e != cudaSuccess) return e;
    const int64_t nchunk = n * (k / (out_dtype == 0 ? 4 : 8));
    int64_t blocks = (nchunk + kDequantThreads * kDequantUnroll - 1) / (kDequantThreads * kDequantUnroll);
    const int64_t cap = static_cast<int64_t>(sms) * 8;  // up to 8 CTAs of 256 threads per SM
    if (blocks > cap) blocks = cap;
    const unsigned g = static_cast<unsigned>(blocks);
    if (out_dtype == 1)
        dequantize_kernel<1, SK><<<g, kDequantThreads, 0, st>>>(codes, scales, k, nchunk, gshift, w);
    else if (out_dtype == 2)
        dequantize_kernel<2, SK><<<g, kDequantThreads, 0, st>>>(codes, scales, k, nchunk, gshift, w);
    else
        dequantize_kernel<0, SK><<<g, kDequantThreads, 0, st>>>(codes, scales, k, nchunk, gshift, w);
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* codes, const float* scales, int64_t n, int64_t k, int out_dtype,
                              void* w, cudaStream_t st) {
    return launch_dq<0>(codes, scales, n, k, 0, out_dtype, w, st);
}

cudaError_t launch_dequantize_grouped(const uint8_t* codes, const void* scales, bool e8m0, int group, int64_t n,
                                      int64_t k, int out_dtype, void* w, cudaStream_t st) {
    const int gshift = group == 32 ? 5 : group == 64 ? 6 : 7;
    return e8m0 ? launch_dq<2>(codes, scales, n, k, 5, out_dtype, w, st)
                : launch_dq<1>(codes, scales, n, k, gshift, out_dtype, w, st);
}

}  // namespace fp8w
