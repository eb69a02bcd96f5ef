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

}  // namespace fp8w
