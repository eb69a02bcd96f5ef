// gemv.cu -- kernel K2: the M = 1 linear layer (GEMV) on CUDA cores.
//
// Page "kadirnar/kernel-agent fp8-weights", section "Dequantise in
// registers": 128-bit streaming loads of 16 e4m3 codes past L1
// (ld.global.nc.L1::no_allocate), hardware e4m3x2 -> f16x2 conversion in
// registers, fp32 FMA, warp-shuffle reduction, scale (and bias) applied once
// per output in the epilogue.
//
// GB300 layout of the work: the reduction dimension is split over the whole
// CTA (thread t owns the 16-code chunks t, t+T, t+2T, ... of every row), so
// each thread keeps its slice of x in fp32 registers for the life of the CTA
// and the codes are the only HBM stream.  A persistent grid of
// (SMs x resident CTAs) walks the rows interleaved (CTA b takes rows
// b, b+G, b+2G, ...), R rows per step, which keeps the per-SM work within
// one row of equal.  Per step each thread has R x C independent 16-byte
// loads in flight.  The R partial sums are reduced across each warp by a
// transposing shuffle tree (R-1 + log2(32/R) shuffles for R rows) and across
// warps through shared memory.  HBM bytes per output channel: K (codes) + 4
// (scale) + 4 (bias) + 2 (y); x (2K bytes) is read once per CTA from L2.
#include <mutex>

#include "fp8w_device.cuh"
#include "fp8w_internal.h"

namespace fp8w {

constexpr int kGemvMaxThreads = 256;

// Reduce R per-thread values across a warp.  On return, lane l holds the
// warp total of row l / (32 / R) if l % (32 / R) == 0.
template <int R>
__device__ __forceinline__ float warp_reduce_rows(float (&p)[R]) {
    const int lane = threadIdx.x & 31;
    float v[R];
#pragma unroll
    for (int i = 0; i < R; ++i) v[i] = p[i];
    int count = R;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (count > 1) {
            const bool upper = (lane & off) != 0;
            const int half = count / 2;
#pragma unroll
            for (int i = 0; i < R / 2; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            count = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
    return v[0];
}

// x chunk (16 activations) -> fp32 registers.
template <bool kBf16>
__device__ __forceinline__ void load_x_chunk(const uint16_t* x, int64_t chunk, float (&xr)[16]) {
    const uint4* p = reinterpret_cast<const uint4*>(x + chunk * 16);
    const uint4 a = __ldg(p), b = __ldg(p + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if constexpr (kBf16) {
            xr[2 * i] = bf16_lo_to_f32(w[i]);
            xr[2 * i + 1] = bf16_hi_to_f32(w[i]);
        } else {
            xr[2 * i] = f16_lo_to_f32(w[i]);
            xr[2 * i + 1] = f16_hi_to_f32(w[i]);
        }
    }
}

// acc += sum over 16 codes of x * e4m3(code).
__device__ __forceinline__ float dot16(const uint4 c, const float (&xr)[16], float acc) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h01, h23;
        e4m3x4_to_f16x2(w[q], h01, h23);
        acc = fmaf(xr[4 * q + 0], f16_lo_to_f32(h01), acc);
        acc = fmaf(xr[4 * q + 1], f16_hi_to_f32(h01), acc);
        acc = fmaf(xr[4 * q + 2], f16_lo_to_f32(h23), acc);
        acc = fmaf(xr[4 * q + 3], f16_hi_to_f32(h23), acc);
    }
    return acc;
}

template <int C, int R, bool kBf16>
__global__ void __launch_bounds__(kGemvMaxThreads) gemv_kernel(const uint16_t* __restrict__ x,
                                                               const uint8_t* __restrict__ codes,
                                                               const float* __restrict__ scales,
                                                               const float* __restrict__ bias,
                                                               uint16_t* __restrict__ y, int64_t n, int64_t k) {
    __shared__ float red[2][R][kGemvMaxThreads / 32];
    const int T = blockDim.x;
    const int nwarps = T >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nchunks = k >> 4;
    const int64_t per_pass = static_cast<int64_t>(T) * C;
    const int64_t npasses = (nchunks + per_pass - 1) / per_pass;
    const int64_t G = gridDim.x;

    float xr[C][16];
    auto load_x = [&](int64_t pass) {
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const int64_t ch = pass * per_pass + threadIdx.x + static_cast<int64_t>(T) * j;
            if (ch < nchunks) {
                load_x_chunk<kBf16>(x, ch, xr[j]);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) xr[j][e] = 0.0f;
            }
        }
    };
    if (npasses == 1) load_x(0);

    int buf = 0;
    for (int64_t step = 0;; ++step) {
        const int64_t first = blockIdx.x + G * step * R;
        if (first >= n) break;
        float p[R];
#pragma unroll
        for (int r = 0; r < R; ++r) p[r] = 0.0f;
        for (int64_t pass = 0; pass < npasses; ++pass) {
            if (npasses > 1) load_x(pass);
            uint4 cw[R][C];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = first + G * r;
#pragma unroll
                for (int j = 0; j < C; ++j) {
                    const int64_t ch = pass * per_pass + threadIdx.x + static_cast<int64_t>(T) * j;
                    if (row < n && ch < nchunks)
                        cw[r][j] = ldg_stream_v4(codes + row * k + ch * 16);
                    else
                        cw[r][j] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int j = 0; j < C; ++j) p[r] = dot16(cw[r][j], xr[j], p[r]);
        }
        const float wsum = warp_reduce_rows<R>(p);
        constexpr int kStride = 32 / R;
        if ((lane % kStride) == 0) red[buf][lane / kStride][warp] = wsum;
        __syncthreads();
        if (threadIdx.x < R) {
            const int64_t row = first + G * threadIdx.x;
            if (row < n) {
                float acc = 0.0f;
                for (int w = 0; w < nwarps; ++w) acc += red[buf][threadIdx.x][w];
                const float b = bias ? bias[row] : 0.0f;
                y[row] = round_out<kBf16>(fmaf(acc, scales[row], b));
            }
        }
        buf ^= 1;
    }
}

template <int C, int R, bool kBf16>
static cudaError_t launch_cfg(const LinearArgs& a, int threads, cudaStream_t st) {
    auto kern = gemv_kernel<C, R, kBf16>;
    // resident CTAs per SM, per device and block size (8 warp counts)
    static int cache[64][kGemvMaxThreads / 32 + 1];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = 0, occ = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        int& slot = cache[dev][threads / 32];
        if (slot == 0) {
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, 0);
            if (e != cudaSuccess) return e;
            slot = sms * (occ < 1 ? 1 : occ);
        }
        sms = slot;
        occ = 1;
    }
    int64_t grid = static_cast<int64_t>(sms) * occ;
    if (grid > a.n) grid = a.n;
    kern<<<static_cast<unsigned>(grid), threads, 0, st>>>(static_cast<const uint16_t*>(a.x), a.codes, a.scales,
                                                          a.bias, static_cast<uint16_t*>(a.y), a.n, a.k);
    return cudaGetLastError();
}

template <bool kBf16>
static cudaError_t launch_dt(const LinearArgs& a, cudaStream_t st) {
    const int64_t nchunks = a.k / 16;
    // chunks per thread: fit the row in one pass of <= 256 threads when possible
    if (nchunks <= 256) {
        const int threads = static_cast<int>(((nchunks + 31) / 32) * 32);
        return launch_cfg<1, 8, kBf16>(a, threads, st);
    }
    if (nchunks <= 512) {
        const int threads = static_cast<int>((((nchunks + 1) / 2 + 31) / 32) * 32);
        return launch_cfg<2, 4, kBf16>(a, threads, st);
    }
    int threads = static_cast<int>((((nchunks + 3) / 4 + 31) / 32) * 32);
    if (threads > kGemvMaxThreads) threads = kGemvMaxThreads;
    return launch_cfg<4, 2, kBf16>(a, threads, st);
}

cudaError_t launch_gemv(const LinearArgs& a, cudaStream_t st) {
    return a.act == 1 ? launch_dt<true>(a, st) : launch_dt<false>(a, st);
}

}  // namespace fp8w
