// gemv.cu -- kernel K2: the M = 1 linear layer (GEMV) on CUDA cores.
//
// Page "kadirnar/kernel-agent fp8-weights", section "Dequantise in
// registers": the codes are streamed once past L1, each pair is converted
// to f16x2 by the hardware e4m3x2 conversion (exact) and widened to fp32,
// fp32 FMA against x, a shuffle reduction, scale (and bias) applied once per
// output in the epilogue.
//
// GB300 layout of the work:
//  * Persistent grid, one CTA per SM; CTA c owns the contiguous rows
//    [c*N/P, (c+1)*N/P), so every SM streams the same bytes (+-1 row).
//  * The last warp moves R whole rows per stage (R*K contiguous bytes) with
//    one 1-D TMA bulk copy into a shared-memory ring of ~160 KB, so ~160 KB
//    per SM is in flight without occupying registers.
//  * 16 compute warps (512 threads).  A row's 16-code chunks are spread over
//    T_row threads (G = 512 / T_row row groups work on different rows);
//    each thread keeps its chunks of x in fp32 registers for the whole
//    kernel, so after start-up the codes are the only HBM stream.
//  * Per stage, each group reduces its rows with a transposing shuffle tree
//    and shared memory; one thread per row applies scale and bias.
// HBM bytes per output channel: K (codes) + 4 (scale) + 4 (bias) + 2 (y).
// K > 16384 (a row longer than a stage) runs the chunked variant at the end
// of this file.
#include <mutex>

#include "fp8w_device.cuh"
#include "fp8w_internal.h"

namespace fp8w {

static __device__ int g_gemv_error;

constexpr int kGemvComputeThreads = 512;
constexpr int kGemvThreads = kGemvComputeThreads + 32;
constexpr int kGemvRingBytes = 160 * 1024;
constexpr int kGemvMaxRowsPerStage = 32;
constexpr int kGemvMaxStages = 16;
constexpr int kGemvMaxK = 16384;

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

// f16x2 -> two fp32 (halves selected in the register, no extraction).
__device__ __forceinline__ void f16x2_to_f32x2(uint32_t h, float& lo, float& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
}

// acc += sum over 16 codes of x * e4m3(code).
__device__ __forceinline__ float dot16(const uint4 c, const float (&xr)[16], float acc) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h01, h23;
        e4m3x4_to_f16x2(w[q], h01, h23);
        float a, b, c2, d;
        f16x2_to_f32x2(h01, a, b);
        f16x2_to_f32x2(h23, c2, d);
        acc = fmaf(xr[4 * q + 0], a, acc);
        acc = fmaf(xr[4 * q + 1], b, acc);
        acc = fmaf(xr[4 * q + 2], c2, acc);
        acc = fmaf(xr[4 * q + 3], d, acc);
    }
    return acc;
}

__device__ __forceinline__ void compute_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kGemvComputeThreads) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

struct GemvGeom {
    int rows_per_stage;  // R
    int stages;          // S
    int t_row;           // threads per row
    int groups;          // 512 / t_row
    uint32_t stage_bytes;
};

// C = chunks per thread, RPG = rows per group per stage (R / groups).
template <int C, int RPG, bool kBf16>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                const float* __restrict__ bias, uint16_t* __restrict__ y, int64_t n, int64_t k, GemvGeom geo) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t ring = smem_u32(smem);
    const uint32_t bar_full = ring + kGemvRingBytes;                 // [S]
    const uint32_t bar_empty = bar_full + 8 * kGemvMaxStages;       // [S]
    float* red = reinterpret_cast<float*>(smem + kGemvRingBytes + 16 * kGemvMaxStages);  // [R][16 warps]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + kGemvMaxRowsPerStage * 16);
    // written only by compute threads before a compute barrier, so they all
    // read the same value after it and leave the loop together
    volatile int* cmp_abort = abort_flag + 1;

    const int S = geo.stages, R = geo.rows_per_stage;
    const int64_t P = gridDim.x;
    const int64_t row0 = blockIdx.x * n / P, row1 = (blockIdx.x + 1) * n / P;
    const int64_t nst = (row1 - row0 + R - 1) / R;
    const int warp = threadIdx.x >> 5;
    const int nwarps_compute = kGemvComputeThreads / 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, nwarps_compute);
        }
        *abort_flag = 0;
        *cmp_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the next kernel in the stream may start its prologue; it waits for
    // this grid before touching global memory
    pdl_launch_dependents();

    if (warp == nwarps_compute) {
        // ---------------------------------------------------- producer --
        if ((threadIdx.x & 31) == 0) {
            const uint64_t pol = policy_evict_first();
            pdl_wait();  // the codes may come from the previous kernel
            int64_t issued = 0;
            int s = 0;
            uint32_t ph = 0;  // stage slot and its phase, advanced without division
            for (int64_t st = 0; st < nst; ++st) {
                if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    atomicCAS(&g_gemv_error, 0, kErrWaitSlot);
                    break;
                }
                const int64_t r0 = row0 + st * R;
                const int64_t rows = (row1 - r0) < R ? (row1 - r0) : R;
                const uint32_t bytes = static_cast<uint32_t>(rows * k);
                mbar_arrive_expect_tx(bar_full + 8 * s, bytes);
                bulk_load(ring + s * geo.stage_bytes, codes + r0 * k, bytes, bar_full + 8 * s, pol);
                ++issued;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag) {
                for (int64_t st = (issued > S ? issued - S : 0); st < issued; ++st)
                    if (!mbar_wait_drain(bar_full + 8 * (st % S), static_cast<uint32_t>((st / S) & 1)))
                        atomicCAS(&g_gemv_error, 0, kErrWaitDrain);
            }
        }
        return;
    }

    // -------------------------------------------------------- compute --
    const int t = threadIdx.x;
    const int g = t / geo.t_row, tr = t % geo.t_row;
    const int lane = t & 31;
    const int64_t nchunks = k >> 4;
    pdl_wait();  // x, scales and bias may come from the previous kernel, and y may still be read by it
    float xr[C][16];
#pragma unroll
    for (int j = 0; j < C; ++j) {
        const int64_t ch = tr + static_cast<int64_t>(geo.t_row) * j;
        if (ch < nchunks) {
            load_x_chunk<kBf16>(x, ch, xr[j]);
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) xr[j][e] = 0.0f;
        }
    }
    const int warps_per_row = geo.t_row >> 5;
    const int warp_in_group = (t % geo.t_row) >> 5;
    int s = 0;
    uint32_t ph = 0;
    for (int64_t st = 0; st < nst; ++st) {
        const int64_t r0 = row0 + st * R;
        // the epilogue threads fetch their row's scale and bias before the
        // stage's data arrives, off the critical path
        float sc = 0.0f, b = 0.0f;
        if (t < R && r0 + t < row1) {
            sc = scales[r0 + t];
            b = bias ? bias[r0 + t] : 0.0f;
        }
        if (!mbar_wait_warp(bar_full + 8 * s, ph, abort_flag)) {
            *cmp_abort = 1;
            *abort_flag = 1;
            atomicCAS(&g_gemv_error, 0, kErrWaitTma);
        }
        compute_bar();
        if (*cmp_abort) break;
        const uint8_t* stage = smem + s * geo.stage_bytes;
        float p[RPG];
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            p[i] = 0.0f;
            const int rr = g + i * geo.groups;  // row within the stage
            if (r0 + rr < row1) {
                const uint8_t* rowp = stage + static_cast<int64_t>(rr) * k;
#pragma unroll
                for (int j = 0; j < C; ++j) {
                    const int64_t ch = tr + static_cast<int64_t>(geo.t_row) * j;
                    if (ch < nchunks) p[i] = dot16(*reinterpret_cast<const uint4*>(rowp + ch * 16), xr[j], p[i]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
        const float wsum = warp_reduce_rows<RPG>(p);
        constexpr int kStride = 32 / RPG;
        if ((lane % kStride) == 0) red[(g + (lane / kStride) * geo.groups) * 16 + warp_in_group] = wsum;
        compute_bar();
        if (t < R) {
            const int64_t row = r0 + t;
            if (row < row1) {
                float acc = 0.0f;
                for (int w = 0; w < warps_per_row; ++w) acc += red[t * 16 + w];
                y[row] = round_out<kBf16>(fmaf(acc, sc, b));
            }
        }
        // red is rewritten only after the next stage's first compute_bar
    }
}

// ------------------------------------------------ long rows (K > 16384) --
// Rows longer than a stage: one warp-contiguous pass per row, x re-read
// from L2 per row (correct, not tuned).
template <bool kBf16>
__global__ void __launch_bounds__(256) gemv_long_kernel(const uint16_t* __restrict__ x,
                                                        const uint8_t* __restrict__ codes,
                                                        const float* __restrict__ scales,
                                                        const float* __restrict__ bias, uint16_t* __restrict__ y,
                                                        int64_t n, int64_t k) {
    __shared__ float red[8];
    const int64_t nchunks = k >> 4;
    for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
        float acc = 0.0f;
        for (int64_t ch = threadIdx.x; ch < nchunks; ch += 256) {
            float xr[16];
            load_x_chunk<kBf16>(x, ch, xr);
            acc = dot16(ldg_stream_v4(codes + row * k + ch * 16), xr, acc);
        }
        float v[1] = {acc};
        const float wsum = warp_reduce_rows<1>(v);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = wsum;
        __syncthreads();
        if (threadIdx.x == 0) {
            float s = 0.0f;
            for (int w = 0; w < 8; ++w) s += red[w];
            const float b = bias ? bias[row] : 0.0f;
            y[row] = round_out<kBf16>(fmaf(s, scales[row], b));
        }
        __syncthreads();
    }
}

static constexpr uint32_t gemv_smem_bytes() {
    return kGemvRingBytes + 16 * kGemvMaxStages + kGemvMaxRowsPerStage * 16 * 4 + 16 + 128;  // + flags, align
}

template <int C, int RPG, bool kBf16>
static cudaError_t launch_cfg(const LinearArgs& a, const GemvGeom& geo, int sms, cudaStream_t st) {
    auto kern = gemv_kernel<C, RPG, kBf16>;
    static std::once_flag attr_once[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, gemv_smem_bytes());
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t grid = a.n < sms ? a.n : sms;
    // programmatic dependent launch: set-up overlaps the previous kernel's tail
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = gemv_smem_bytes();
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint16_t*>(a.x), a.codes, a.scales, a.bias,
                              static_cast<uint16_t*>(a.y), a.n, a.k, geo);
}

template <bool kBf16>
static cudaError_t launch_dt(const LinearArgs& a, cudaStream_t st) {
    int sms = 0;
    cudaError_t e = device_sm_count(sms);
    if (e != cudaSuccess) return e;
    if (a.k > kGemvMaxK) {
        const int64_t grid = a.n < 4 * sms ? a.n : 4 * sms;
        gemv_long_kernel<kBf16><<<static_cast<unsigned>(grid), 256, 0, st>>>(
            static_cast<const uint16_t*>(a.x), a.codes, a.scales, a.bias, static_cast<uint16_t*>(a.y), a.n, a.k);
        return cudaGetLastError();
    }
    const int64_t nchunks = a.k / 16;
    GemvGeom geo;
    geo.t_row = static_cast<int>(nchunks >= kGemvComputeThreads ? kGemvComputeThreads : ((nchunks + 31) / 32) * 32);
    // t_row must divide 512: round up to 32, 64, 128, 256 or 512
    int tr = 32;
    while (tr < geo.t_row) tr *= 2;
    geo.t_row = tr;
    geo.groups = kGemvComputeThreads / geo.t_row;
    // ~16 KB per stage: rows = groups x (1, 2 or 4), at most 32
    int64_t target = 16384 / a.k;
    if (target > kGemvMaxRowsPerStage) target = kGemvMaxRowsPerStage;
    int rpg_sel = 1;
    while (rpg_sel < 4 && static_cast<int64_t>(geo.groups) * rpg_sel * 2 <= target) rpg_sel *= 2;
    const int rows = geo.groups * rpg_sel;
    geo.rows_per_stage = rows;
    geo.stage_bytes = static_cast<uint32_t>(((rows * a.k + 127) / 128) * 128);
    geo.stages = static_cast<int>(kGemvRingBytes / geo.stage_bytes);
    if (geo.stages > kGemvMaxStages) geo.stages = kGemvMaxStages;
    const int rpg = rows / geo.groups;
    const int c = static_cast<int>((nchunks + geo.t_row - 1) / geo.t_row);
    if (c == 1 && rpg == 1) return launch_cfg<1, 1, kBf16>(a, geo, sms, st);
    if (c == 1 && rpg == 2) return launch_cfg<1, 2, kBf16>(a, geo, sms, st);
    if (c == 1 && rpg == 4) return launch_cfg<1, 4, kBf16>(a, geo, sms, st);
    if (c == 2 && rpg == 1) return launch_cfg<2, 1, kBf16>(a, geo, sms, st);
    return cudaErrorNotSupported;
}

cudaError_t launch_gemv(const LinearArgs& a, cudaStream_t st) {
    return a.act == 1 ? launch_dt<true>(a, st) : launch_dt<false>(a, st);
}

int read_gemv_device_error() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof v) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof zero);
    return v;
}

}  // namespace fp8w
