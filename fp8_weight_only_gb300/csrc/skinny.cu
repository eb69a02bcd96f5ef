// skinny.cu -- kernel K3: the 2 <= M <= 32 linear layer on the tcgen05 tensor
// cores, "swap-AB": the weight channels are the 128-row A operand and the
// tokens the narrow B operand.
//
// Page "kadirnar/kernel-agent fp8-weights", section "Dequantise in
// registers" (skinny GEMM: the weight as the A operand, 16-bit MMA in the
// activations' type, each code converted once and reused for every token,
// several channel tiles and split-K to share the activation traffic).  That
// design is written for mma.sync on sm_80..sm_120; this one is built for
// sm_103a:
//
//  * A CTA owns one tile of 128 output channels and a contiguous range of
//    k-blocks (128 k each).  CTAs that split the same tile along k form one
//    thread-block cluster (1, 2, 4 or 8 CTAs) and reduce their fp32 partial
//    tiles through distributed shared memory, so no global scratch is used.
//  * Warp 0 streams, per k-block, the 128 x 128 code tile and the M x 128
//    activation tile into shared memory with TMA (128-byte swizzle; rows past
//    N or M and k past K are zero-filled), several stages ahead.
//  * Warps 2..5 dequantise: thread r reads the 128 codes of channel r
//    (bank-conflict-free through the swizzle), converts them exactly to
//    bf16 / fp16 in registers and writes them with tcgen05.st into TMEM,
//    where they form the A operand of the MMA (A from tensor memory, so the
//    dequantised weight never passes through shared memory).
//  * Warp 1 issues tcgen05.mma.kind::f16 (M = 128, N = 16 or 32 tokens,
//    K = 16) with A in TMEM, B (activations, K-major) in shared memory and
//    the fp32 accumulator in TMEM, and returns each stage with
//    tcgen05.commit.
//  * Epilogue: the accumulator is read back with tcgen05.ld (thread r holds
//    channel r for every token), reduced over the cluster if split, and
//    y = round(fma(acc, scale, bias)) is stored.
//
// Every wait is bounded in time: on a timeout the CTA records an error code,
// raises a shared abort flag, drains its in-flight copies and MMAs, frees
// TMEM and finishes.
#include <mutex>

#include "fp8w_device.cuh"
#include "fp8w_internal.h"

namespace fp8w {

static __device__ int g_skinny_error;

constexpr int kThreads = 192;          // 6 warps
constexpr int kTileN = 128;            // output channels per CTA (MMA M)
constexpr int kBlockK = 128;           // k per stage
constexpr int kStages = 4;             // shared-memory (TMA) stages
constexpr int kTmemStages = 3;         // TMEM A-operand stages
constexpr int kTmemCols = 256;         // allocation per CTA (<= 2 CTAs per SM)
constexpr int kTmemAStageCols = kBlockK / 2;  // 16-bit pairs per 32-bit column
constexpr int kTmemDCol = kTmemStages * kTmemAStageCols;  // 192
constexpr uint32_t kCodeStageBytes = kTileN * kBlockK;   // 16 KB

template <int NT>
struct SkinnySmem {
    static constexpr uint32_t kXBoxBytes = NT * 128;            // 64 k x NT rows x 2 B
    static constexpr uint32_t kXStageBytes = 2 * kXBoxBytes;    // 128 k
    static constexpr uint32_t kCodesOff = 0;
    static constexpr uint32_t kXOff = kCodesOff + kStages * kCodeStageBytes;
    static constexpr uint32_t kBarOff = kXOff + kStages * kXStageBytes;
    // barriers: full, cempty, xempty [kStages]; afull, aempty [kTmemStages]; dfull
    static constexpr uint32_t kNumBars = 3 * kStages + 2 * kTmemStages + 1;
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
    static constexpr uint32_t kBytes = kMiscOff + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-B alignment
    static_assert(NT * kTileN * 4 <= kStages * kCodeStageBytes, "reduction buffer aliases code stages");
    // at most two CTAs per SM, so two 256-column TMEM allocations never wait
    static_assert(3 * (kAlloc + 1024) > 228 * 1024, "shared memory must cap residency at 2 CTAs/SM");
};

template <bool kBf16>
__device__ __forceinline__ void dequant16(const uint4 c, uint32_t (&out)[8]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if constexpr (kBf16) {
            e4m3x4_to_bf16x2(w[q], out[2 * q], out[2 * q + 1]);
        } else {
            e4m3x4_to_f16x2(w[q], out[2 * q], out[2 * q + 1]);
        }
    }
}

__device__ __forceinline__ void record_error(int code, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(&g_skinny_error, 0, code);
}

template <int NT, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x,
                  const float* __restrict__ scales, const float* __restrict__ bias, uint16_t* __restrict__ y,
                  int m_rows, int m_row0, int64_t n, int64_t k, int split) {
    using L = SkinnySmem<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto cempty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto xempty = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
    auto afull = [&](int t) { return bar0 + 8u * (3 * kStages + t); };
    auto aempty = [&](int t) { return bar0 + 8u * (3 * kStages + kTmemStages + t); };
    const uint32_t dfull = bar0 + 8u * (3 * kStages + 2 * kTmemStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = split > 1 ? cluster_ctarank() : 0u;
    const int64_t tile = blockIdx.x / split;
    const int64_t n0 = tile * kTileN;
    const int64_t nkb = (k + kBlockK - 1) / kBlockK;
    const int64_t kb_begin = nkb * rank / split;
    const int64_t kb_end = nkb * (rank + 1) / split;
    const int iters = static_cast<int>(kb_end - kb_begin);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(cempty(s), 4);
            mbar_init(xempty(s), 1);
        }
        for (int t = 0; t < kTmemStages; ++t) {
            mbar_init(afull(t), 4);
            mbar_init(aempty(t), 1);
        }
        mbar_init(dfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&map_codes);
        tma_prefetch_desc(&map_x);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_first();
            const uint64_t pol_keep = policy_evict_last();
            int issued = 0;
            for (int it = 0; it < iters; ++it) {
                const int s = it % kStages;
                const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
                if (!mbar_wait(cempty(s), ph ^ 1u, abort_flag) || !mbar_wait(xempty(s), ph ^ 1u, abort_flag)) {
                    record_error(kErrWaitSlot, abort_flag);
                    break;
                }
                const int32_t kk = static_cast<int32_t>((kb_begin + it) * kBlockK);
                const uint32_t xs = sbase + L::kXOff + s * L::kXStageBytes;
                mbar_arrive_expect_tx(full(s), kCodeStageBytes + L::kXStageBytes);
                tma_load_2d(sbase + L::kCodesOff + s * kCodeStageBytes, &map_codes, kk,
                            static_cast<int32_t>(n0), full(s), pol_stream);
                tma_load_2d(xs, &map_x, kk, m_row0, full(s), pol_keep);
                tma_load_2d(xs + L::kXBoxBytes, &map_x, kk + 64, m_row0, full(s), pol_keep);
                ++issued;
            }
            if (*abort_flag) {
                // let every copy still in flight land before the CTA exits
                for (int it = (issued > kStages ? issued - kStages : 0); it < issued; ++it) {
                    if (!mbar_wait_drain(full(it % kStages), static_cast<uint32_t>((it / kStages) & 1)))
                        atomicCAS(&g_skinny_error, 0, kErrWaitDrain);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBf16, NT);
            const uint32_t d_tmem = tmem + kTmemDCol;
            for (int it = 0; it < iters; ++it) {
                const int s = it % kStages, t = it % kTmemStages;
                const uint32_t ps = static_cast<uint32_t>((it / kStages) & 1);
                const uint32_t pt = static_cast<uint32_t>((it / kTmemStages) & 1);
                if (!mbar_wait(full(s), ps, abort_flag) || !mbar_wait(afull(t), pt, abort_flag)) {
                    record_error(kErrWaitDequant, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t xs = sbase + L::kXOff + s * L::kXStageBytes;
#pragma unroll
                for (int q = 0; q < kBlockK / 16; ++q) {
                    const uint32_t a_tmem = tmem + t * kTmemAStageCols + q * 8;
                    const uint64_t b_desc = smem_desc_sw128_kmajor(xs + (q >> 2) * L::kXBoxBytes + (q & 3) * 32);
                    mma_f16_ts(d_tmem, a_tmem, b_desc, idesc, (it | q) != 0);
                }
                tc_commit(aempty(t));
                tc_commit(xempty(s));
            }
            // dfull completes when every MMA issued above has finished
            tc_commit(dfull);
        }
    } else {
        // ------------------------------------------ dequant (warps 2-5) --
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // channel within the tile == TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        for (int it = 0; it < iters; ++it) {
            const int s = it % kStages, t = it % kTmemStages;
            const uint32_t ps = static_cast<uint32_t>((it / kStages) & 1);
            const uint32_t pt = static_cast<uint32_t>((it / kTmemStages) & 1);
            if (!mbar_wait_warp(full(s), ps, abort_flag)) {
                record_error(kErrWaitTma, abort_flag);
                break;
            }
            const uint8_t* row = smem + L::kCodesOff + s * kCodeStageBytes + r * 128;
            uint4 c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(cempty(s));
            if (!mbar_wait_warp(aempty(t), pt ^ 1u, abort_flag)) {
                record_error(kErrWaitMma, abort_flag);
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t v[8];
                dequant16<kBf16>(c[j], v);
                tmem_st_x8(lane_addr + t * kTmemAStageCols + j * 8, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(t));
        }

        // --------------------------------------------------- epilogue --
        float acc[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j] = 0.0f;
        if (iters > 0 && mbar_wait_warp(dfull, 0, abort_flag)) {
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < NT / 16; ++h) {
                uint32_t v[16];
                tmem_ld_x16(lane_addr + kTmemDCol + h * 16, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[h * 16 + j] = __uint_as_float(v[j]);
            }
        } else if (iters > 0) {
            record_error(kErrWaitMma, abort_flag);
        }
        if (split == 1) {
            const int64_t col = n0 + r;
            if (col < n && !*abort_flag) {
                const float sc = scales[col];
                const float b = bias ? bias[col] : 0.0f;
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    if (j < m_rows) y[static_cast<int64_t>(j) * n + col] = round_out<kBf16>(fmaf(acc[j], sc, b));
            }
        } else {
            float* red = reinterpret_cast<float*>(smem + L::kCodesOff);
#pragma unroll
            for (int j = 0; j < NT; ++j) red[j * kTileN + r] = acc[j];
        }
    }

    __syncthreads();
    if (split > 1) {
        cluster_sync_all();
        if (warp >= 2 && !*abort_flag) {
            const int e = threadIdx.x - 64;
            const int rows_per = kTileN / split;
            const uint32_t red_base = sbase + L::kCodesOff;
            const int items = rows_per * m_rows;
            for (int i = e; i < items; i += 128) {
                const int j = i / rows_per;
                const int rr = static_cast<int>(rank) * rows_per + i % rows_per;
                const uint32_t off = static_cast<uint32_t>((j * kTileN + rr) * 4);
                float sum = 0.0f;
                for (int p = 0; p < split; ++p) sum += ld_shared_cluster_f32(mapa_shared(red_base + off, p));
                const int64_t col = n0 + rr;
                if (col < n) {
                    const float b = bias ? bias[col] : 0.0f;
                    y[static_cast<int64_t>(j) * n + col] = round_out<kBf16>(fmaf(sum, scales[col], b));
                }
            }
        }
        cluster_sync_all();
    }
    if (warp == 1) {
        // every MMA must have finished before its TMEM is released
        if (iters > 0 && !mbar_wait_drain(dfull, 0)) atomicCAS(&g_skinny_error, 0, kErrWaitDrain);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host --

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

static bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
};

static cudaError_t device_info(DeviceInfo& info) {
    static DeviceInfo cache[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev].sms == 0) {
        e = cudaDeviceGetAttribute(&cache[dev].sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    info = cache[dev];
    return cudaSuccess;
}

// Cluster size along k for a grid of `tiles` channel tiles: the one (1, 2, 4,
// 8) that spreads CTAs most evenly over the SMs, keeping >= 2 k-blocks each.
static int choose_split(int64_t tiles, int64_t nkb, int sms) {
    int best = 1;
    double best_util = -1.0;
    for (int s = 1; s <= 8; s *= 2) {
        if (s > 1 && nkb / s < 2) break;
        const int64_t ctas = tiles * s;
        const int64_t per_sm = (ctas + sms - 1) / sms;
        if (per_sm > 2 && s > 1) break;
        const double util = static_cast<double>(ctas) / static_cast<double>(per_sm * sms);
        if (util > best_util + 1e-9) {
            best_util = util;
            best = s;
        }
    }
    return best;
}

template <int NT, bool kBf16>
static cudaError_t launch_nt(const LinearArgs& a, int split, cudaStream_t st) {
    using L = SkinnySmem<NT>;
    auto kern = skinny_kernel<NT, kBf16>;
    static std::once_flag attr_once[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    });
    if (attr_err != cudaSuccess) return attr_err;

    DeviceInfo info;
    e = device_info(info);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (a.n + kTileN - 1) / kTileN;
    const int64_t nkb = (a.k + kBlockK - 1) / kBlockK;
    if (split <= 0) split = choose_split(tiles, nkb, info.sms);

    CUtensorMap map_codes, map_x;
    if (!encode_2d(&map_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, static_cast<uint64_t>(a.k),
                   static_cast<uint64_t>(a.n), static_cast<uint64_t>(a.k), kBlockK, kTileN))
        return cudaErrorInvalidValue;
    if (!encode_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.x, static_cast<uint64_t>(a.k),
                   static_cast<uint64_t>(a.m), static_cast<uint64_t>(a.k) * 2, 64, NT))
        return cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * split), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    uint16_t* yp = static_cast<uint16_t*>(a.y);
    for (int64_t m0 = 0; m0 < a.m; m0 += 32) {
        const int rows = static_cast<int>(a.m - m0 < 32 ? a.m - m0 : 32);
        e = cudaLaunchKernelEx(&cfg, kern, map_codes, map_x, a.scales, a.bias, yp + m0 * a.n, rows,
                               static_cast<int>(m0), a.n, a.k, split);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int skinny_max_split() { return 8; }

cudaError_t launch_skinny(const LinearArgs& a, int split, cudaStream_t st) {
    const bool bf16 = a.act == 1;
    if (a.m <= 16) return bf16 ? launch_nt<16, true>(a, split, st) : launch_nt<16, false>(a, split, st);
    return bf16 ? launch_nt<32, true>(a, split, st) : launch_nt<32, false>(a, split, st);
}

int read_skinny_device_error() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_skinny_error, sizeof v) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_skinny_error, &zero, sizeof zero);
    return v;
}

}  // namespace fp8w
