// skinny.cu -- kernel K3: the M <= 32 linear layer on the tcgen05 tensor cores,
// "swap-AB": the weight channels are the 128-row A operand, the tokens the
// narrow B operand.
//
// Page "kadirnar/kernel-agent fp8-weights", section "Dequantise in
// registers" (skinny GEMM: the weight as the A operand, a 16-bit MMA in the
// activations' type, every code converted once and reused for every token,
// split-K so that all the GPU streams the weight).  That design targets
// mma.sync on sm_80..sm_120; this one is built for sm_103a:
//
//  * Persistent stream-K grid, one CTA per SM.  The work is the list of
//    units (channel tile of 128, k-block of 128); CTA c takes the contiguous
//    units [c*U/P, (c+1)*U/P), so every SM streams the same number of code
//    bytes (+-1 unit).  A tile that straddles CTAs is finished by the last
//    contributor to arrive: partial fp32 tiles go to a caller-provided
//    workspace and are summed in CTA order (deterministic); nothing waits on
//    another CTA.
//  * Warp 0 streams each unit's 128 x 128 code tile and its M x 128
//    activation tile into an 8-stage shared-memory ring with TMA (128-byte
//    swizzle; rows past N or M and k past K read as zeros).
//  * Four dequantising warpgroups take the units round-robin: thread r
//    reads the 128 codes of channel r (conflict-free through the swizzle),
//    converts them exactly to bf16 / fp16 in registers and stores them with
//    tcgen05.st into a 6-slot TMEM ring, where they are the A operand of the
//    MMA (A from tensor memory: the dequantised weight never touches shared
//    memory).
//  * Warp 1 issues tcgen05.mma.kind::f16 (M = 128, N = 16 or 32 tokens,
//    K = 16) into one of two TMEM accumulators, and returns stages with
//    tcgen05.commit.
//  * One epilogue warpgroup reads a finished accumulator with tcgen05.ld
//    (thread r holds channel r for every token) while the next tile
//    accumulates in the other buffer, and stores y = round(fma(acc, scale,
//    bias)) or, for a split tile, its partial.
//
// Every wait is bounded in time: on a timeout the CTA records an error code,
// raises an abort flag that ends every role's loop, lets its in-flight
// copies and MMAs finish, frees TMEM and exits.
#include <mutex>

#include "fp8w_device.cuh"
#include "fp8w_internal.h"

namespace fp8w {

static __device__ int g_skinny_error;

constexpr int kTileN = 128;                 // output channels per tile (MMA M)
constexpr int kBlockK = 128;                // k per unit / stage
constexpr int kStages = 8;                  // shared-memory ring
constexpr int kASlots = 6;                  // TMEM A-operand ring
constexpr int kDequantGroups = 4;           // dequantising warpgroups
constexpr int kFirstDequantWarp = 6;        // warps 0 TMA, 1 MMA, 2-5 epilogue
constexpr int kThreads = 32 * (kFirstDequantWarp + 4 * kDequantGroups);  // 704
constexpr int kTmemCols = 512;              // one CTA per SM
constexpr int kAColsPerSlot = kBlockK / 2;  // two 16-bit values per column
constexpr int kDCol0 = kASlots * kAColsPerSlot;  // 384: accumulators at 384, 416
constexpr uint32_t kCodeStageBytes = kTileN * kBlockK;  // 16 KB
constexpr int kMaxNT = 32;

template <int NT>
struct SkinnySmem {
    static constexpr uint32_t kXBoxBytes = NT * 128;          // 64 k x NT rows x 2 B
    static constexpr uint32_t kXStageBytes = 2 * kXBoxBytes;  // 128 k
    static constexpr uint32_t kCodesOff = 0;
    static constexpr uint32_t kXOff = kCodesOff + kStages * kCodeStageBytes;
    static constexpr uint32_t kBarOff = kXOff + kStages * kXStageBytes;
    // full, cempty, xempty [kStages]; afull, aempty [kASlots]; dready, dfree [2]; drain
    static constexpr uint32_t kNumBars = 3 * kStages + 2 * kASlots + 5;
    // tmem base, abort flag, last-contributor flag, epilogue abort flag
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
    static constexpr uint32_t kBytes = kMiscOff + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
    static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// Workspace: [kMaxCtas arrival counters (uint32)][2 partial-tile slots per
// CTA, each 128 channels x kMaxNT fp32, channel-major].  The counters must
// be zero before the first call; every call leaves them zero.  Their region
// has a fixed size, so calls with different grids never overlap it.
constexpr int kMaxCtas = 1024;
constexpr size_t kWsCountersBytes = kMaxCtas * 4;
__host__ __device__ constexpr size_t ws_slot_floats() { return static_cast<size_t>(kMaxNT) * kTileN; }
size_t skinny_workspace_bytes(int p) { return kWsCountersBytes + 2 * static_cast<size_t>(p) * ws_slot_floats() * 4; }
// A CTA takes at least this many units, so a small matrix is not split into
// more partial tiles than it has k-blocks to share.
constexpr int64_t kMinUnitsPerCta = 4;

struct Partition {
    int64_t units, p, nkb;
    __device__ __forceinline__ int64_t begin(int64_t c) const { return c * units / p; }
    // CTA whose range holds unit u
    __device__ __forceinline__ int64_t owner(int64_t u) const {
        int64_t c = u * p / units;
        while (c + 1 < p && begin(c + 1) <= u) ++c;
        while (c > 0 && begin(c) > u) --c;
        return c;
    }
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

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int NT, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x,
                  const float* __restrict__ scales, const float* __restrict__ bias, uint16_t* __restrict__ y,
                  uint8_t* __restrict__ workspace, int m_rows, int m_row0, int64_t n, int64_t k) {
    using L = SkinnySmem<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto cempty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto xempty = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
    auto afull = [&](int t) { return bar0 + 8u * (3 * kStages + t); };
    auto aempty = [&](int t) { return bar0 + 8u * (3 * kStages + kASlots + t); };
    auto dready = [&](int d) { return bar0 + 8u * (3 * kStages + 2 * kASlots + d); };
    auto dfree = [&](int d) { return bar0 + 8u * (3 * kStages + 2 * kASlots + 2 + d); };
    const uint32_t drain = bar0 + 8u * (3 * kStages + 2 * kASlots + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);
    volatile int* ep_abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 12);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles = (n + kTileN - 1) / kTileN;
    const int64_t nkb = (k + kBlockK - 1) / kBlockK;
    const Partition part{tiles * nkb, static_cast<int64_t>(gridDim.x), nkb};
    const int64_t c = blockIdx.x;
    const int64_t u0 = part.begin(c), u1 = part.begin(c + 1);
    const int iters = static_cast<int>(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(cempty(s), 4);
            mbar_init(xempty(s), 1);
        }
        for (int t = 0; t < kASlots; ++t) {
            mbar_init(afull(t), 4);
            mbar_init(aempty(t), 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(dready(d), 1);
            mbar_init(dfree(d), 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *ep_abort = 0;
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
        // ---------------------------------------------------- TMA producer --
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
                const int64_t u = u0 + it;
                const int32_t kk = static_cast<int32_t>((u % nkb) * kBlockK);
                const int32_t row = static_cast<int32_t>((u / nkb) * kTileN);
                const uint32_t xs = sbase + L::kXOff + s * L::kXStageBytes;
                mbar_arrive_expect_tx(full(s), kCodeStageBytes + L::kXStageBytes);
                tma_load_2d(sbase + L::kCodesOff + s * kCodeStageBytes, &map_codes, kk, row, full(s), pol_stream);
                tma_load_2d(xs, &map_x, kk, m_row0, full(s), pol_keep);
                tma_load_2d(xs + L::kXBoxBytes, &map_x, kk + 64, m_row0, full(s), pol_keep);
                ++issued;
            }
            if (*abort_flag) {
                for (int it = (issued > kStages ? issued - kStages : 0); it < issued; ++it)
                    if (!mbar_wait_drain(full(it % kStages), static_cast<uint32_t>((it / kStages) & 1)))
                        atomicCAS(&g_skinny_error, 0, kErrWaitDrain);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer --
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBf16, NT);
            int seg = -1;
            for (int it = 0; it < iters; ++it) {
                const int64_t u = u0 + it;
                const bool first = (it == 0) || (u % nkb == 0);
                const bool last = (it == iters - 1) || (u % nkb == nkb - 1);
                if (first) {
                    ++seg;
                    // the epilogue must have drained this accumulator (two segments ago)
                    if (!mbar_wait(dfree(seg & 1), static_cast<uint32_t>(((seg >> 1) & 1) ^ 1), abort_flag)) {
                        record_error(kErrWaitMma, abort_flag);
                        break;
                    }
                }
                const int s = it % kStages, t = it % kASlots;
                if (!mbar_wait(full(s), static_cast<uint32_t>((it / kStages) & 1), abort_flag) ||
                    !mbar_wait(afull(t), static_cast<uint32_t>((it / kASlots) & 1), abort_flag)) {
                    record_error(kErrWaitDequant, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t xs = sbase + L::kXOff + s * L::kXStageBytes;
                const uint32_t d_tmem = tmem + kDCol0 + (seg & 1) * 32;
#pragma unroll
                for (int q = 0; q < kBlockK / 16; ++q) {
                    const uint32_t a_tmem = tmem + t * kAColsPerSlot + q * 8;
                    const uint64_t b_desc = smem_desc_sw128_kmajor(xs + (q >> 2) * L::kXBoxBytes + (q & 3) * 32);
                    mma_f16_ts(d_tmem, a_tmem, b_desc, idesc, !(first && q == 0));
                }
                tc_commit(aempty(t));
                tc_commit(xempty(s));
                if (last) tc_commit(dready(seg & 1));
            }
            // every MMA issued above completes before TMEM is released
            tc_commit(drain);
            if (!mbar_wait_drain(drain, 0)) atomicCAS(&g_skinny_error, 0, kErrWaitDrain);
        }
    } else if (warp < kFirstDequantWarp) {
        // ------------------------------------------- epilogue (warps 2-5) --
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // channel within the tile == TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const int etid = threadIdx.x - 64;  // 0..127
        uint32_t* counters = reinterpret_cast<uint32_t*>(workspace);
        float* slots = reinterpret_cast<float*>(workspace + kWsCountersBytes);
        int seg = 0;
        for (int64_t u = u0; u < u1; ++seg) {
            const int64_t tile = u / nkb;
            const int64_t seg_end = (tile + 1) * nkb < u1 ? (tile + 1) * nkb : u1;
            const bool whole = (u == tile * nkb) && (seg_end == (tile + 1) * nkb);
            const int d = seg & 1;
            float acc[NT];
            if (!mbar_wait_warp(dready(d), static_cast<uint32_t>((seg >> 1) & 1), abort_flag)) {
                if (lane == 0) *ep_abort = 1;
                record_error(kErrWaitMma, abort_flag);
            }
            // the four epilogue warps leave together (ep_abort is written only
            // by them, before this barrier), so their named barriers stay matched
            epilogue_bar();
            if (*ep_abort) break;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < NT / 16; ++h) {
                uint32_t v[16];
                tmem_ld_x16(lane_addr + kDCol0 + d * 32 + h * 16, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[h * 16 + j] = __uint_as_float(v[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dfree(d));

            const int64_t col = tile * kTileN + r;
            if (whole) {
                if (col < n) {
                    const float sc = scales[col];
                    const float b = bias ? bias[col] : 0.0f;
#pragma unroll
                    for (int j = 0; j < NT; ++j)
                        if (j < m_rows) y[static_cast<int64_t>(j) * n + col] = round_out<kBf16>(fmaf(acc[j], sc, b));
                }
            } else {
                // partial tile: publish, count, and let the last contributor finish
                const int64_t slot = 2 * c + (seg == 0 ? 0 : 1);
                float4* mine = reinterpret_cast<float4*>(slots + slot * ws_slot_floats() + r * kMaxNT);
#pragma unroll
                for (int j = 0; j < NT / 4; ++j)
                    mine[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
                __threadfence();
                epilogue_bar();
                const int64_t c_lo = part.owner(tile * nkb);
                const int64_t c_hi = part.owner((tile + 1) * nkb - 1);
                if (etid == 0) {
                    const uint32_t old = atomicAdd(&counters[c_lo], 1u);
                    const bool is_last = old == static_cast<uint32_t>(c_hi - c_lo);
                    if (is_last) atomicExch(&counters[c_lo], 0u);
                    *last_flag = is_last ? 1 : 0;
                }
                epilogue_bar();
                if (*last_flag) {
                    __threadfence();
                    float sum[NT];
#pragma unroll
                    for (int j = 0; j < NT; ++j) sum[j] = 0.0f;
                    // contributors in CTA order: the result does not depend on who is last
                    for (int64_t cc = c_lo; cc <= c_hi; ++cc) {
                        const int64_t cs = 2 * cc + ((part.begin(cc) / nkb) == tile ? 0 : 1);
                        const float4* src = reinterpret_cast<const float4*>(slots + cs * ws_slot_floats() + r * kMaxNT);
                        float4 v[NT / 4];
#pragma unroll
                        for (int j = 0; j < NT / 4; ++j) v[j] = __ldcg(src + j);
#pragma unroll
                        for (int j = 0; j < NT / 4; ++j) {
                            sum[4 * j] += v[j].x;
                            sum[4 * j + 1] += v[j].y;
                            sum[4 * j + 2] += v[j].z;
                            sum[4 * j + 3] += v[j].w;
                        }
                    }
                    if (col < n) {
                        const float sc = scales[col];
                        const float b = bias ? bias[col] : 0.0f;
#pragma unroll
                        for (int j = 0; j < NT; ++j)
                            if (j < m_rows) y[static_cast<int64_t>(j) * n + col] = round_out<kBf16>(fmaf(sum[j], sc, b));
                    }
                }
                epilogue_bar();
            }
            u = seg_end;
        }
    } else {
        // -------------------------------- dequantising warpgroups (6-21) --
        const int group = (warp - kFirstDequantWarp) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        for (int it = group; it < iters; it += kDequantGroups) {
            const int s = it % kStages, t = it % kASlots;
            if (!mbar_wait_warp(full(s), static_cast<uint32_t>((it / kStages) & 1), abort_flag)) {
                record_error(kErrWaitTma, abort_flag);
                break;
            }
            const uint8_t* row = smem + L::kCodesOff + s * kCodeStageBytes + r * 128;
            uint4 cw[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) cw[j] = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(cempty(s));
            if (!mbar_wait_warp(aempty(t), static_cast<uint32_t>(((it / kASlots) & 1) ^ 1), abort_flag)) {
                record_error(kErrWaitMma, abort_flag);
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t v[8];
                dequant16<kBf16>(cw[j], v);
                tmem_st_x8(lane_addr + t * kAColsPerSlot + j * 8, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(t));
        }
    }

    __syncthreads();
    if (warp == 1) {
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

cudaError_t device_sm_count(int& sms) {
    static int cache[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == 0) {
        e = cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    sms = cache[dev];
    return cudaSuccess;
}

// CTAs of the persistent grid: one per SM, each with >= kMinUnitsPerCta
// units when there are enough, never more than kMaxCtas.
int64_t skinny_grid(int64_t n, int64_t k, int sms) {
    const int64_t units = ((n + kTileN - 1) / kTileN) * ((k + kBlockK - 1) / kBlockK);
    int64_t p = units / kMinUnitsPerCta;
    if (p < 1) p = 1;
    if (p > sms) p = sms;
    if (p > kMaxCtas) p = kMaxCtas;
    return p;
}

template <int NT, bool kBf16>
static cudaError_t launch_nt(const LinearArgs& a, void* workspace, cudaStream_t st) {
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
    int sms = 0;
    e = device_sm_count(sms);
    if (e != cudaSuccess) return e;

    CUtensorMap map_codes, map_x;
    if (!encode_2d(&map_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, static_cast<uint64_t>(a.k),
                   static_cast<uint64_t>(a.n), static_cast<uint64_t>(a.k), kBlockK, kTileN))
        return cudaErrorInvalidValue;
    if (!encode_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.x, static_cast<uint64_t>(a.k),
                   static_cast<uint64_t>(a.m), static_cast<uint64_t>(a.k) * 2, 64, NT))
        return cudaErrorInvalidValue;

    const int64_t grid = skinny_grid(a.n, a.k, sms);
    uint16_t* yp = static_cast<uint16_t*>(a.y);
    for (int64_t m0 = 0; m0 < a.m; m0 += kMaxNT) {
        const int rows = static_cast<int>(a.m - m0 < kMaxNT ? a.m - m0 : kMaxNT);
        kern<<<static_cast<unsigned>(grid), kThreads, L::kAlloc, st>>>(
            map_codes, map_x, a.scales, a.bias, yp + m0 * a.n, static_cast<uint8_t*>(workspace), rows,
            static_cast<int>(m0), a.n, a.k);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t skinny_workspace_size(int sms) { return skinny_workspace_bytes(sms); }

cudaError_t launch_skinny(const LinearArgs& a, void* workspace, cudaStream_t st) {
    const bool bf16 = a.act == 1;
    if (a.m <= 16) return bf16 ? launch_nt<16, true>(a, workspace, st) : launch_nt<16, false>(a, workspace, st);
    return bf16 ? launch_nt<32, true>(a, workspace, st) : launch_nt<32, false>(a, workspace, st);
}

int read_skinny_device_error() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_skinny_error, sizeof v) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_skinny_error, &zero, sizeof zero);
    return v;
}

}  // namespace fp8w
