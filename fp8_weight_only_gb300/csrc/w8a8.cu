// w8a8.cu -- kernel K5: the W8A8 linear layer on the tcgen05 tensor cores.
//
// Page "tensormux Write an FP8 kernel", "Required reasoning process": the
// activations are quantised per token and the weights per output channel,
// both to e4m3 with scale = amax / 448 and a saturating conversion; the GEMM
// multiplies the codes with fp32 accumulation and the epilogue multiplies
// the accumulator by both scales (steps 2, 4 and 5).  Page "kadirnar/
// kernel-agent fp8-weights", section "Tensor cores and libraries on sm_120",
// names the e4m3 x e4m3 tensor-core MMA as this separate target.
//
//   y[m, n] = round_out( fma( acc[m, n] * sx[m], sw[n], bias[n] ) ),
//   acc[m, n] = sum_k e4m3(qx[m, k]) * e4m3(qw[n, k])       (fp32)
//
// Both operands are e4m3 codes, so nothing is converted on the way: TMA
// brings a 128-channel x 128-code weight tile and the matching BN-token x
// 128-code activation tile into one shared-memory stage (128-byte swizzle,
// rows past N, M or K read as zeros), and one warp issues four
// tcgen05.mma.kind::f8f6f4 per stage (M = 128 channels, N = BN tokens,
// K = 32 codes; both operands by shared-memory descriptor; the products of
// two e4m3 values are exact in fp32) into an fp32 accumulator in TMEM.
//   warp 0     TMA producer of the stages (weight tiles evict-first, they
//              are read once; activation tiles evict-last, every channel
//              tile re-reads them)
//   warp 1     MMA issue; owns TMEM
//   warps 2-5  epilogue: thread r holds channel r of the tile for every
//              token, TMEM -> fma(acc * sx, sw, bias) -> one rounding -> y
// Launch shapes:
//   - persistent CTAs, one per SM, walk the output tiles (128 channels x BN
//     tokens, the token tiles of one weight block adjacent); D is
//     double-buffered in TMEM so the epilogue drains a tile while the next
//     accumulates;
//   - when the tiles fill well under the GPU (few channels and few tokens,
//     the decode shapes), each tile's k-blocks are split evenly over a
//     thread-block cluster of 2..8 CTAs; at the end each rank adds up, in
//     rank order, a slice of the tile's channels from every rank's fp32
//     partial through distributed shared memory.
// `early` (the weights were complete before the preceding kernel started):
// the producer issues the first stages' weight tiles before waiting for the
// previous grid, so the weight stream starts while that grid drains; the
// activation tiles, the scales and y wait for it as usual.
// Every wait is bounded; a CTA that gives up records a code, raises its
// abort flag, lets its copies and MMAs land and frees TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fp8w_device.cuh"
#include "fp8w_internal.h"

namespace fp8w {

static __device__ int g_w8a8_error;

namespace {

constexpr int kWM = 128;                  // channels a tile (MMA M, TMEM lanes)
constexpr int kWK = 128;                  // codes of k a stage (one 128-byte swizzle row)
constexpr uint32_t kWABytes = kWM * kWK;  // 16 KB
constexpr int kWThreads = 192;
constexpr int kWMmaWarp = 1, kWFirstEpiWarp = 2;
constexpr int kWBarTmem = 1;              // named barrier: MMA warp + epilogue warps
constexpr int kWMaxSplit = 8;             // portable cluster size
constexpr int kWMinKbPerCta = 4;          // a split CTA takes at least this many k-blocks

// A stage holds kG k-blocks (fetched by one 3-D copy per operand when k %
// 128 == 0, else one k-block by 2-D copies): the weight tiles first, then
// the activation tiles.  Large copies matter: a 2-D copy of 128 rows x 128
// bytes streams ~54 GB/s per SM, a 3-D one of four k-blocks ~128 GB/s.
template <int BN>
struct W8Smem {
    static constexpr int kG = BN <= 16 ? 4 : BN <= 64 ? 3 : BN == 128 ? 2 : 1;
    static constexpr uint32_t kBBytes = BN * kWK;
    static constexpr uint32_t kXOff = kG * kWABytes;                 // activation tiles within a stage
    static constexpr uint32_t kStageBytes = kG * (kWABytes + kBBytes);  // a multiple of 1024
    static constexpr int kStages = BN == 256 ? 4 : 3;
    static constexpr uint32_t kBarOff = kStages * kStageBytes;
    // full, empty [kStages] | dfull, dempty [2] | drain
    static constexpr uint32_t kNumBars = 2 * kStages + 4 + 1;
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;  // TMEM base, abort flag
    static constexpr uint32_t kBytes = kMiscOff + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
    static_assert(kAlloc <= 227 * 1024, "shared memory");
    static constexpr uint32_t kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
    static_assert(kTmemCols <= 512, "TMEM columns");
    // a split rank's partial tile (token-major fp32) reuses the stage ring
    static_assert(static_cast<uint32_t>(BN) * kWM * 4 <= kBarOff, "partial tile fits in the ring");
};

// Instruction descriptor for kind::f8f6f4: fp32 accumulator, A and B e4m3
// (format 0), both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t n) {
    return (1u << 4)              // D format: f32
           | (0u << 7)            // A format: e4m3
           | (0u << 10)           // B format: e4m3
           | ((n >> 3) << 17)     // N / 8
           | ((128u >> 4) << 24); // M / 16
}

// D[tmem] (+)= A[smem] * B[smem] over K = 32 e4m3 codes, issued by one
// elected lane of a converged warp.
__device__ __forceinline__ void mma_e4m3_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

__device__ __forceinline__ void w8a8_error(int code, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(&g_w8a8_error, 0, 5000 + code);
}

}  // namespace

template <int BN, bool kBf16>
__global__ void __launch_bounds__(kWThreads, 1)
    w8a8_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                const float* __restrict__ sx, const float* __restrict__ sw, const float* __restrict__ bias,
                uint16_t* __restrict__ y, int64_t m, int64_t n, int64_t k, int split, int early, int g3) {
    using L = W8Smem<BN>;
    constexpr int kS = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kS + s); };
    auto dfull = [&](int d) { return bar0 + 8u * (2 * kS + d); };
    auto dempty = [&](int d) { return bar0 + 8u * (2 * kS + 2 + d); };
    const uint32_t drain = bar0 + 8u * (2 * kS + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ttiles = (m + BN - 1) / BN;
    const int64_t tiles = ((n + kWM - 1) / kWM) * ttiles;
    const int nkb = static_cast<int>((k + kWK - 1) / kWK);
    // split: cluster c / split takes tile c / split, its rank an even share
    // of the k-blocks; otherwise tiles blockIdx.x, + gridDim.x, ... whole
    const int rank = split > 1 ? static_cast<int>(blockIdx.x % split) : 0;
    const int64_t t_first = split > 1 ? blockIdx.x / split : blockIdx.x;
    const int64_t t_step = split > 1 ? tiles : gridDim.x;
    const int kb0 = split > 1 ? rank * nkb / split : 0;
    const int kb1 = split > 1 ? (rank + 1) * nkb / split : nkb;
    // k-blocks a stage, and the bytes its copies deliver (a 3-D box always
    // delivers kG tiles, zeros past k)
    const int gk = g3 ? L::kG : 1;
    const uint32_t stage_tx = static_cast<uint32_t>(gk) * (kWABytes + L::kBBytes);

    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < kS; ++s) {
                mbar_init(full(s), 1);
                mbar_init(empty(s), 1);  // MMA commit
            }
            for (int d = 0; d < 2; ++d) {
                mbar_init(dfull(d), 1);
                mbar_init(dempty(d), 4);  // the four epilogue warps
            }
            mbar_init(drain, 1);
            *abort_flag = 0;
            tma_prefetch_desc(&map_w);
            tma_prefetch_desc(&map_x);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    uint32_t tmem = 0;
    if (warp >= kWMmaWarp) {
        if (warp == kWMmaWarp) {
            tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        asm volatile("bar.sync %0, %1;" ::"n"(kWBarTmem), "n"(kWThreads - 32) : "memory");
        tc_fence_after();
        tmem = *tmem_slot;
    }

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            // weight tiles of the first stages, before the dependency wait
            auto load_w = [&](uint32_t st, int kb, int64_t cb, uint32_t bar) {
                if (g3) tma_load_3d(st, &map_w, 0, static_cast<int32_t>(cb * kWM), kb, bar, pol_w);
                else tma_load_2d(st, &map_w, kb * kWK, static_cast<int32_t>(cb * kWM), bar, pol_w);
            };
            auto load_x = [&](uint32_t st, int kb, int64_t tb, uint32_t bar) {
                if (g3) tma_load_3d(st + L::kXOff, &map_x, 0, static_cast<int32_t>(tb * BN), kb, bar, pol_x);
                else tma_load_2d(st + L::kXOff, &map_x, kb * kWK, static_cast<int32_t>(tb * BN), bar, pol_x);
            };
            int pre = 0;
            if (early) {
                for (int64_t t = t_first; t < tiles && pre < kS; t += t_step) {
                    const int64_t cb = t / ttiles;
                    for (int kb = kb0; kb < kb1 && pre < kS; kb += gk, ++pre) {
                        mbar_arrive_expect_tx(full(pre), stage_tx);
                        load_w(sbase + pre * L::kStageBytes, kb, cb, full(pre));
                    }
                    if (split > 1) break;
                }
            }
            pdl_wait();  // the activation codes may come from the previous kernel
            int64_t i = 0;
            bool ok = true;
            for (int64_t t = t_first; t < tiles && ok; t += t_step) {
                const int64_t cb = t / ttiles, tb = t - cb * ttiles;
                for (int kb = kb0; kb < kb1; kb += gk, ++i) {
                    const int s = static_cast<int>(i % kS);
                    const uint32_t st = sbase + s * L::kStageBytes;
                    if (i >= pre) {
                        if (!mbar_wait(empty(s), static_cast<uint32_t>((i / kS) & 1) ^ 1u, abort_flag)) {
                            w8a8_error(kErrWaitSlot, abort_flag);
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full(s), stage_tx);
                        load_w(st, kb, cb, full(s));
                    }
                    load_x(st, kb, tb, full(s));
                }
                if (split > 1) break;
            }
            if (*abort_flag) {
                // the copies still in flight land before the CTA exits (a
                // failed wait happens only at i >= pre, so every stage issued
                // early has its activation tile too)
                const int64_t issued = i;
                for (int64_t j = (issued > kS ? issued - kS : 0); j < issued; ++j)
                    if (!mbar_wait_drain(full(static_cast<int>(j % kS)), static_cast<uint32_t>((j / kS) & 1)))
                        atomicCAS(&g_w8a8_error, 0, 5000 + kErrWaitDrain);
            }
        }
    } else if (warp == kWMmaWarp) {
        // ----------------------------------------------------- MMA issue --
        constexpr uint32_t idesc = idesc_e4m3(BN);
        int64_t i = 0;
        int tile_n = 0;
        bool ok = true;
        for (int64_t t = t_first; t < tiles && ok; t += t_step, ++tile_n) {
            const int d = tile_n & 1;
            if (!mbar_wait_warp(dempty(d), static_cast<uint32_t>((tile_n >> 1) & 1) ^ 1u, abort_flag)) {
                if (lane == 0) w8a8_error(kErrWaitMma, abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(d * BN);
            for (int kb = kb0; kb < kb1; kb += gk, ++i) {
                const int s = static_cast<int>(i % kS);
                if (!mbar_wait_warp(full(s), static_cast<uint32_t>((i / kS) & 1), abort_flag)) {
                    if (lane == 0) w8a8_error(kErrWaitTma, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = sbase + s * L::kStageBytes;
                const uint32_t b_addr = a_addr + L::kXOff;
                // the stage's k-blocks that are this CTA's (a 3-D box past kb1
                // brings the next rank's, or zeros past k)
                const int nb = kb1 - kb < gk ? kb1 - kb : gk;
                for (int g = 0; g < nb; ++g) {
#pragma unroll
                    for (int kk = 0; kk < kWK / 32; ++kk)
                        mma_e4m3_ss_warp(d_tmem, smem_desc_sw128_kmajor(a_addr + g * kWABytes + kk * 32),
                                         smem_desc_sw128_kmajor(b_addr + g * L::kBBytes + kk * 32), idesc,
                                         kb > kb0 || g > 0 || kk > 0);
                }
                tc_commit_warp(empty(s));  // the stage is free once these MMAs have read it
                __syncwarp();
            }
            if (!ok) break;
            tc_commit_warp(dfull(d));
            __syncwarp();
            if (split > 1) break;
        }
        // every MMA issued above completes before TMEM is released
        tc_commit_warp(drain);
        if (!mbar_wait_drain(drain, 0) && lane == 0) atomicCAS(&g_w8a8_error, 0, 5000 + kErrWaitDrain);
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue --
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // channel within the tile == TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        pdl_wait();  // the activation scales may come from the previous kernel; y may still be read
        int tile_n = 0;
        for (int64_t t = t_first; t < tiles; t += t_step, ++tile_n) {
            const int64_t cb = t / ttiles, tb = t - cb * ttiles;
            const int d = tile_n & 1;
            if (!mbar_wait_warp(dfull(d), static_cast<uint32_t>((tile_n >> 1) & 1), abort_flag)) {
                if (lane == 0) w8a8_error(kErrWaitMma, abort_flag);
                break;
            }
            tc_fence_after();
            const int64_t col = cb * kWM + r;
            const float scw = col < n ? sw[col] : 0.0f;
            const float b = (bias && col < n) ? bias[col] : 0.0f;
            const int64_t tok0 = tb * BN;
            const int ntok = static_cast<int>(m - tok0 < BN ? m - tok0 : BN);
            float* pt = reinterpret_cast<float*>(smem);  // split: this rank's partial, token-major
            for (int c0 = 0; c0 < ntok; c0 += 16) {
                uint32_t v[16];
                tmem_ld_x16_sync(lane_addr + static_cast<uint32_t>(d * BN + c0), v);
                if (split > 1) {
                    // every MMA of this CTA is done, so the stage ring is free
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (c0 + q < ntok) pt[(c0 + q) * kWM + r] = __uint_as_float(v[q]);
                } else if (col < n) {
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (c0 + q < ntok) {
                            const int64_t tok = tok0 + c0 + q;
                            y[tok * n + col] = round_out<kBf16>(fmaf(__uint_as_float(v[q]) * __ldg(sx + tok), scw, b));
                        }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(d));
            if (split > 1) break;
        }
    }

    __syncthreads();
    if (split > 1) {
        // this rank adds up channels [ch0, ch0 + nch) of the tile over all
        // ranks, in rank order, and writes y
        const bool red = warp >= kWFirstEpiWarp;
        const int etid = threadIdx.x - 32 * kWFirstEpiWarp;  // 0..127
        const int nch = kWM / split;
        const int ch = rank * nch + (red ? etid % nch : 0);
        const int64_t t = t_first;
        const int64_t cb = t / ttiles, tb = t - cb * ttiles;
        const int64_t col = cb * kWM + ch;
        const int64_t tok0 = tb * BN;
        const int ntok = static_cast<int>(m - tok0 < BN ? m - tok0 : BN);
        float scw = 0.0f, b = 0.0f;
        if (red && col < n) {
            scw = sw[col];
            b = bias ? bias[col] : 0.0f;
        }
        cluster_sync_all();  // every rank's partial is in its shared memory
        if (red && !*abort_flag && col < n) {
            const uint32_t pt = sbase;
            const int tstep = kWM / nch;
            for (int tk = etid / nch; tk < ntok; tk += tstep) {
                const uint32_t off = pt + static_cast<uint32_t>((tk * kWM + ch) * 4);
                float v[kWMaxSplit];
#pragma unroll
                for (int rr = 0; rr < kWMaxSplit; ++rr)
                    if (rr < split) v[rr] = ld_shared_cluster_f32(mapa_shared(off, rr));
                float acc = 0.0f;
#pragma unroll
                for (int rr = 0; rr < kWMaxSplit; ++rr)
                    if (rr < split) acc += v[rr];
                const int64_t tok = tok0 + tk;
                y[tok * n + col] = round_out<kBf16>(fmaf(acc * __ldg(sx + tok), scw, b));
            }
        }
        cluster_sync_all();  // no rank leaves while its partial may still be read
    }
    if (warp == kWMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// ------------------------------------------------------------------ host --

template <int BN, bool kBf16>
static cudaError_t launch_w8a8_bn(const W8A8Args& a, cudaStream_t st) {
    using L = W8Smem<BN>;
    auto kern = w8a8_kernel<BN, kBf16>;
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
    // 3-D copies of kG k-blocks when k is whole k-blocks, else 2-D of one
    CUtensorMap map_w, map_x;
    const bool g3 = a.k % kWK == 0 && L::kG > 1;
    if (g3) {
        if (!encode_3d_blocks(&map_w, a.w_codes, static_cast<uint64_t>(a.n), static_cast<uint64_t>(a.k), kWM, L::kG) ||
            !encode_3d_blocks(&map_x, a.x_codes, static_cast<uint64_t>(a.m), static_cast<uint64_t>(a.k), BN, L::kG))
            return cudaErrorInvalidValue;
    } else {
        if (!encode_2d(&map_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_codes, static_cast<uint64_t>(a.k),
                       static_cast<uint64_t>(a.n), static_cast<uint64_t>(a.k), kWK, kWM))
            return cudaErrorInvalidValue;
        if (!encode_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.x_codes, static_cast<uint64_t>(a.k),
                       static_cast<uint64_t>(a.m), static_cast<uint64_t>(a.k), kWK, BN))
            return cudaErrorInvalidValue;
    }
    const int64_t tiles = ((a.n + kWM - 1) / kWM) * ((a.m + BN - 1) / BN);
    const int64_t nkb = (a.k + kWK - 1) / kWK;
    // whole tiles on persistent CTAs when they nearly fill the GPU, else each
    // tile split over a cluster (a power of two), each rank with at least
    // kWMinKbPerCta k-blocks
    int split = 1;
    if (10 * tiles < 7 * static_cast<int64_t>(sms))
        while (split * 2 <= kWMaxSplit && tiles * split * 2 <= sms && split * 2 * kWMinKbPerCta <= nkb) split *= 2;
    const int64_t grid = split > 1 ? tiles * split : (tiles < sms ? tiles : sms);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(split);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kWThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = split > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, map_w, map_x, a.x_scales, a.w_scales, a.bias, static_cast<uint16_t*>(a.y),
                              a.m, a.n, a.k, split, a.early ? 1 : 0, g3 ? 1 : 0);
}

cudaError_t launch_w8a8(const W8A8Args& a, cudaStream_t st) {
    const bool bf16 = a.out == 1;
    if (a.m <= 16) return bf16 ? launch_w8a8_bn<16, true>(a, st) : launch_w8a8_bn<16, false>(a, st);
    if (a.m <= 32) return bf16 ? launch_w8a8_bn<32, true>(a, st) : launch_w8a8_bn<32, false>(a, st);
    if (a.m <= 64) return bf16 ? launch_w8a8_bn<64, true>(a, st) : launch_w8a8_bn<64, false>(a, st);
    if (a.m <= 128) return bf16 ? launch_w8a8_bn<128, true>(a, st) : launch_w8a8_bn<128, false>(a, st);
    return bf16 ? launch_w8a8_bn<256, true>(a, st) : launch_w8a8_bn<256, false>(a, st);
}

int read_w8a8_device_error() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_w8a8_error, sizeof v) != cudaSuccess) return -1;
    if (v != 0 && cudaMemcpyToSymbol(g_w8a8_error, &zero, sizeof zero) != cudaSuccess) return -1;
    return v;
}

}  // namespace fp8w
