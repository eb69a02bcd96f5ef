// prefill.cu -- kernel K4: the linear layer for many tokens (m > 64) as one
// tcgen05 GEMM with both operands in shared memory.
//
// Page "kadirnar/kernel-agent fp8-weights", section "The contract":
// y[m, n] = round(scale[n] * sum_k x[m, k] * e4m3(q[n, k]) + bias[n]), fp32
// accumulation, one rounding.  For prefill shapes the work is compute-bound,
// so each weight tile is dequantised into shared memory once and multiplied
// by a wide token tile, instead of re-streaming the weight for every 64
// tokens as the skinny kernel (K3) would.
//
// A CTA (one per SM, persistent) walks output tiles of 128 weight rows x BN
// tokens (BN = 128 or 256); the tiles of one weight block are adjacent in
// the walk, so CTAs that run together share it through L2.  K advances in
// blocks of 64 (one 128-byte swizzle atom of 16-bit values a row).
//   warp 0      code tiles (128 rows x 128 codes, 16 KB, TMA, 128-byte
//               swizzle) into their ring
//   warp 2      x tiles (BN tokens x 64) into theirs, independently
//   warp 1      MMA issue: per k-block four tcgen05.mma (M = 128, N = BN,
//               K = 16), A and B by shared-memory descriptor, D in TMEM
//               (two accumulators, so the epilogue drains one tile while
//               the next accumulates)
//   warps 4-7   epilogue: TMEM -> fmaf(acc, scale, bias) -> bf16/fp16 -> y
//   warps 16-19 (per-group form only) the second epilogue warpgroup
//   warps 8-15  two dequantising warpgroups: warpgroup h converts the k-blocks
//               with h = (index in the tile) % 2, one weight row a thread,
//               e4m3 -> bf16/fp16 exactly (value * 2^-120 by byte moves, then
//               * 2^120, or the hardware e4m3 -> f16 conversion), written in
//               the 128-byte swizzled K-major layout the descriptor reads
// Every wait is bounded; a CTA that gives up records a code, raises its abort
// flag, lets its copies and MMAs land and frees TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fp8w_device.cuh"
#include "fp8w_internal.h"

namespace fp8w {

static __device__ int g_prefill_error;

namespace {

constexpr int kPM = 128;                          // weight rows a tile (MMA M, TMEM lanes)
constexpr int kPK = 64;                           // k of an A or x stage
constexpr int kPCodeK = 128;                      // k of a code stage (two k-blocks)
constexpr uint32_t kPCodeBytes = kPM * kPCodeK;   // 16 KB
constexpr uint32_t kPABytes = kPM * kPK * 2;      // 16 KB
constexpr int kPThreads = 512;
constexpr int kPThreadsGrouped = 640;             // + the second epilogue warpgroup
constexpr int kPMmaWarp = 1, kPXWarp = 2, kPFirstEpiWarp = 4, kPFirstDqWarp = 8, kPSecondEpiWarp = 16;
constexpr int kPGAcc = 4;                         // per-group form: group accumulators (128 columns each)
constexpr int kPBarTmem = 1;                      // named barrier: MMA warp + epilogue warps

// Ring depths: the code ring is the deepest, since each CTA streams its
// weight rows from HBM with about a microsecond of copy latency to cover;
// x tiles come from L2.  Both fill 224 KB of shared memory.
template <int BN>
struct PrefillSmem {
    static constexpr int kPCS = BN == 128 ? 6 : 4;  // code stages (16 KB)
    static constexpr int kPAS = 4;                  // dequantised A stages (16 KB)
    static constexpr int kPXS = BN == 128 ? 4 : 3;  // x stages (BN x 64 x 2 B)
    static constexpr uint32_t kXBytes = BN * kPK * 2;
    static constexpr uint32_t kCodesOff = 0;
    static constexpr uint32_t kAOff = kCodesOff + kPCS * kPCodeBytes;
    static constexpr uint32_t kXOff = kAOff + kPAS * kPABytes;
    static constexpr uint32_t kBarOff = kXOff + kPXS * kXBytes;
    // cfull, cempty [kPCS] | afull, aempty [kPAS] | xfull, xempty [kPXS] | dfull, dempty [2] | drain |
    // gfull, gfree [kPGAcc] (per-group form)
    static constexpr uint32_t kGBar0 = 2 * kPCS + 2 * kPAS + 2 * kPXS + 4 + 1;
    static constexpr uint32_t kNumBars = kGBar0 + 2 * kPGAcc;
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;  // TMEM base, abort flag
    static constexpr uint32_t kBytes = kMiscOff + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
    static_assert(kAlloc <= 227 * 1024, "shared memory");
    static constexpr uint32_t kTmemCols = 2 * BN;
    static_assert(kTmemCols <= 512, "TMEM columns");
    static_assert(kPGAcc * BN <= 512 || BN != 128, "TMEM columns (per-group form)");
};

__device__ __forceinline__ void prefill_error(int code, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(&g_prefill_error, 0, 4000 + code);
}

}  // namespace

// The scale forms (kMode):
//  kModeRow      scales[n], in the epilogue.
//  kModeMxFold   E8M0 scale bytes e8[n, k / 32] (page "11. Inference with
//                NVFP4/MXFP8", section "MXFP8-Style FP8"; bf16 only, k % 128
//                == 0): each 32-code group's power of two is folded into the
//                dequantised weight, exactly, and the epilogue adds only the
//                bias.
//  kModeGrouped  one scale per run of gsz = 32, 64 or 128 codes of a row,
//                fp32 scales[n, k / gsz] or E8M0 bytes e8[n, k / 32] (page
//                "B04 Precision & Quantization", section "Post-training
//                quantization versus quantization-aware training", the
//                granularity table's per-group row).  BN = 128: each group's
//                MMAs go to their own TMEM accumulator (a ring of kPGAcc), and
//                eight epilogue warps (two per TMEM lane quarter, 64 tokens
//                each) add every group's sums times its scale into fp32 totals
//                held in registers.
template <int BN, bool kBf16, int kMode>
__global__ void __launch_bounds__(kMode == kModeGrouped ? kPThreadsGrouped : kPThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x,
                   const float* __restrict__ scales, const uint8_t* __restrict__ e8, const float* __restrict__ bias,
                   uint16_t* __restrict__ y, int64_t m, int64_t n, int64_t k, int early, int gsz) {
    constexpr bool kMx = kMode == kModeMxFold;
    constexpr bool kGrp = kMode == kModeGrouped;
    static_assert(!kMx || kBf16, "MX-style scales fold into bf16 weights only");
    static_assert(!kGrp || BN == 128, "per-group form: 128-token tiles");
    using L = PrefillSmem<BN>;
    constexpr int kPCS = L::kPCS, kPAS = L::kPAS, kPXS = L::kPXS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto cfull = [&](int s) { return bar0 + 8u * s; };
    auto cempty = [&](int s) { return bar0 + 8u * (kPCS + s); };
    auto afull = [&](int s) { return bar0 + 8u * (2 * kPCS + s); };
    auto aempty = [&](int s) { return bar0 + 8u * (2 * kPCS + kPAS + s); };
    auto xfull = [&](int s) { return bar0 + 8u * (2 * kPCS + 2 * kPAS + s); };
    auto xempty = [&](int s) { return bar0 + 8u * (2 * kPCS + 2 * kPAS + kPXS + s); };
    auto dfull = [&](int d) { return bar0 + 8u * (2 * kPCS + 2 * kPAS + 2 * kPXS + d); };
    auto dempty = [&](int d) { return bar0 + 8u * (2 * kPCS + 2 * kPAS + 2 * kPXS + 2 + d); };
    const uint32_t drain = bar0 + 8u * (2 * kPCS + 2 * kPAS + 2 * kPXS + 4);
    auto gfull = [&](int b) { return bar0 + 8u * (L::kGBar0 + b); };
    auto gfree = [&](int b) { return bar0 + 8u * (L::kGBar0 + kPGAcc + b); };
    constexpr uint32_t kTmemCols = kGrp ? 512u : L::kTmemCols;
    constexpr int kEpiWarps = kGrp ? 8 : 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t token_tiles = (m + BN - 1) / BN;
    const int64_t tiles = ((n + kPM - 1) / kPM) * token_tiles;
    const int nkb = static_cast<int>((k + kPK - 1) / kPK);          // k-blocks a tile
    const int ncs = static_cast<int>((k + kPCodeK - 1) / kPCodeK);  // code stages a tile

    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < kPCS; ++s) {
                mbar_init(cfull(s), 1);
                mbar_init(cempty(s), 8);  // the eight dequantising warps
            }
            for (int s = 0; s < kPAS; ++s) {
                mbar_init(afull(s), 4);   // the four warps of one warpgroup
                mbar_init(aempty(s), 1);  // MMA commit
            }
            for (int s = 0; s < kPXS; ++s) {
                mbar_init(xfull(s), 1);
                mbar_init(xempty(s), 1);
            }
            for (int d = 0; d < 2; ++d) {
                mbar_init(dfull(d), 1);
                mbar_init(dempty(d), 4);  // the four epilogue warps
            }
            mbar_init(drain, 1);
            for (int b = 0; b < kPGAcc; ++b) {
                mbar_init(gfull(b), 1);           // MMA commit
                mbar_init(gfree(b), kEpiWarps);   // every epilogue warp (per-group form)
            }
            *abort_flag = 0;
            tma_prefetch_desc(&map_codes);
            tma_prefetch_desc(&map_x);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    uint32_t tmem = 0;
    const bool epi_warp = (warp >= kPFirstEpiWarp && warp < kPFirstDqWarp) || (kGrp && warp >= kPSecondEpiWarp);
    if (warp == kPMmaWarp || epi_warp) {
        if (warp == kPMmaWarp) {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        asm volatile("bar.sync %0, %1;" ::"n"(kPBarTmem), "n"(32 * (1 + kEpiWarps)) : "memory");
        tc_fence_after();
        tmem = *tmem_slot;
    }

    if (warp == 0) {
        // --------------------------------------------------- code producer --
        if (lane == 0) {
            const uint64_t pol_codes = policy_evict_first();
            // the codes may come from the previous kernel, unless the caller
            // states that they were complete before it started
            if (!early) pdl_wait();
            int64_t cs_n = 0;  // code stages issued
            for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
                const int64_t cb = t / token_tiles;
                bool ok = true;
                for (int cs = 0; cs < ncs; ++cs) {
                    const int s = static_cast<int>(cs_n % kPCS);
                    if (!mbar_wait(cempty(s), static_cast<uint32_t>((cs_n / kPCS) & 1) ^ 1u, abort_flag)) {
                        prefill_error(kErrWaitSlot, abort_flag);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(cfull(s), kPCodeBytes);
                    tma_load_2d(sbase + L::kCodesOff + s * kPCodeBytes, &map_codes, cs * kPCodeK,
                                static_cast<int32_t>(cb * kPM), cfull(s), pol_codes);
                    ++cs_n;
                }
                if (!ok) break;
            }
            if (*abort_flag) {
                // let the copies still in flight land before the CTA exits
                for (int64_t i = (cs_n > kPCS ? cs_n - kPCS : 0); i < cs_n; ++i)
                    if (!mbar_wait_drain(cfull(static_cast<int>(i % kPCS)), static_cast<uint32_t>((i / kPCS) & 1)))
                        atomicCAS(&g_prefill_error, 0, 4000 + kErrWaitDrain);
            }
        }
    } else if (warp == kPXWarp) {
        // ------------------------------------------------------ x producer --
        if (lane == 0) {
            const uint64_t pol_x = policy_evict_last();
            pdl_wait();  // x may come from the previous kernel
            int64_t kb_n = 0;  // k-blocks issued
            for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
                const int64_t cb = t / token_tiles, tb = t - cb * token_tiles;
                bool ok = true;
                for (int j = 0; j < nkb; ++j) {
                    const int xs = static_cast<int>(kb_n % kPXS);
                    if (!mbar_wait(xempty(xs), static_cast<uint32_t>((kb_n / kPXS) & 1) ^ 1u, abort_flag)) {
                        prefill_error(kErrWaitSlot, abort_flag);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(xfull(xs), L::kXBytes);
                    tma_load_2d(sbase + L::kXOff + xs * L::kXBytes, &map_x, j * kPK, static_cast<int32_t>(tb * BN),
                                xfull(xs), pol_x);
                    ++kb_n;
                }
                if (!ok) break;
            }
            if (*abort_flag) {
                for (int64_t i = (kb_n > kPXS ? kb_n - kPXS : 0); i < kb_n; ++i)
                    if (!mbar_wait_drain(xfull(static_cast<int>(i % kPXS)), static_cast<uint32_t>((i / kPXS) & 1)))
                        atomicCAS(&g_prefill_error, 0, 4000 + kErrWaitDrain);
            }
        }
    } else if (kGrp && warp == kPMmaWarp) {
        // ------------------------------------- MMA issue, per-group form --
        // The MMA at k = kg starts group kg / gsz when kg % gsz == 0 (into
        // accumulator Gc % kPGAcc, once the epilogue has drained its last
        // group) and ends it when kg + 16 reaches the next multiple of gsz
        // (k % gsz == 0, so no group is cut off by the end of k).
        constexpr uint32_t idesc = idesc_f16(kBf16, BN);
        // accumulators hold at most one k-block (g = 128 takes two, one per
        // 64-code half, each scaled by the group's scale)
        const int asz = gsz < kPK ? gsz : kPK;
        int64_t kb_n = 0;
        int Gc = 0, gb = 0;  // accumulators issued (below 2^31), and the current one
        uint32_t g_tmem = tmem;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            for (int j = 0; j < nkb; ++j, ++kb_n) {
                const int as = static_cast<int>(kb_n % kPAS), xs = static_cast<int>(kb_n % kPXS);
                if (!mbar_wait_warp(afull(as), static_cast<uint32_t>((kb_n / kPAS) & 1), abort_flag) ||
                    !mbar_wait_warp(xfull(xs), static_cast<uint32_t>((kb_n / kPXS) & 1), abort_flag)) {
                    if (lane == 0) prefill_error(kErrWaitDequant, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = sbase + L::kAOff + as * kPABytes;
                const uint32_t x_addr = sbase + L::kXOff + xs * L::kXBytes;
#pragma unroll
                for (int kk = 0; kk < kPK / 16; ++kk) {
                    const int64_t kg = static_cast<int64_t>(j) * kPK + kk * 16;
                    if (kg >= k) break;
                    const int qg = static_cast<int>(kg & (asz - 1));
                    if (qg == 0) {
                        gb = Gc & (kPGAcc - 1);
                        if (!mbar_wait_warp(gfree(gb), static_cast<uint32_t>(((Gc / kPGAcc) & 1) ^ 1), abort_flag)) {
                            if (lane == 0) prefill_error(kErrWaitMma, abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        g_tmem = tmem + static_cast<uint32_t>(gb * BN);
                    }
                    mma_f16_ss_warp(g_tmem, smem_desc_sw128_kmajor(a_addr + kk * 32),
                                    smem_desc_sw128_kmajor(x_addr + kk * 32), idesc, qg != 0);
                    if (qg + 16 == asz) {
                        tc_commit_warp(gfull(gb));
                        ++Gc;
                    }
                }
                // both stages are free once these MMAs have read them
                tc_commit_warp(aempty(as));
                tc_commit_warp(xempty(xs));
                __syncwarp();
                if (!ok) break;
            }
        }
        // every MMA issued above completes before TMEM is released
        tc_commit_warp(drain);
        if (!mbar_wait_drain(drain, 0) && lane == 0) atomicCAS(&g_prefill_error, 0, 4000 + kErrWaitDrain);
        __syncwarp();
    } else if (kGrp && epi_warp) {
        // --------------------------------------- epilogue, per-group form --
        // Warps 4-7 take tokens 0-63 of a tile, warps 16-19 tokens 64-127
        // (warp w reads TMEM lanes 32 (w % 4) ..); thread r holds weight row
        // r's totals for its 64 tokens as fp32 pairs.
        const int quarter = warp & 3;
        const int half = warp >= kPSecondEpiWarp ? 1 : 0;
        const int r = quarter * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(half * 64);
        const int nsc = static_cast<int>(e8 ? (k >> 5) : k / gsz);  // scales a row == groups a tile
        const int asz = gsz < kPK ? gsz : kPK;                       // k of an accumulator
        const int apg = gsz / asz;                                   // accumulators a group (1 or 2)
        const int nacc = nsc * apg;                                  // accumulators a tile
        auto scale_at = [&](int64_t col, int j) -> float {
            if (col >= n) return 0.0f;  // rows past n hold zero codes
            return e8 ? e8m0_to_f32(__ldg(e8 + col * nsc + j)) : __ldg(scales + col * nsc + j);
        };
        pdl_wait();  // y may still be read, and the scales written, by the previous kernel
        int Gc = 0;  // accumulators drained (below 2^31: tiles a CTA x k / 32)
        bool ok = true;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            const int64_t cb = t / token_tiles, tb = t - cb * token_tiles;
            const int64_t col = cb * kPM + r;
            const int64_t tok0 = tb * BN;
            const int ntok = static_cast<int>(m - tok0 < BN ? m - tok0 : BN);
            const int mine = ntok - half * 64;  // tokens of this warp's half (may be <= 0)
            uint64_t tot2[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) tot2[i] = 0ull;
            float s_next = scale_at(col, 0);
            for (int ai = 0; ai < nacc; ++ai, ++Gc) {
                // accumulator ai is (part of) group ai / apg
                const float s = s_next;
                if (ai + 1 < nacc && (ai + 1) % apg == 0) s_next = scale_at(col, (ai + 1) / apg);
                const int gb = Gc & (kPGAcc - 1);
                if (!mbar_wait_warp(gfull(gb), static_cast<uint32_t>((Gc / kPGAcc) & 1), abort_flag)) {
                    if (lane == 0) prefill_error(kErrWaitMma, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t s2 = pack2(s, s);
                // 32 tokens a round trip (two loads in flight)
#pragma unroll
                for (int c = 0; c < 4; c += 2) {
                    if (c * 16 >= mine) break;
                    uint32_t v0[16], v1[16];
                    tmem_ld2_x16_sync(lane_addr + static_cast<uint32_t>(gb * BN + c * 16),
                                      lane_addr + static_cast<uint32_t>(gb * BN + c * 16 + 16), v0, v1);
                    ffma2_x16(tot2 + c * 8, v0, s2);
                    ffma2_x16(tot2 + c * 8 + 8, v1, s2);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(gfree(gb));
            }
            if (!ok) break;
            if (col < n) {
                const float b = bias ? bias[col] : 0.0f;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    if (i >= mine) break;
                    const float v = __uint_as_float(static_cast<uint32_t>(tot2[i >> 1] >> (32 * (i & 1))));
                    y[(tok0 + half * 64 + i) * n + col] = round_out<kBf16>(v + b);
                }
            }
        }
    } else if (warp == kPMmaWarp) {
        // ------------------------------------------------------ MMA issue --
        constexpr uint32_t idesc = idesc_f16(kBf16, BN);
        int64_t kb_n = 0;
        int tile_n = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tile_n) {
            const int d = tile_n & 1;
            if (!mbar_wait_warp(dempty(d), static_cast<uint32_t>((tile_n >> 1) & 1) ^ 1u, abort_flag)) {
                if (lane == 0) prefill_error(kErrWaitMma, abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(d * BN);
            for (int j = 0; j < nkb; ++j, ++kb_n) {
                const int as = static_cast<int>(kb_n % kPAS), xs = static_cast<int>(kb_n % kPXS);
                if (!mbar_wait_warp(afull(as), static_cast<uint32_t>((kb_n / kPAS) & 1), abort_flag) ||
                    !mbar_wait_warp(xfull(xs), static_cast<uint32_t>((kb_n / kPXS) & 1), abort_flag)) {
                    if (lane == 0) prefill_error(kErrWaitDequant, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = sbase + L::kAOff + as * kPABytes;
                const uint32_t x_addr = sbase + L::kXOff + xs * L::kXBytes;
#pragma unroll
                for (int kk = 0; kk < kPK / 16; ++kk)
                    mma_f16_ss_warp(d_tmem, smem_desc_sw128_kmajor(a_addr + kk * 32),
                                    smem_desc_sw128_kmajor(x_addr + kk * 32), idesc, j > 0 || kk > 0);
                // both stages are free once these MMAs have read them
                tc_commit_warp(aempty(as));
                tc_commit_warp(xempty(xs));
                __syncwarp();
            }
            if (!ok) break;
            tc_commit_warp(dfull(d));
            __syncwarp();
        }
        // every MMA issued above completes before TMEM is released
        tc_commit_warp(drain);
        if (!mbar_wait_drain(drain, 0) && lane == 0) atomicCAS(&g_prefill_error, 0, 4000 + kErrWaitDrain);
        __syncwarp();
    } else if (warp >= kPFirstEpiWarp && warp < kPFirstDqWarp) {
        // ------------------------------------------------------- epilogue --
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // weight row within the tile == TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        pdl_wait();  // y may still be read by the previous kernel
        int tile_n = 0;
        for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++tile_n) {
            const int64_t cb = t / token_tiles, tb = t - cb * token_tiles;
            const int d = tile_n & 1;
            if (!mbar_wait_warp(dfull(d), static_cast<uint32_t>((tile_n >> 1) & 1), abort_flag)) {
                if (lane == 0) prefill_error(kErrWaitMma, abort_flag);
                break;
            }
            tc_fence_after();
            const int64_t col = cb * kPM + r;
            const float sc = kMx ? 1.0f : col < n ? scales[col] : 0.0f;
            const float b = (bias && col < n) ? bias[col] : 0.0f;
            const int64_t tok0 = tb * BN;
            const int ntok = static_cast<int>(m - tok0 < BN ? m - tok0 : BN);
            for (int c0 = 0; c0 < ntok; c0 += 16) {
                uint32_t v[16];
                tmem_ld_x16_sync(lane_addr + static_cast<uint32_t>(d * BN + c0), v);
                if (col < n) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (c0 + i < ntok)
                            y[(tok0 + c0 + i) * n + col] = round_out<kBf16>(fmaf(__uint_as_float(v[i]), sc, b));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty(d));
        }
    } else if (warp >= kPFirstDqWarp && warp < kPFirstDqWarp + 8) {
        // ---------------------------------------------------- dequantising --
        const int h = (warp - kPFirstDqWarp) >> 2;  // warpgroup: k-blocks with j % 2 == h
        const int r = (warp & 3) * 32 + lane;       // weight row of the tile
        const uint32_t swz = static_cast<uint32_t>(r & 7);
        // MX: the row's two scale bytes of this warpgroup's k-blocks, loaded
        // one of them ahead; (mx_t, mx_j) is the one after the current
        uint32_t mx_next = 0x7F7Fu;
        int64_t mx_t = blockIdx.x;
        int mx_j = h;
        auto mx_load = [&]() -> uint32_t {
            const int64_t wrow = (mx_t / token_tiles) * kPM + r;
            return wrow < n ? static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(e8 + wrow * (k >> 5)) + mx_j))
                            : 0x7F7Fu;  // rows past n hold zero codes: any scale does
        };
        auto mx_step = [&]() {
            if (mx_t < tiles && mx_j < nkb) mx_next = mx_load();
            mx_j += 2;
            if (mx_j >= nkb) {
                mx_j = h;
                mx_t += gridDim.x;
            }
        };
        if constexpr (kMx) {
            if (!early) pdl_wait();  // the scales may come from the previous kernel
            mx_step();
        }
        int64_t cs_n = 0, kb_base = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, kb_base += nkb) {
            for (int cs = 0; cs < ncs; ++cs, ++cs_n) {
                const int s = static_cast<int>(cs_n % kPCS);
                if (!mbar_wait_warp(cfull(s), static_cast<uint32_t>((cs_n / kPCS) & 1), abort_flag)) {
                    if (lane == 0) prefill_error(kErrWaitTma, abort_flag);
                    ok = false;
                    break;
                }
                const int j = 2 * cs + h;
                const bool mine = j < nkb;
                // this warpgroup's half of the row: chunks 4h .. 4h + 3 (64 codes)
                uint4 cw[4];
                const uint32_t row = sbase + L::kCodesOff + s * kPCodeBytes + static_cast<uint32_t>(r) * 128u;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    cw[q] = mine ? lds128(row + (((4u * h + q) ^ swz) << 4)) : make_uint4(0u, 0u, 0u, 0u);
                __syncwarp();
                if (lane == 0) mbar_arrive(cempty(s));
                if (!mine) continue;
                const int64_t kb = kb_base + j;
                const int as = static_cast<int>(kb % kPAS);
                if (!mbar_wait_warp(aempty(as), static_cast<uint32_t>((kb / kPAS) & 1) ^ 1u, abort_flag)) {
                    if (lane == 0) prefill_error(kErrWaitMma, abort_flag);
                    ok = false;
                    break;
                }
                const uint32_t arow = sbase + L::kAOff + as * kPABytes + static_cast<uint32_t>(r) * 128u;
                // MX: the k-block's two groups (chunks 0-1 and 2-3); a byte above
                // 134 anywhere in the warp takes two multiplies
                uint32_t mx_word = 0u, mul[2] = {kBf16x2Pow2_120, kBf16x2Pow2_120};
                bool twice = false;
                if constexpr (kMx) {
                    mx_word = mx_next;
                    mx_step();
                    twice = __any_sync(0xffffffffu, (mx_word & 0xFFu) > 134u || (mx_word >> 8) > 134u);
                    if (!twice) {
                        mul[0] = mx_first_mul(mx_word & 0xFFu);
                        mul[1] = mx_first_mul(mx_word >> 8);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t v[8];
                    const uint32_t w4[4] = {cw[q].x, cw[q].y, cw[q].z, cw[q].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if constexpr (kMx) {
                            e4m3x4_to_bf16x2_mul(w4[e], v[2 * e], v[2 * e + 1], mul[q >> 1]);
                        } else if constexpr (kBf16) {
                            e4m3x4_to_bf16x2(w4[e], v[2 * e], v[2 * e + 1]);
                        } else {
                            e4m3x4_to_f16x2(w4[e], v[2 * e], v[2 * e + 1]);
                        }
                    }
                    if constexpr (kMx) {
                        if (twice) {
                            const uint32_t m2 = mx_second_mul((mx_word >> (8 * (q >> 1))) & 0xFFu);
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = bf16x2_mul(v[e], m2);
                        }
                    }
                    // 16 values = logical chunks 2q and 2q + 1 of the A row
                    sts128(arow + (((2u * q) ^ swz) << 4), v[0], v[1], v[2], v[3]);
                    sts128(arow + (((2u * q + 1u) ^ swz) << 4), v[4], v[5], v[6], v[7]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull(as));
            }
        }
    }

    __syncthreads();
    if (warp == kPMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int BN, bool kBf16, int kMode = kModeRow>
static cudaError_t launch_bn(const LinearArgs& a, cudaStream_t st) {
    using L = PrefillSmem<BN>;
    constexpr bool kMx = kMode == kModeMxFold;
    constexpr bool kGrp = kMode == kModeGrouped;
    auto kern = prefill_kernel<BN, kBf16, kMode>;
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
                   static_cast<uint64_t>(a.n), static_cast<uint64_t>(a.k), kPCodeK, kPM))
        return cudaErrorInvalidValue;
    if (!encode_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.x, static_cast<uint64_t>(a.k),
                   static_cast<uint64_t>(a.m), static_cast<uint64_t>(a.k) * 2, kPK, BN))
        return cudaErrorInvalidValue;
    const int64_t tiles = ((a.n + kPM - 1) / kPM) * ((a.m + BN - 1) / BN);
    const int64_t grid = tiles < sms ? tiles : sms;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGrp ? kPThreadsGrouped : kPThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool bytes = kMx || (kGrp && a.e8m0);
    const float* sc = bytes ? nullptr : a.scales;
    const uint8_t* e8 = bytes ? reinterpret_cast<const uint8_t*>(a.scales) : nullptr;
    return cudaLaunchKernelEx(&cfg, kern, map_codes, map_x, sc, e8, a.bias, static_cast<uint16_t*>(a.y), a.m, a.n,
                              a.k, a.early ? 1 : 0, kGrp ? static_cast<int>(a.group) : 0);
}

cudaError_t launch_prefill(const LinearArgs& a, cudaStream_t st) {
    const bool bf16 = a.act == 1;
    if (a.group != 0 && (!a.e8m0 || !bf16)) {
        // per-group scales (fp32, or E8M0 bytes with fp16 activations)
        if (a.k % a.group != 0 || (a.group != 32 && a.group != 64 && a.group != 128) || (a.e8m0 && a.group != 32))
            return cudaErrorInvalidValue;
        return bf16 ? launch_bn<128, true, kModeGrouped>(a, st) : launch_bn<128, false, kModeGrouped>(a, st);
    }
    if (a.e8m0) {
        // MX-style scales: bf16 activations, k % 128 == 0 (checked by the caller)
        if (!bf16 || a.group != 32 || a.k % 128 != 0) return cudaErrorInvalidValue;
        return a.m <= 128 ? launch_bn<128, true, kModeMxFold>(a, st) : launch_bn<256, true, kModeMxFold>(a, st);
    }
    // 128-token tiles up to 128 tokens, 256 beyond
    if (a.m <= 128) return bf16 ? launch_bn<128, true>(a, st) : launch_bn<128, false>(a, st);
    return bf16 ? launch_bn<256, true>(a, st) : launch_bn<256, false>(a, st);
}

int read_prefill_device_error() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof v) != cudaSuccess) return -1;
    if (v != 0 && cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof zero) != cudaSuccess) return -1;
    return v;
}

}  // namespace fp8w
