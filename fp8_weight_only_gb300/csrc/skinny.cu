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
//  * Persistent grid, at most one CTA per SM.  The work is the list of units
//    (channel tile of 128, k-block of 128); CTA c takes the contiguous units
//    [c*U/P, (c+1)*U/P).  P is the tile count when that nearly fills the GPU
//    (every tile whole, nothing to combine), else a multiple of it or the SM
//    count (stream-K).  A tile that straddles CTAs is finished by the last
//    contributor to arrive: partial fp32 tiles go to a caller-provided
//    workspace and are summed in CTA order (deterministic); nothing waits on
//    another CTA.  A CTA first runs the partial piece at the end of its
//    range, so its fix-ups overlap its other work.
//  * Units are dealt round-robin to three lanes; lane g is dequantising
//    warpgroup g plus MMA issuer g, with private rings in shared memory and
//    TMEM, so every mbarrier has one producer and one in-order consumer.
//    (Consumers taking turns on one shared ring could run two phases ahead
//    of a slow one and pass a completed phase of the same parity.)
//  * Warp 0 streams each unit's 128 x 128 code tile into its lane's code
//    slots, and warp 4 its M x 128 activation tile into the lane's
//    activation slots, with TMA (128-byte swizzle; rows past N or M and k past
//    K read as zeros).  A code tile is freed as soon as it has been read, an
//    activation tile when its MMAs are done.
//  * In each lane, thread r of the warpgroup reads the 128 codes of channel
//    r (conflict-free through the swizzle), converts them exactly to bf16 /
//    fp16 in registers and stores them with tcgen05.st into the lane's TMEM A
//    slot, where they are the A operand of the MMA (A from tensor memory: the
//    dequantised weight never touches shared memory).
//  * Each lane's MMA warp (one issuing thread) issues tcgen05.mma.kind::f16
//    (M = 128, N = 16 or 32 tokens, K = 16) into the lane's double-buffered
//    TMEM accumulator and returns slots with tcgen05.commit.  A tcgen05.mma
//    costs its issuing thread tens of cycles whatever its size, so one issuer
//    could not keep up with the weight stream at N <= 32; three can.
//  * One epilogue warpgroup reads the lanes' accumulators of a finished tile
//    with tcgen05.ld (thread r holds channel r for every token), sums them in
//    a fixed order while the next tile accumulates, and stores
//    y = round(fma(acc, scale, bias)) or, for a split tile, its partial.
//  * The control loops divide nothing per unit: a cursor walks (tile,
//    k-block), since a 64-bit division costs a lone thread hundreds of cycles.
//
// Every wait is bounded: on a timeout the CTA records an error code (the
// role and the barrier that gave up), raises an abort flag that ends every
// role's loop, lets its in-flight copies and MMAs finish, frees TMEM and
// exits.
#include <mutex>

#include "fp8w_device.cuh"
#include "fp8w_internal.h"
#include "../../include/fp8w.h"

namespace fp8w {

static __device__ int g_skinny_error;

constexpr int kTileN = 128;                 // output channels per tile (MMA M)
constexpr int kBlockK = 128;                // k per unit
constexpr int kLanes = 3;                   // dequant warpgroup + MMA issuer pairs
// warps: 0 code TMA, 1..3 MMA issuers (warp 1 also owns TMEM), 4 x TMA,
// 5..8 epilogue, 9..20 dequant (4 per lane)
constexpr int kXWarp = 1 + kLanes;
constexpr int kFirstEpilogueWarp = kXWarp + 1;
constexpr int kFirstDequantWarp = kFirstEpilogueWarp + 4;
constexpr int kThreads = 32 * (kFirstDequantWarp + 4 * kLanes);  // 672
constexpr int kTmemCols = 512;              // one CTA per SM
constexpr int kAColsPerSlot = kBlockK / 2;  // two 16-bit values per column
constexpr int kDCol0 = kLanes * kAColsPerSlot;  // 192: accumulators after the A slots
constexpr uint32_t kCodeStageBytes = kTileN * kBlockK;  // 16 KB
constexpr int kMaxNT = 32;
static_assert(kDCol0 + kLanes * 2 * kMaxNT <= kTmemCols, "TMEM columns");

template <int NT>
struct SkinnySmem {
    // per lane: code slots (freed once read) and activation slots (freed
    // when the MMA is done), as many as ~221 KB of shared memory holds
    static constexpr int kCodeSlots = NT == 16 ? 4 : 3;
    static constexpr int kXSlots = NT == 16 ? 2 : 3;
    static constexpr uint32_t kXBoxBytes = NT * 128;          // 64 k x NT rows x 2 B
    static constexpr uint32_t kXStageBytes = 2 * kXBoxBytes;  // 128 k
    static constexpr uint32_t kCodesOff = 0;
    static constexpr uint32_t kXOff = kCodesOff + kLanes * kCodeSlots * kCodeStageBytes;
    static constexpr uint32_t kBarOff = kXOff + kLanes * kXSlots * kXStageBytes;
    // per lane: cfull, cempty [kCodeSlots]; xfull, xempty [kXSlots]; afull;
    // aempty; dready, dfree [2]; drain
    static constexpr uint32_t kBarsPerLane = 2 * kCodeSlots + 2 * kXSlots + 7;
    static constexpr uint32_t kNumBars = kLanes * kBarsPerLane;
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
constexpr size_t skinny_workspace_bytes(int p) {
    return kWsCountersBytes + 2 * static_cast<size_t>(p) * ws_slot_floats() * 4;
}
// A split CTA takes at least this many units, so a small matrix is not cut
// into more partial tiles than it has k-blocks to share.
constexpr int64_t kMinUnitsPerCta = 4;
// Contributors' partials are read this many at a time, all loads in flight
// before any add.
constexpr int kFixupBatch = 2;

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

// Walks a CTA's units in processing order without divisions: (tile, kb) of
// the current unit; after the moved piece [t_last*nkb, u1) it jumps to u0.
struct UnitCursor {
    int it, len0;
    int tile, kb, nkb;
    int tile0, kb0;  // position of u0
    __device__ __forceinline__ void next() {
        ++it;
        if (it == len0) {
            tile = tile0;
            kb = kb0;
        } else if (++kb == nkb) {
            kb = 0;
            ++tile;
        }
    }
    // units left in the current tile within the current piece
    __device__ __forceinline__ int seg_left(int iters) const {
        const int piece_end = it < len0 ? len0 : iters;
        return min(nkb - kb, piece_end - it);
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

// The recorded code is role * 1000 + 1 + the barrier's index in shared
// memory (0 when no barrier applies), so a report names the wait that gave up.
__device__ __forceinline__ void record_error(int code, volatile int* abort_flag, uint32_t bar = 0, uint32_t bar0 = 0) {
    *abort_flag = 1;
    atomicCAS(&g_skinny_error, 0, code * 1000 + (bar ? static_cast<int>((bar - bar0) / 8) + 1 : 0));
}

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Arrival count of a split tile: release orders this CTA's partial stores
// (made visible to this thread by the preceding CTA barrier) before the
// increment; acquire orders the last contributor's reads after it.
__device__ __forceinline__ uint32_t arrive_acq_rel(uint32_t* counter) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// lane g has a unit among [it0, it0 + len) iff one index is = g mod kLanes
__device__ __forceinline__ bool lane_has(int g, int it0, int len) {
    return len >= kLanes || ((g - it0 % kLanes + kLanes) % kLanes) < len;
}

template <int NT, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x,
                  const float* __restrict__ scales, const float* __restrict__ bias, uint16_t* __restrict__ y,
                  uint8_t* __restrict__ workspace, int m_rows, int m_row0, int64_t n, int64_t k) {
    using L = SkinnySmem<NT>;
    constexpr int kCS = L::kCodeSlots, kXS = L::kXSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto lbar = [&](int g, int i) { return bar0 + 8u * (g * L::kBarsPerLane + i); };
    auto cfull = [&](int g, int s) { return lbar(g, s); };
    auto cempty = [&](int g, int s) { return lbar(g, kCS + s); };
    auto xfull = [&](int g, int s) { return lbar(g, 2 * kCS + s); };
    auto xempty = [&](int g, int s) { return lbar(g, 2 * kCS + kXS + s); };
    auto afull = [&](int g) { return lbar(g, 2 * kCS + 2 * kXS); };
    auto aempty = [&](int g) { return lbar(g, 2 * kCS + 2 * kXS + 1); };
    auto dready = [&](int g, int d) { return lbar(g, 2 * kCS + 2 * kXS + 2 + d); };
    auto dfree = [&](int g, int d) { return lbar(g, 2 * kCS + 2 * kXS + 4 + d); };
    auto drain = [&](int g) { return lbar(g, 2 * kCS + 2 * kXS + 6); };
    auto code_smem = [&](int g, int s) { return L::kCodesOff + (g * kCS + s) * kCodeStageBytes; };
    auto x_smem = [&](int g, int s) { return L::kXOff + (g * kXS + s) * L::kXStageBytes; };
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
    // Processing order: when the range ends inside a tile, that partial
    // piece [t_last*nkb, u1) runs first, then the rest from u0.
    const int64_t t_first = u0 / nkb, t_last = (u1 - 1) / nkb;
    const int kb_first = static_cast<int>(u0 - t_first * nkb);
    const bool moved = t_last > t_first && (u1 % nkb) != 0;
    const int len0 = moved ? static_cast<int>(u1 - t_last * nkb) : 0;
    auto cursor0 = [=]() {
        UnitCursor cu;
        cu.it = 0;
        cu.len0 = len0;
        cu.nkb = static_cast<int>(nkb);
        cu.tile0 = static_cast<int>(t_first);
        cu.kb0 = kb_first;
        cu.tile = moved ? static_cast<int>(t_last) : static_cast<int>(t_first);
        cu.kb = moved ? 0 : kb_first;
        return cu;
    };

    if (threadIdx.x == 0) {
        for (int g = 0; g < kLanes; ++g) {
            for (int s = 0; s < kCS; ++s) {
                mbar_init(cfull(g, s), 1);
                mbar_init(cempty(g, s), 4);
            }
            for (int s = 0; s < kXS; ++s) {
                mbar_init(xfull(g, s), 1);
                mbar_init(xempty(g, s), 1);
            }
            mbar_init(afull(g), 4);
            mbar_init(aempty(g), 1);
            for (int d = 0; d < 2; ++d) {
                mbar_init(dready(g, d), 1);
                mbar_init(dfree(g, d), 4);
            }
            mbar_init(drain(g), 1);
        }
        *abort_flag = 0;
        *ep_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&map_codes);
        tma_prefetch_desc(&map_x);
    }
    __syncthreads();
    // let the next kernel in the stream start launching; its CTAs wait for
    // this grid to complete before they read or write global memory
    pdl_launch_dependents();
    // TMEM is allocated by warp 1 while the code producer already streams;
    // every other warp meets warp 1 at named barrier 2 first.
    uint32_t tmem = 0;
    if (warp != 0) {
        if (warp == 1) {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        asm volatile("bar.sync 2, %0;" ::"n"(kThreads - 32) : "memory");
        tc_fence_after();
        tmem = *tmem_slot;
    }

    if (warp == 0) {
        // ----------------------------------------------- code-tile producer --
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_first();
            pdl_wait();
            UnitCursor cu = cursor0();
            int g = 0, j = 0;  // lane of the unit, and its index within the lane
            int issued = 0;
            for (int it = 0; it < iters; ++it, cu.next()) {
                const int s = j % kCS;
                if (!mbar_wait(cempty(g, s), static_cast<uint32_t>(((j / kCS) & 1) ^ 1), abort_flag)) {
                    record_error(kErrWaitSlot, abort_flag, cempty(g, s), bar0);
                    break;
                }
                mbar_arrive_expect_tx(cfull(g, s), kCodeStageBytes);
                tma_load_2d(sbase + code_smem(g, s), &map_codes, cu.kb * kBlockK, cu.tile * kTileN, cfull(g, s),
                            pol_stream);
                ++issued;
                if (++g == kLanes) {
                    g = 0;
                    ++j;
                }
            }
            if (*abort_flag) {
                // let every copy still in flight land before the CTA exits:
                // the last fills of each lane's slots
                for (int g2 = 0; g2 < kLanes; ++g2) {
                    const int n_g2 = (issued - g2 + kLanes - 1) / kLanes;
                    for (int jj = (n_g2 > kCS ? n_g2 - kCS : 0); jj < n_g2; ++jj)
                        if (!mbar_wait_drain(cfull(g2, jj % kCS), static_cast<uint32_t>((jj / kCS) & 1)))
                            atomicCAS(&g_skinny_error, 0, kErrWaitDrain * 1000);
                }
            }
        }
    } else if (warp == kXWarp) {
        // ----------------------------------------- activation-tile producer --
        if (lane == 0) {
            const uint64_t pol_keep = policy_evict_last();
            pdl_wait();
            UnitCursor cu = cursor0();
            int g = 0, j = 0;
            int issued = 0;
            for (int it = 0; it < iters; ++it, cu.next()) {
                const int s = j % kXS;
                if (!mbar_wait(xempty(g, s), static_cast<uint32_t>(((j / kXS) & 1) ^ 1), abort_flag)) {
                    record_error(kErrWaitSlot, abort_flag, xempty(g, s), bar0);
                    break;
                }
                const int32_t kk = cu.kb * kBlockK;
                const uint32_t xs = sbase + x_smem(g, s);
                mbar_arrive_expect_tx(xfull(g, s), L::kXStageBytes);
                tma_load_2d(xs, &map_x, kk, m_row0, xfull(g, s), pol_keep);
                tma_load_2d(xs + L::kXBoxBytes, &map_x, kk + 64, m_row0, xfull(g, s), pol_keep);
                ++issued;
                if (++g == kLanes) {
                    g = 0;
                    ++j;
                }
            }
            if (*abort_flag) {
                for (int g2 = 0; g2 < kLanes; ++g2) {
                    const int n_g2 = (issued - g2 + kLanes - 1) / kLanes;
                    for (int jj = (n_g2 > kXS ? n_g2 - kXS : 0); jj < n_g2; ++jj)
                        if (!mbar_wait_drain(xfull(g2, jj % kXS), static_cast<uint32_t>((jj / kXS) & 1)))
                            atomicCAS(&g_skinny_error, 0, kErrWaitDrain * 1000);
                }
            }
        }
    } else if (warp < kXWarp) {
        // ---------------------------------------------- MMA issuers (1..3) --
        const int me = warp - 1;
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBf16, NT);
            UnitCursor cu = cursor0();
            int seg = 0;
            int j = 0;  // this lane's units so far
            bool failed = false;
            for (int it = 0; it < iters && !failed; ++seg) {
                // one segment (the units of one tile) per pass
                const int seg_len = cu.seg_left(iters);
                const int d = seg & 1;
                const uint32_t d_tmem = tmem + kDCol0 + (me * 2 + d) * NT;
                // the epilogue has drained this accumulator (two segments ago)
                if (!mbar_wait(dfree(me, d), static_cast<uint32_t>(((seg >> 1) & 1) ^ 1), abort_flag)) {
                    record_error(kErrWaitMma, abort_flag, dfree(me, d), bar0);
                    break;
                }
                bool mine_first = true, any = false;
                for (int jj = 0; jj < seg_len; ++jj, ++it, cu.next()) {
                    if (it % kLanes != me) continue;
                    const int s = j % kXS;
                    if (!mbar_wait(xfull(me, s), static_cast<uint32_t>((j / kXS) & 1), abort_flag)) {
                        record_error(kErrWaitTma, abort_flag, xfull(me, s), bar0);
                        failed = true;
                        break;
                    }
                    if (!mbar_wait(afull(me), static_cast<uint32_t>(j & 1), abort_flag)) {
                        record_error(kErrWaitDequant, abort_flag, afull(me), bar0);
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xs = sbase + x_smem(me, s);
#pragma unroll
                    for (int q = 0; q < kBlockK / 16; ++q) {
                        const uint32_t a_tmem = tmem + me * kAColsPerSlot + q * 8;
                        const uint64_t b_desc =
                            smem_desc_sw128_kmajor(xs + (q >> 2) * L::kXBoxBytes + (q & 3) * 32);
                        mma_f16_ts(d_tmem, a_tmem, b_desc, idesc, !(mine_first && q == 0));
                    }
                    mine_first = false;
                    any = true;
                    tc_commit(aempty(me));
                    tc_commit(xempty(me, s));
                    ++j;
                }
                if (failed) break;
                // the accumulator is ready when this lane's MMAs of the tile are done
                if (any)
                    tc_commit(dready(me, d));
                else
                    mbar_arrive(dready(me, d));
            }
            // every MMA issued above completes before TMEM is released
            tc_commit(drain(me));
            if (!mbar_wait_drain(drain(me), 0)) atomicCAS(&g_skinny_error, 0, kErrWaitDrain * 1000);
        }
    } else if (warp < kFirstDequantWarp) {
        // ------------------------------------------- epilogue (warps 5-8) --
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // channel within the tile == TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const int etid = threadIdx.x - 32 * kFirstEpilogueWarp;  // 0..127
        uint32_t* counters = reinterpret_cast<uint32_t*>(workspace);
        float* slots = reinterpret_cast<float*>(workspace + kWsCountersBytes);
        pdl_wait();  // the workspace and y may still be in use by the previous grid
        int seg = 0;
        UnitCursor cu = cursor0();
        for (int it = 0; it < iters; ++seg) {
            // segment: the units of one tile, contiguous in processing order
            const int seg_len = cu.seg_left(iters);
            const int64_t tile = cu.tile;
            const bool whole = cu.kb == 0 && seg_len == cu.nkb;
            const int it0 = it;
            it += seg_len;
            for (int jj = 0; jj < seg_len; ++jj) cu.next();
            const int d = seg & 1;
            bool ok = true;
            for (int g = 0; g < kLanes; ++g)
                ok = mbar_wait_warp(dready(g, d), static_cast<uint32_t>((seg >> 1) & 1), abort_flag) && ok;
            if (!ok) {
                if (lane == 0) *ep_abort = 1;
                record_error(kErrWaitMma, abort_flag);
            }
            // the four epilogue warps leave together (ep_abort is written only
            // by them, before this barrier), so their named barriers stay matched
            epilogue_bar();
            if (*ep_abort) break;
            tc_fence_after();
            const int64_t col = tile * kTileN + r;
            const float sc = col < n ? scales[col] : 0.0f;
            const float b = (bias && col < n) ? bias[col] : 0.0f;
            const int64_t slot = 2 * c + (tile == t_first ? 0 : 1);
            float* mine = slots + slot * ws_slot_floats() + r * kMaxNT;
            // 16 tokens at a time: sum the lanes' accumulators in a fixed
            // order, then store y (whole tile) or publish the partial
#pragma unroll 1
            for (int h = 0; h < NT / 16; ++h) {
                float acc[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
#pragma unroll
                for (int g = 0; g < kLanes; ++g) {
                    if (!lane_has(g, it0, seg_len)) continue;
                    uint32_t v[16];
                    tmem_ld_x16(lane_addr + kDCol0 + (g * 2 + d) * NT + h * 16, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 16; ++q) acc[q] += __uint_as_float(v[q]);
                }
                if (whole) {
                    if (col < n) {
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            if (h * 16 + q < m_rows)
                                y[static_cast<int64_t>(h * 16 + q) * n + col] = round_out<kBf16>(fmaf(acc[q], sc, b));
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(mine + h * 16);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                for (int g = 0; g < kLanes; ++g) mbar_arrive(dfree(g, d));

            if (!whole) {
                // partial tile: count, and let the last contributor finish it
                epilogue_bar();
                const int64_t c_lo = part.owner(tile * nkb);
                const int64_t c_hi = part.owner((tile + 1) * nkb - 1);
                if (etid == 0) {
                    const uint32_t old = arrive_acq_rel(&counters[c_lo]);
                    const bool is_last = old == static_cast<uint32_t>(c_hi - c_lo);
                    if (is_last) atomicExch(&counters[c_lo], 0u);
                    *last_flag = is_last ? 1 : 0;
                }
                epilogue_bar();
                if (*last_flag) {
                    // every contributor after c_lo starts inside this tile (its
                    // first slot); c_lo used its first slot only if it starts
                    // exactly at the tile's first unit
                    const bool lo_first = part.begin(c_lo) == tile * nkb;
#pragma unroll 1
                    for (int h = 0; h < NT / 16; ++h) {
                        float acc[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
                        // contributors in CTA order (the result does not depend on
                        // which CTA arrives last), kFixupBatch at a time
                        for (int64_t cb = c_lo; cb <= c_hi; cb += kFixupBatch) {
                            float4 v[kFixupBatch][4];
#pragma unroll
                            for (int e = 0; e < kFixupBatch; ++e) {
                                const int64_t cc = cb + e;
                                if (cc <= c_hi) {
                                    const int64_t cs = 2 * cc + ((cc > c_lo || lo_first) ? 0 : 1);
                                    const float4* src = reinterpret_cast<const float4*>(
                                        slots + cs * ws_slot_floats() + r * kMaxNT + h * 16);
#pragma unroll
                                    for (int q = 0; q < 4; ++q) v[e][q] = __ldcg(src + q);
                                } else {
#pragma unroll
                                    for (int q = 0; q < 4; ++q) v[e][q] = make_float4(0.f, 0.f, 0.f, 0.f);
                                }
                            }
#pragma unroll
                            for (int e = 0; e < kFixupBatch; ++e) {
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    acc[4 * q] += v[e][q].x;
                                    acc[4 * q + 1] += v[e][q].y;
                                    acc[4 * q + 2] += v[e][q].z;
                                    acc[4 * q + 3] += v[e][q].w;
                                }
                            }
                        }
                        if (col < n) {
#pragma unroll
                            for (int q = 0; q < 16; ++q)
                                if (h * 16 + q < m_rows)
                                    y[static_cast<int64_t>(h * 16 + q) * n + col] =
                                        round_out<kBf16>(fmaf(acc[q], sc, b));
                        }
                    }
                }
                epilogue_bar();
            }
        }
    } else {
        // ------------------------------- dequantising warpgroups (9-20) --
        const int group = (warp - kFirstDequantWarp) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t a_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + group * kAColsPerSlot;
        int j = 0;  // this lane's units so far
        for (int it = group; it < iters; it += kLanes, ++j) {
            const int s = j % kCS;
            if (!mbar_wait_warp(cfull(group, s), static_cast<uint32_t>((j / kCS) & 1), abort_flag)) {
                record_error(kErrWaitTma, abort_flag, cfull(group, s), bar0);
                break;
            }
            const uint8_t* row = smem + code_smem(group, s) + r * 128;
            uint4 cw[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) cw[q] = *reinterpret_cast<const uint4*>(row + ((q ^ (r & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(cempty(group, s));
            // the first half is converted while the lane's previous MMAs may
            // still be reading the A slot
            uint32_t v0[4][8];
#pragma unroll
            for (int q = 0; q < 4; ++q) dequant16<kBf16>(cw[q], v0[q]);
            if (!mbar_wait_warp(aempty(group), static_cast<uint32_t>((j & 1) ^ 1), abort_flag)) {
                record_error(kErrWaitMma, abort_flag, aempty(group), bar0);
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_st_x8(a_addr + q * 8, v0[q]);
#pragma unroll
            for (int q = 4; q < 8; ++q) {
                uint32_t v[8];
                dequant16<kBf16>(cw[q], v);
                tmem_st_x8(a_addr + q * 8, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(group));
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

// CTAs of the persistent grid.  Whole tiles when the tile count nearly
// fills the GPU (no partial tiles, no fix-up); when it is well below the SM
// count, each tile split evenly over s CTAs; otherwise stream-K over the SMs.
// A split CTA gets at least kMinUnitsPerCta units, and P <= kMaxCtas.
int64_t skinny_grid(int64_t n, int64_t k, int sms) {
    const int64_t tiles = (n + kTileN - 1) / kTileN;
    const int64_t nkb = (k + kBlockK - 1) / kBlockK;
    const int64_t units = tiles * nkb;
    const int64_t cap = sms < kMaxCtas ? sms : kMaxCtas;
    int64_t p;
    if (tiles <= cap && 10 * tiles >= 7 * cap) {
        p = tiles;
    } else if (tiles < cap) {
        int64_t split = cap / tiles;
        const int64_t most = nkb / kMinUnitsPerCta;
        if (split > most) split = most;
        if (split < 1) split = 1;
        p = tiles * split;
    } else {
        p = units / kMinUnitsPerCta;
        if (p > cap) p = cap;
    }
    if (p < 1) p = 1;
    return p;
}

template <int NT, bool kBf16>
static cudaError_t launch_nt(const LinearArgs& a, void* workspace, int ctas, cudaStream_t st) {
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

    // every CTA gets at least one unit: the fix-up counts CTAs, so an empty
    // range inside a split tile would leave that tile unfinished
    const int64_t units = ((a.n + kTileN - 1) / kTileN) * ((a.k + kBlockK - 1) / kBlockK);
    int64_t grid = ctas > 0 ? ctas : skinny_grid(a.n, a.k, sms);
    if (grid > units) grid = units;
    // programmatic dependent launch: this grid's prologue (barrier set-up,
    // TMEM allocation) overlaps the tail of the previous kernel in the
    // stream; every role waits for that kernel before touching global memory
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    uint16_t* yp = static_cast<uint16_t*>(a.y);
    for (int64_t m0 = 0; m0 < a.m; m0 += kMaxNT) {
        const int rows = static_cast<int>(a.m - m0 < kMaxNT ? a.m - m0 : kMaxNT);
        e = cudaLaunchKernelEx(&cfg, kern, map_codes, map_x, a.scales, a.bias, yp + m0 * a.n,
                               static_cast<uint8_t*>(workspace), rows, static_cast<int>(m0), a.n, a.k);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t skinny_workspace_size(int sms) { return skinny_workspace_bytes(sms < kMaxCtas ? sms : kMaxCtas); }

cudaError_t launch_skinny(const LinearArgs& a, void* workspace, int ctas, cudaStream_t st) {
    const bool bf16 = a.act == 1;
    if (a.m <= 16)
        return bf16 ? launch_nt<16, true>(a, workspace, ctas, st) : launch_nt<16, false>(a, workspace, ctas, st);
    return bf16 ? launch_nt<32, true>(a, workspace, ctas, st) : launch_nt<32, false>(a, workspace, ctas, st);
}

// Library-owned scratch for fp8w_linear_noalloc: the workspace of a grid of
// up to kStaticScratchCtas CTAs, in device memory that exists as soon as this
// module is loaded on a device, so that entry point allocates nothing.
constexpr int kStaticScratchCtas = 160;
constexpr size_t kStaticScratchBytes = skinny_workspace_bytes(kStaticScratchCtas);
static_assert(kStaticScratchBytes == FP8W_STATIC_SCRATCH_BYTES, "fp8w.h states the static scratch size");
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

size_t static_scratch_bytes() { return kStaticScratchBytes; }

// First call on a device (with that device current): look up the array's
// address and enqueue a clear of its arrival counters on `st`, ahead of the
// kernel that will use them.  Later calls return the cached address.
cudaError_t static_scratch(void** ptr, cudaStream_t st) {
    static std::mutex mu;
    static void* ptrs[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        e = cudaMemsetAsync(p, 0, kWsCountersBytes, st);
        if (e != cudaSuccess) return e;
        ptrs[dev] = p;
    }
    *ptr = ptrs[dev];
    return cudaSuccess;
}

int read_skinny_device_error() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_skinny_error, sizeof v) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_skinny_error, &zero, sizeof zero);
    return v;
}

}  // namespace fp8w
