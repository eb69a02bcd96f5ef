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
//    (channel tile of 128, k-block of 128).  Three launch shapes:
//    - whole tiles, one CTA each, when the tile count nearly fills the GPU;
//    - split: fewer tiles than SMs, each tile's k-blocks divided evenly over
//      a thread-block cluster of 2, 4 or 8 CTAs, whose fp32 partials are
//      summed through distributed shared memory at the end (each CTA adds
//      up, in rank order, a slice of the tile's channels from every rank);
//    - stream-K: more tiles than SMs; CTA c takes the contiguous units
//      [c*U/P, (c+1)*U/P), and a tile that straddles CTAs is finished by the
//      last contributor: partial fp32 tiles go to a caller-provided workspace
//      and are summed in CTA order (deterministic); no CTA waits on another.
//    A CTA takes its units in order, so the piece at the start of its range
//    (the end of a tile another CTA began) is done first and published
//    early; the CTA holding the start of that tile finishes it last and, as
//    every other contributor has arrived by then, sums their partials
//    straight from its registers without publishing its own.
//  * Warp 0 streams each unit's 128 x 128 code tile with TMA (128-byte
//    swizzle; rows past N and k past K read as zeros) into the code ring of
//    one of three dequantising warpgroups (units are dealt round-robin);
//    warp 1 streams the unit's M x 128 activation tile (an L2 hit) into a
//    ring read by the MMA warps.  The activation ring is deeper than the code
//    rings, so each activation tile enters the SM's TMA queue no later than
//    its unit's code tile and never waits behind the whole code ring.  The
//    two producer warps set up their own barriers and start streaming
//    without waiting for the other warps to come up.  Every ring has one
//    producer and one in-order consumer.
//  * In each warpgroup, thread r reads the 128 codes of channel r
//    (conflict-free through the swizzle), converts them exactly to bf16 /
//    fp16 in registers and stores them with tcgen05.st into one of the
//    group's two TMEM A slots, where they are the A operand of the MMA (A
//    from tensor memory: the dequantised weight never touches shared
//    memory).  Two slots let a group convert the next unit while the MMAs
//    still read the previous one.
//  * Unit u uses A slot u % 6 (warpgroup u % 3, its slot (u / 3) % 2) and
//    activation slot u % kXSlots.
//  * Warps 2 and 3, the MMA warps, take alternate units in order and issue
//    each unit's eight tcgen05.mma.kind::f16 (M = 128, N = 16 or 32 tokens,
//    K = 16) into their own TMEM accumulator of the tile (double-buffered
//    across tiles), then free the operand slots with tcgen05.commit.  Each
//    warp runs its loop whole and elect.sync picks the issuing lane (issued
//    that way an MMA costs the warp ~20-30 cycles); a warp tests its next
//    unit's barriers, without blocking, before this unit's MMAs, because a
//    barrier wait costs about as much as a unit's eight MMAs.  One issuing
//    warp per accumulator keeps that accumulator's MMAs in order; two keep up
//    with the weight stream.
//  * One epilogue warpgroup reads a finished tile's two accumulators with
//    tcgen05.ld (thread r holds channel r for every token), adds them in a
//    fixed order while the next tile accumulates, and stores
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
constexpr int kLanes = 3;                   // dequantising warpgroups
constexpr int kASlots = 2;                  // TMEM A slots per warpgroup
// warps: 0 code TMA, 1 activation TMA, 2-3 MMA (warp 2 also owns TMEM),
// 4..7 epilogue, 8..19 the dequantising warpgroups (4 warps each)
constexpr int kXWarp = 1;
constexpr int kMmaWarp = 2;
constexpr int kMmaWarps = 2;
constexpr int kFirstEpilogueWarp = kMmaWarp + kMmaWarps;
constexpr int kFirstDequantWarp = kFirstEpilogueWarp + 4;
constexpr int kThreads = 32 * (kFirstDequantWarp + 4 * kLanes);  // 640
// named barriers: 0 __syncthreads, 1 epilogue, 2 TMEM ready, 3 start-up
constexpr uint32_t kBarEpilogue = 1, kBarTmem = 2, kBarStart = 3;
constexpr int kTmemCols = 512;              // one CTA per SM
constexpr int kAColsPerSlot = kBlockK / 2;  // two 16-bit values per column
constexpr int kDCol0 = kLanes * kASlots * kAColsPerSlot;  // 384: accumulators after the A slots
constexpr uint32_t kCodeStageBytes = kTileN * kBlockK;  // 16 KB
constexpr int kMaxNT = 64;

template <int NT>
struct SkinnySmem {
    // per warpgroup: freed as soon as read (9 tiles in flight per SM: deeper
    // rings on every SM make the HBM stream slower, not faster)
    static constexpr int kCodeSlots = NT <= 32 ? 3 : 2;
    static constexpr int kXSlots = NT == 16 ? 12 : 8;  // activation ring (freed when the unit's MMAs are done)
    // accumulator buffers per MMA warp: two (the epilogue drains one tile
    // while the next accumulates) where TMEM has room, one for 64 tokens
    static constexpr int kDBuf = NT <= 32 ? 2 : 1;
    static_assert(kDCol0 + kMmaWarps * kDBuf * NT <= kTmemCols, "TMEM columns");
    static_assert(kXSlots % kMmaWarps == 0 && (kLanes * kASlots) % kMmaWarps == 0, "slots alternate between MMA warps");
    static constexpr uint32_t kXBoxBytes = NT * 128;          // 64 k x NT rows x 2 B
    static constexpr uint32_t kXStageBytes = 2 * kXBoxBytes;  // 128 k
    static constexpr uint32_t kCodesOff = 0;
    static constexpr uint32_t kXOff = kCodesOff + kLanes * kCodeSlots * kCodeStageBytes;
    static constexpr uint32_t kBarOff = kXOff + kXSlots * kXStageBytes;
    // per warpgroup: cfull, cempty [kCodeSlots]
    static constexpr uint32_t kBarsPerLane = 2 * kCodeSlots;
    // then: aready [6]; udone [kDoneSlots]; xfull [kXSlots]; dfree [2];
    // dready [MMA warp][2]; drain [MMA warp].  udone(u % kDoneSlots) completes
    // a phase when unit u's MMAs are done: it frees the unit's A slot (for
    // unit u + 6) and its activation slot (for unit u + kXSlots) with one
    // commit; kDoneSlots is a multiple of both ring sizes, so each waiter
    // finds the phase of the unit it waits for.
    static constexpr int kASlotsAll = kLanes * kASlots;
    static constexpr int kDoneSlots = NT == 16 ? 12 : 24;
    static_assert(kDoneSlots % kASlotsAll == 0 && kDoneSlots % kXSlots == 0, "unit-done ring");
    static constexpr uint32_t kLaneBars = kLanes * kBarsPerLane;
    static constexpr uint32_t kNumBars = kLaneBars + kASlotsAll + kDoneSlots + kXSlots + 2 + 3 * kMmaWarps;
    // tmem base, abort flag, last-contributor flag, epilogue abort flag
    static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
    static constexpr uint32_t kBytes = kMiscOff + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
    static_assert(kAlloc <= 227 * 1024, "shared memory");
    // arrivals per phase: cempty, aready and dfree one per warp of a
    // warpgroup, the others one
    static __device__ __forceinline__ uint32_t arrivals(uint32_t i) {
        if (i < kLaneBars) return (i % kBarsPerLane) >= static_cast<uint32_t>(kCodeSlots) ? 4u : 1u;
        const uint32_t gi = i - kLaneBars;
        if (gi < static_cast<uint32_t>(kASlotsAll)) return 4u;  // aready
        const uint32_t di = static_cast<uint32_t>(kASlotsAll + kDoneSlots + kXSlots);
        return (gi == di || gi == di + 1) ? 4u : 1u;            // dfree
    }
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
// Tokens whose cluster partials one thread loads before adding them up.
constexpr int kRedBatch = 4;

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

// Walks a CTA's units in order without divisions: (tile, kb) of the current
// unit.
struct UnitCursor {
    int it;
    int tile, kb, nkb;
    __device__ __forceinline__ void next() {
        ++it;
        if (++kb == nkb) {
            kb = 0;
            ++tile;
        }
    }
    // units left in the current tile within the CTA's range
    __device__ __forceinline__ int seg_left(int iters) const { return min(nkb - kb, iters - it); }
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

// MX-style scales (page "11. Inference with NVFP4/MXFP8", section
// "MXFP8-Style FP8"): one E8M0 byte b per 32 codes, worth 2^e, e = b - 127.
// It is folded into the dequantised weight, whose bf16 value * 2^e is exact
// wherever it is a bf16 number (the codes have 4 significant bits).  The
// multiplier of a group is 2^(120 + e), a bf16 number for b <= 134; a warp
// holding a larger byte multiplies by 2^120 and then by 2^e (b = 0: the
// subnormal 2^-127; 0xFF: NaN), which rounds the same product once.
__device__ __forceinline__ void dequant16_mx(const uint4 c, uint32_t (&out)[8], uint32_t mul) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) e4m3x4_to_bf16x2_mul(w[q], out[2 * q], out[2 * q + 1], mul);
}

// The recorded code is role * 1000 + 1 + the barrier's index in shared
// memory (0 when no barrier applies), so a report names the wait that gave up.
__device__ __forceinline__ void record_error(int code, volatile int* abort_flag, uint32_t bar = 0, uint32_t bar0 = 0) {
    *abort_flag = 1;
    atomicCAS(&g_skinny_error, 0, code * 1000 + (bar ? static_cast<int>((bar - bar0) / 8) + 1 : 0));
}

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync %0, 128;" ::"n"(kBarEpilogue) : "memory"); }

// Arrival count of a split tile: release orders this CTA's partial stores
// (made visible to this thread by the preceding CTA barrier) before the
// increment; acquire orders the last contributor's reads after it.
__device__ __forceinline__ uint32_t arrive_acq_rel(uint32_t* counter) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// kMx: the weight carries E8M0 scale bytes e8[n, k / 32] (bf16 activations,
// k % 128 == 0) instead of per-row scales; they enter the dequantised
// weight, and the epilogue adds only the bias.
template <int NT, bool kBf16, bool kMx = false>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x,
                  const float* __restrict__ scales, const uint8_t* __restrict__ e8, const float* __restrict__ bias,
                  uint16_t* __restrict__ y, uint8_t* __restrict__ workspace, int m_rows, int m_row0, int64_t n,
                  int64_t k, int split, int early) {
    static_assert(!kMx || kBf16, "MX-style scales fold into bf16 weights only");
    using L = SkinnySmem<NT>;
    constexpr int kCS = L::kCodeSlots, kXS = L::kXSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto lbar = [&](int g, int i) { return bar0 + 8u * (g * L::kBarsPerLane + i); };
    auto cfull = [&](int g, int s) { return lbar(g, s); };
    auto cempty = [&](int g, int s) { return lbar(g, kCS + s); };
    constexpr int kAS = L::kASlotsAll;
    auto gbar = [&](int i) { return bar0 + 8u * (L::kLaneBars + i); };
    constexpr int kDone = L::kDoneSlots;
    auto aready = [&](int r) { return gbar(r); };
    auto udone = [&](int i) { return gbar(kAS + i); };
    auto xfull = [&](int s) { return gbar(kAS + kDone + s); };
    auto dfree = [&](int d) { return gbar(kAS + kDone + kXS + d); };
    auto dready = [&](int w, int d) { return gbar(kAS + kDone + kXS + 2 + 2 * w + d); };
    auto drain = [&](int w) { return gbar(kAS + kDone + kXS + 2 + 2 * kMmaWarps + w); };
    // unit v's MMAs are done (v < 0: nothing to wait for)
    auto done_bar = [&](int v) { return udone(v % kDone); };
    auto done_parity = [&](int v) { return static_cast<uint32_t>((v / kDone) & 1); };
    auto code_smem = [&](int g, int s) { return L::kCodesOff + (g * kCS + s) * kCodeStageBytes; };
    auto x_smem = [&](int s) { return L::kXOff + s * L::kXStageBytes; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);
    volatile int* ep_abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 12);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles = (n + kTileN - 1) / kTileN;
    const int64_t nkb = (k + kBlockK - 1) / kBlockK;
    const Partition part{tiles * nkb, static_cast<int64_t>(gridDim.x), nkb};
    const int64_t c = blockIdx.x;
    // split launches: cluster c / split takes tile c / split, its rank c % split
    // an even share of the k-blocks; otherwise the contiguous range of units
    const int64_t u0 = split > 1 ? (c / split) * nkb + (c % split) * nkb / split : part.begin(c);
    const int64_t u1 = split > 1 ? (c / split) * nkb + (c % split + 1) * nkb / split : part.begin(c + 1);
    const int iters = static_cast<int>(u1 - u0);
    const int64_t t_first = u0 / nkb;
    const int kb_first = static_cast<int>(u0 - t_first * nkb);
    auto cursor0 = [=]() {
        UnitCursor cu;
        cu.it = 0;
        cu.nkb = static_cast<int>(nkb);
        cu.tile = static_cast<int>(t_first);
        cu.kb = kb_first;
        return cu;
    };

    // Start-up: warp 1 sets up the activation ring's barriers, warp 0 all the
    // others; each then arrives at the start-up barrier without waiting and
    // begins streaming, while the other warps wait there for both.
    if (warp <= kXWarp) {
        // warp 1 sets up udone and xfull, [xb0, xb1): it is the first to wait on udone
        const uint32_t xb0 = static_cast<uint32_t>(L::kLaneBars + kAS);
        const uint32_t xb1 = xb0 + static_cast<uint32_t>(kDone + kXS);
        if (warp == 0) {
            for (uint32_t i = lane; i < L::kNumBars; i += 32)
                if (i < xb0 || i >= xb1) mbar_init(bar0 + 8 * i, L::arrivals(i));
        } else {
            for (uint32_t i = xb0 + lane; i < xb1; i += 32) mbar_init(bar0 + 8 * i, L::arrivals(i));
            __syncwarp();
        }
        if (lane == 0) {
            *abort_flag = 0;  // written by both producer warps before either can raise it
            if (warp == 0) *ep_abort = 0;
            tma_prefetch_desc(warp == 0 ? &map_codes : &map_x);
        }
        fence_mbar_init();
        asm volatile("bar.arrive %0, %1;" ::"n"(kBarStart), "n"(kThreads) : "memory");
    } else {
        asm volatile("bar.sync %0, %1;" ::"n"(kBarStart), "n"(kThreads) : "memory");
    }
    // let the next kernel in the stream start launching; its CTAs wait for
    // this grid to complete before they read or write global memory
    pdl_launch_dependents();
    // TMEM is allocated by the MMA warp while the producers already stream;
    // the warps that use it meet the MMA warp at a named barrier first.
    uint32_t tmem = 0;
    if (warp >= kMmaWarp) {
        if (warp == kMmaWarp) {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        asm volatile("bar.sync %0, %1;" ::"n"(kBarTmem), "n"(kThreads - 32 * kMmaWarp) : "memory");
        tc_fence_after();
        tmem = *tmem_slot;
    }

    if (warp == 0) {
        // ----------------------------------------------- code-tile producer --
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_first();
            // the codes may come from the previous kernel, unless the caller
            // states that they were complete before it started
            if (!early) pdl_wait();
            UnitCursor cu = cursor0();
            int g = 0, j = 0;  // warpgroup of the unit, and its index within the group
            int s = 0;         // == j % kCS
            uint32_t ph = 0;   // == (j / kCS) & 1
            int issued = 0;
            for (int it = 0; it < iters; ++it, cu.next()) {
                if (!mbar_wait(cempty(g, s), ph ^ 1u, abort_flag)) {
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
                    if (++s == kCS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // let every copy still in flight land before the CTA exits:
                // the last fills of each group's slots
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
            pdl_wait();  // x may come from the previous kernel
            UnitCursor cu = cursor0();
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            for (int it = 0; it < iters; ++it, cu.next()) {
                // the slot's previous unit (it - kXS) must be done
                if (it >= kXS && !mbar_wait(done_bar(it - kXS), done_parity(it - kXS), abort_flag)) {
                    record_error(kErrWaitSlot, abort_flag, done_bar(it - kXS), bar0);
                    break;
                }
                const int32_t kk = cu.kb * kBlockK;
                const uint32_t xs = sbase + x_smem(s);
                mbar_arrive_expect_tx(xfull(s), L::kXStageBytes);
                tma_load_2d(xs, &map_x, kk, m_row0, xfull(s), pol_keep);
                tma_load_2d(xs + L::kXBoxBytes, &map_x, kk + 64, m_row0, xfull(s), pol_keep);
                ++issued;
                if (++s == kXS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag) {
                for (int jj = (issued > kXS ? issued - kXS : 0); jj < issued; ++jj)
                    if (!mbar_wait_drain(xfull(jj % kXS), static_cast<uint32_t>((jj / kXS) & 1)))
                        atomicCAS(&g_skinny_error, 0, kErrWaitDrain * 1000);
            }
        }
    } else if (warp < kFirstEpilogueWarp) {
        // ----------------------------------------------------- MMA warps --
        // Warp w issues the units it with it % 2 == w.  The whole warp runs
        // the loop (every condition is warp-uniform) and elect.sync picks the
        // lane that issues and commits.  Both warps walk every unit to keep
        // the tile segments in step.
        const int w = warp - kMmaWarp;
        constexpr uint32_t idesc = idesc_f16(kBf16, NT);
        UnitCursor cu = cursor0();
        int seg = 0, jj = 0;
        int seg_len = iters > 0 ? cu.seg_left(iters) : 0;
        int ra = w, rx = w;          // slots of this warp's next unit: A (unit % 6), activation (unit % kXS)
        uint32_t pa = 0, px = 0;     // their phase parities
        bool mine_in_seg = false;    // this warp has issued into the segment's accumulator
        bool failed = false;
        if (w < iters && (!mbar_wait_warp(aready(ra), pa, abort_flag) || !mbar_wait_warp(xfull(rx), px, abort_flag))) {
            if (lane == 0) record_error(kErrWaitDequant, abort_flag, aready(ra), bar0);
            failed = true;
        }
        for (int it = 0; it < iters && !failed; ++it) {
            const int d = seg % L::kDBuf;
            if (jj == 0 &&
                !mbar_wait_warp(dfree(d), static_cast<uint32_t>(((seg / L::kDBuf) & 1) ^ 1), abort_flag)) {
                // the epilogue has not drained this accumulator (two segments ago)
                if (lane == 0) record_error(kErrWaitMma, abort_flag, dfree(d), bar0);
                break;
            }
            if ((it & 1) == w) {
                // test this warp's next unit (it + 2) now; the answer is used
                // after this unit's MMAs, which hide the tests' latency
                const int ran = ra + kMmaWarps >= kAS ? ra + kMmaWarps - kAS : ra + kMmaWarps;
                const int rxn = rx + kMmaWarps >= kXS ? rx + kMmaWarps - kXS : rx + kMmaWarps;
                const uint32_t pan = ran < ra ? pa ^ 1u : pa;
                const uint32_t pxn = rxn < rx ? px ^ 1u : px;
                const bool more = it + kMmaWarps < iters;
                const bool next_a = !more || mbar_test_wait(aready(ran), pan);
                const bool next_x = !more || mbar_test_wait(xfull(rxn), pxn);
                tc_fence_after();
                const uint32_t xs = sbase + x_smem(rx);
                const uint32_t a_tmem = tmem + ra * kAColsPerSlot;  // slot ra = (group ra % 3, A slot ra / 3)
                const uint32_t d_tmem = tmem + kDCol0 + (w * L::kDBuf + d) * NT;
#pragma unroll
                for (int q = 0; q < kBlockK / 16; ++q) {
                    const uint64_t b_desc = smem_desc_sw128_kmajor(xs + (q >> 2) * L::kXBoxBytes + (q & 3) * 32);
                    mma_f16_ts_warp(d_tmem, a_tmem + q * 8, b_desc, idesc, mine_in_seg || q > 0);
                }
                tc_commit_warp(done_bar(it));  // frees the unit's A and activation slots
                mine_in_seg = true;
                ra = ran;
                rx = rxn;
                pa = pan;
                px = pxn;
                if (more && !__all_sync(0xffffffffu, next_a) && !mbar_wait_warp(aready(ra), pa, abort_flag)) {
                    if (lane == 0) record_error(kErrWaitDequant, abort_flag, aready(ra), bar0);
                    failed = true;
                }
                if (more && !failed && !__all_sync(0xffffffffu, next_x) &&
                    !mbar_wait_warp(xfull(rx), px, abort_flag)) {
                    if (lane == 0) record_error(kErrWaitTma, abort_flag, xfull(rx), bar0);
                    failed = true;
                }
            }
            cu.next();
            if (++jj == seg_len) {
                // this warp's accumulator is ready when its MMAs of the tile are
                // done (at once if it had no unit in the tile)
                if (mine_in_seg) {
                    tc_commit_warp(dready(w, d));
                } else if (lane == 0) {
                    mbar_arrive(dready(w, d));
                }
                __syncwarp();
                mine_in_seg = false;
                ++seg;
                jj = 0;
                if (it + 1 < iters) seg_len = cu.seg_left(iters);
            }
        }
        // every MMA issued above completes before TMEM is released
        tc_commit_warp(drain(w));
        if (!mbar_wait_drain(drain(w), 0) && lane == 0) atomicCAS(&g_skinny_error, 0, kErrWaitDrain * 1000);
        __syncwarp();
    } else if (warp < kFirstDequantWarp) {
        // ------------------------------------------- epilogue (warps 4-7) --
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
            const int d = seg % L::kDBuf;
            int64_t c_lo = 0, c_hi = 0;
            bool all_in = false;
            if (!whole && split == 1) {
                c_lo = part.owner(tile * nkb);
                c_hi = part.owner((tile + 1) * nkb - 1);
                // every other contributor already arrived: this CTA finishes
                // the tile from its registers (tested while the MMAs run, and
                // again once the accumulator is ready)
                if (etid == 0) all_in = ld_acquire_gpu(&counters[c_lo]) == static_cast<uint32_t>(c_hi - c_lo);
            }
            bool ok = true;
            for (int w = 0; w < kMmaWarps; ++w)
                ok = mbar_wait_warp(dready(w, d), static_cast<uint32_t>((seg / L::kDBuf) & 1), abort_flag) && ok;
            if (!ok) {
                if (lane == 0) *ep_abort = 1;
                record_error(kErrWaitMma, abort_flag);
            }
            if (!whole && split == 1 && etid == 0) {
                if (!all_in) all_in = ld_acquire_gpu(&counters[c_lo]) == static_cast<uint32_t>(c_hi - c_lo);
                *last_flag = all_in ? 1 : 0;
            }
            // the four epilogue warps leave together (ep_abort is written only
            // by them, before this barrier), so their named barriers stay matched
            epilogue_bar();
            if (*ep_abort) break;
            const bool early = !whole && split == 1 && *last_flag;
            tc_fence_after();
            const int64_t col = tile * kTileN + r;
            const float sc = kMx ? 1.0f : col < n ? scales[col] : 0.0f;
            const float b = (bias && col < n) ? bias[col] : 0.0f;
            const int64_t slot = 2 * c + (tile == t_first ? 0 : 1);
            float* mine = slots + slot * ws_slot_floats() + r * kMaxNT;
            const bool lo_first = !whole && part.begin(c_lo) == tile * nkb;
            // every contributor after c_lo starts inside this tile (its first
            // slot); c_lo used its first slot only if it starts exactly at the
            // tile's first unit
            auto slot_of = [&](int64_t cc) -> const float4* {
                const int64_t cs = 2 * cc + ((cc > c_lo || lo_first) ? 0 : 1);
                return reinterpret_cast<const float4*>(slots + cs * ws_slot_floats() + r * kMaxNT);
            };
            // 16 tokens at a time, only as many as there are rows
#pragma unroll 1
            for (int h = 0; h < NT / 16 && h * 16 < m_rows; ++h) {
                // the MMA warps' accumulators, warp 0's first; a warp with no
                // unit in the segment (a one-unit segment) wrote nothing
                float acc[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
#pragma unroll
                for (int w = 0; w < kMmaWarps; ++w) {
                    if (seg_len < kMmaWarps && ((it0 + kMmaWarps - w) % kMmaWarps) >= seg_len) continue;
                    uint32_t v[16];
                    tmem_ld_x16(lane_addr + kDCol0 + (w * L::kDBuf + d) * NT + h * 16, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 16; ++q) acc[q] += __uint_as_float(v[q]);
                }
                if (split > 1) {
                    // this rank's partial tile, token-major, into the free code ring
                    float* pt = reinterpret_cast<float*>(smem + L::kCodesOff);
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (h * 16 + q < m_rows) pt[(h * 16 + q) * kTileN + r] = acc[q];
                } else if (whole || early) {
                    if (early) {
                        // contributors in CTA order, this CTA's own partial from
                        // registers: the same sum the publishing path forms
                        float tot[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) tot[q] = 0.0f;
                        for (int64_t cc = c_lo; cc <= c_hi; ++cc) {
                            if (cc == c) {
#pragma unroll
                                for (int q = 0; q < 16; ++q) tot[q] += acc[q];
                                continue;
                            }
                            float4 v[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                v[q] = h * 16 + 4 * q < m_rows ? __ldcg(slot_of(cc) + h * 4 + q)
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                tot[4 * q] += v[q].x;
                                tot[4 * q + 1] += v[q].y;
                                tot[4 * q + 2] += v[q].z;
                                tot[4 * q + 3] += v[q].w;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 16; ++q) acc[q] = tot[q];
                    }
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
                        if (h * 16 + 4 * q < m_rows)
                            dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dfree(d));

            if (!whole && split == 1) {
                if (early) {
                    // every other contributor has arrived, so nobody else
                    // touches the counter during this launch
                    if (etid == 0) counters[c_lo] = 0u;
                } else {
                    // publish, count, and let the last contributor finish
                    epilogue_bar();
                    if (etid == 0) {
                        const uint32_t old = arrive_acq_rel(&counters[c_lo]);
                        const bool is_last = old == static_cast<uint32_t>(c_hi - c_lo);
                        if (is_last) atomicExch(&counters[c_lo], 0u);
                        *last_flag = is_last ? 1 : 0;
                    }
                    epilogue_bar();
                    if (*last_flag) {
#pragma unroll 1
                        for (int h = 0; h < NT / 16 && h * 16 < m_rows; ++h) {
                            float acc[16];
#pragma unroll
                            for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
                            // contributors in CTA order, kFixupBatch at a time
                            for (int64_t cb = c_lo; cb <= c_hi; cb += kFixupBatch) {
                                float4 v[kFixupBatch][4];
#pragma unroll
                                for (int e = 0; e < kFixupBatch; ++e) {
                                    const int64_t cc = cb + e;
#pragma unroll
                                    for (int q = 0; q < 4; ++q)
                                        v[e][q] = (cc <= c_hi && h * 16 + 4 * q < m_rows)
                                                      ? __ldcg(slot_of(cc) + h * 4 + q)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                                }
#pragma unroll
                                for (int e = 0; e < kFixupBatch; ++e) {
                                    if (cb + e > c_hi) break;
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
                }
                // last_flag is rewritten at the next split segment
                epilogue_bar();
            }
        }
    } else {
        // ------------------------------- dequantising warpgroups (8-19) --
        const int group = (warp - kFirstDequantWarp) >> 2;
        // MX: this thread's row's four scale bytes of a unit (one word), loaded
        // a unit ahead; (mx_tile, mx_kb) is the unit after the current one
        int64_t mx_tile = 0;
        int mx_kb = 0;
        uint32_t mx_next = 0x7F7F7F7Fu;
        auto mx_load = [&](int64_t tile, int kb) -> uint32_t {
            const int64_t row = tile * kTileN + (warp & 3) * 32 + lane;
            // rows past n hold zero codes (the copy's fill): any scale does
            return row < n ? __ldg(reinterpret_cast<const uint32_t*>(e8 + row * (k >> 5) + kb * 4)) : 0x7F7F7F7Fu;
        };
        if constexpr (kMx) {
            if (!early) pdl_wait();  // the scales may come from the previous kernel
            const int64_t u = u0 + group;
            mx_tile = u / nkb;
            mx_kb = static_cast<int>(u - mx_tile * nkb);
            if (group < iters) mx_next = mx_load(mx_tile, mx_kb);
        }
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t a_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        int s = 0;         // == j % kCS
        uint32_t ph = 0;   // == (j / kCS) & 1
        for (int j = 0, it = group; it < iters; it += kLanes, ++j) {
            if (!mbar_wait_warp(cfull(group, s), ph, abort_flag)) {
                record_error(kErrWaitTma, abort_flag, cfull(group, s), bar0);
                break;
            }
            uint32_t mx_word = 0u;
            if constexpr (kMx) {
                mx_word = mx_next;
                mx_kb += kLanes;
                while (mx_kb >= nkb) {
                    mx_kb -= static_cast<int>(nkb);
                    ++mx_tile;
                }
                if (it + kLanes < iters) mx_next = mx_load(mx_tile, mx_kb);
            }
            const uint32_t row = sbase + code_smem(group, s) + r * 128;
            uint4 cw[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) cw[q] = lds128(row + ((q ^ (r & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(cempty(group, s));
            if (++s == kCS) {
                s = 0;
                ph ^= 1u;
            }
            // the first half is converted while the MMAs may still read the slot
            uint32_t v0[4][8];
            uint32_t mul[4];
            bool twice = false;
            if constexpr (kMx) {
                // a byte above 134 anywhere in the warp (0xFF included):
                // two multiplies; otherwise the four 2^(120 + e) at once, the
                // bytes b + 120 (no carry for b <= 134) as bf16 exponent
                // fields in both halves
                twice = __any_sync(0xffffffffu, __vcmpgtu4(mx_word, 0x86868686u) != 0u);
                const uint32_t wb = __vadd4(mx_word, 0x78787878u);
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    mul[g] = twice ? kBf16x2Pow2_120 : __byte_perm(wb, 0u, 0x4040u + 0x0101u * g) << 7;
            }
            // the second multiply of a group's two chunks, when needed
            auto mx_fix = [&](uint32_t (&v)[8], int q) {
                if constexpr (kMx) {
                    if (twice) {
                        const uint32_t m2 = mx_second_mul((mx_word >> (8 * (q >> 1))) & 0xFFu);
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = bf16x2_mul(v[e], m2);
                    }
                }
            };
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if constexpr (kMx) {
                    dequant16_mx(cw[q], v0[q], mul[q >> 1]);
                    mx_fix(v0[q], q);
                } else {
                    dequant16<kBf16>(cw[q], v0[q]);
                }
            }
            // A slot of unit it = group + 3j: it % 6 = group + 3 (j % 2)
            const int r = group + kLanes * (j & 1);
            // the A slot's previous unit (it - 6) must be done
            if (it >= kAS && !mbar_wait_warp(done_bar(it - kAS), done_parity(it - kAS), abort_flag)) {
                record_error(kErrWaitMma, abort_flag, done_bar(it - kAS), bar0);
                break;
            }
            tc_fence_after();
            const uint32_t a_addr = a_lane + r * kAColsPerSlot;
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_st_x8(a_addr + q * 8, v0[q]);
#pragma unroll
            for (int q = 4; q < 8; ++q) {
                uint32_t v[8];
                if constexpr (kMx) {
                    dequant16_mx(cw[q], v, mul[q >> 1]);
                    mx_fix(v, q);
                } else {
                    dequant16<kBf16>(cw[q], v);
                }
                tmem_st_x8(a_addr + q * 8, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(aready(r));
        }
    }

    __syncthreads();
    if (split > 1) {
        // this rank adds up channels [ch0, ch0 + nch) of the tile over all
        // ranks, in rank order, and writes y; split is a power of two, so a
        // thread keeps one channel, whose scale and bias it fetches first
        const bool red_thread = warp >= kFirstEpilogueWarp && warp < kFirstDequantWarp;
        const int etid = threadIdx.x - 32 * kFirstEpilogueWarp;
        const int nch = kTileN / split;
        const int ch = static_cast<int>(c % split) * nch + (red_thread ? etid % nch : 0);
        const int64_t col = (c / split) * kTileN + ch;
        float sc = 0.0f, b = 0.0f;
        if (red_thread && col < n) {
            sc = kMx ? 1.0f : scales[col];
            b = bias ? bias[col] : 0.0f;
        }
        // every rank's partial tile is in its shared memory
        cluster_sync_all();
        if (red_thread && !*ep_abort && iters > 0) {
            const uint32_t pt = sbase + L::kCodesOff;
            if (col < n) {
                // kRedBatch tokens' loads from all ranks are issued before any
                // sum, so their remote round trips overlap
                const int tstep = 128 / nch;
                for (int tok0 = etid / nch; tok0 < m_rows; tok0 += kRedBatch * tstep) {
                    float v[kRedBatch][8];
#pragma unroll
                    for (int e = 0; e < kRedBatch; ++e) {
                        const int tok = tok0 + e * tstep;
                        const uint32_t off = pt + static_cast<uint32_t>((tok * kTileN + ch) * 4);
#pragma unroll
                        for (int rr = 0; rr < 8; ++rr)
                            if (rr < split && tok < m_rows) v[e][rr] = ld_shared_cluster_f32(mapa_shared(off, rr));
                    }
#pragma unroll
                    for (int e = 0; e < kRedBatch; ++e) {
                        const int tok = tok0 + e * tstep;
                        if (tok >= m_rows) break;
                        float t = 0.0f;
#pragma unroll
                        for (int rr = 0; rr < 8; ++rr)
                            if (rr < split) t += v[e][rr];
                        y[static_cast<int64_t>(tok) * n + col] = round_out<kBf16>(fmaf(t, sc, b));
                    }
                }
            }
        }
        // no rank leaves while its partial may still be read
        cluster_sync_all();
    }
    if (warp == kMmaWarp) {
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

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
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
// Launch shape: the grid size, and the cluster size of a split launch (1 =
// whole tiles or stream-K).
struct SkinnyShape {
    int64_t grid;
    int split;
};

constexpr int kMaxSplit = 8;  // portable cluster size

SkinnyShape skinny_shape(int64_t n, int64_t k, int sms) {
    const int64_t tiles = (n + kTileN - 1) / kTileN;
    const int64_t nkb = (k + kBlockK - 1) / kBlockK;
    const int64_t units = tiles * nkb;
    const int64_t cap = sms < kMaxCtas ? sms : kMaxCtas;
    if (tiles <= cap && 10 * tiles >= 7 * cap) return {tiles, 1};
    if (tiles < cap) {
        // each tile over a cluster of split CTAs (a power of two), each CTA
        // with at least kMinUnitsPerCta k-blocks
        int split = 1;
        while (split * 2 <= kMaxSplit && tiles * split * 2 <= cap && split * 2 * kMinUnitsPerCta <= nkb) split *= 2;
        return {tiles * split, split};
    }
    int64_t p = units / kMinUnitsPerCta;
    if (p > cap) p = cap;
    if (p < 1) p = 1;
    return {p, 1};
}

template <int NT, bool kBf16, bool kMx = false>
static cudaError_t launch_nt(const LinearArgs& a, void* workspace, int ctas, cudaStream_t st) {
    using L = SkinnySmem<NT>;
    auto kern = skinny_kernel<NT, kBf16, kMx>;
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
    SkinnyShape shape = ctas > 0 ? SkinnyShape{ctas, 1} : skinny_shape(a.n, a.k, sms);
    if (shape.grid > units) shape.grid = units;
    // programmatic dependent launch: this grid's prologue (barrier set-up,
    // TMEM allocation) overlaps the tail of the previous kernel in the
    // stream; every role waits for that kernel before touching global memory
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(shape.split);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(shape.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = shape.split > 1 ? 2 : 1;
    uint16_t* yp = static_cast<uint16_t*>(a.y);
    for (int64_t m0 = 0; m0 < a.m; m0 += NT) {
        const int rows = static_cast<int>(a.m - m0 < NT ? a.m - m0 : NT);
        const float* sc = kMx ? nullptr : a.scales;
        const uint8_t* e8 = kMx ? reinterpret_cast<const uint8_t*>(a.scales) : nullptr;
        e = cudaLaunchKernelEx(&cfg, kern, map_codes, map_x, sc, e8, a.bias, yp + m0 * a.n,
                               static_cast<uint8_t*>(workspace), rows, static_cast<int>(m0), a.n, a.k, shape.split,
                               a.early ? 1 : 0);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t skinny_workspace_size(int sms) { return skinny_workspace_bytes(sms < kMaxCtas ? sms : kMaxCtas); }

cudaError_t launch_skinny(const LinearArgs& a, void* workspace, int ctas, cudaStream_t st) {
    const bool bf16 = a.act == 1;
    if (a.e8m0) {
        // MX-style scales: bf16 activations, k % 128 == 0 (checked by the caller)
        if (!bf16 || a.group != 32 || a.k % 128 != 0) return cudaErrorInvalidValue;
        if (a.m <= 16) return launch_nt<16, true, true>(a, workspace, ctas, st);
        if (a.m <= 32) return launch_nt<32, true, true>(a, workspace, ctas, st);
        return launch_nt<64, true, true>(a, workspace, ctas, st);
    }
    if (a.m <= 16)
        return bf16 ? launch_nt<16, true>(a, workspace, ctas, st) : launch_nt<16, false>(a, workspace, ctas, st);
    if (a.m <= 32)
        return bf16 ? launch_nt<32, true>(a, workspace, ctas, st) : launch_nt<32, false>(a, workspace, ctas, st);
    // 64 tokens a launch (slabs of 64 beyond): each weight tile is dequantised
    // once for all of them
    return bf16 ? launch_nt<64, true>(a, workspace, ctas, st) : launch_nt<64, false>(a, workspace, ctas, st);
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
