// skinny.cu -- kernel K3: the M <= 64 linear layer on the tcgen05 tensor cores,
// "swap-AB": the weight channels are the 128-row A operand, the tokens the
// narrow B operand.
//
// Page "kadirnar/kernel-agent fp8-weights", section "Dequantise in
// registers" (skinny GEMM: the weight as the A operand, a 16-bit MMA in the
// activations' type, every code converted once and reused for every token,
// split-K so that all the GPU streams the weight).  That design targets
// mma.sync on sm_80..sm_120; this one is built for sm_103a:
//
//  * At most one CTA per SM.  The work is the list of units (channel tile
//    of 128, k-block of 128).  The grid is made of thread-block clusters of
//    `cl` CTAs, each cluster taking `tpc` consecutive tiles and each of its
//    ranks an even, contiguous share of their units:
//    - cl = 1: whole tiles, tpc of them a CTA (one when they nearly fill
//      the GPU);
//    - tpc = 1, cl > 1: few tiles, each split over a cluster;
//    - tpc > 1, cl > 1: more tiles than SMs (or an uneven count), shared.
//    A rank takes the whole tiles of its range first and the one or two
//    tiles it shares with neighbouring ranks last, holding their fp32
//    accumulators in TMEM; at the end it stages them in its idle code ring,
//    and after a cluster barrier every contributor of a shared tile adds up
//    its block of the tile's channels over all contributors' partials, in
//    rank order, through distributed shared memory.  Nothing is written to
//    global memory but y, no state outlives the launch, and the sums do not
//    depend on timing.  The host picks the shape with the fewest units per
//    CTA among those whose clusters all fit on the GPU at once.
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
//    y = round(fma(acc, scale, bias)), or holds a shared tile's partial.
//  * The control loops divide nothing per unit: a cursor walks (tile,
//    k-block), since a 64-bit division costs a lone thread hundreds of cycles.
//
// Every wait is bounded: on a timeout the CTA records an error code (the
// role and the barrier that gave up), raises an abort flag that ends every
// role's loop, lets its in-flight copies and MMAs finish, frees TMEM and
// exits.
#include <mutex>
#include <type_traits>

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
    // per-group scales: the accumulator columns hold a ring of kGAcc group
    // accumulators (NT columns each); gfull [kGAcc], gfree [kGAcc] follow drain
    static constexpr int kGAcc = (kTmemCols - kDCol0) / NT;
    static constexpr uint32_t kGBar0 = kLaneBars + kASlotsAll + kDoneSlots + kXSlots + 2 + 3 * kMmaWarps;
    static constexpr uint32_t kNumBars = kGBar0 + 2 * kGAcc;
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
        if (i >= kGBar0 + kGAcc) return 4u;                     // gfree
        return (gi == di || gi == di + 1) ? 4u : 1u;            // dfree
    }
};

// Partial tiles a rank holds at the end: at most two (the tile its range
// starts in and the one it ends in), each 128 channels x NT tokens of fp32,
// token-major, staged in the code ring once every unit is done.
constexpr int kMaxHeld = 2;
// Cluster sizes up to 16 (beyond 8 where the device allows non-portable
// clusters); the finish reads contributors' partials 8 ranks at a time.
constexpr int kMaxCluster = 16;
constexpr int kRankGroup = 8;
// Outputs whose remote partials one thread loads before adding them up.
constexpr int kRedBatch = 4;

// The units of one cluster: its t_g tiles, tile-major, cluster-local index
// (32-bit: the host keeps a cluster's units below 2^24); rank r takes the
// contiguous range [begin(r), begin(r + 1)).
struct ClusterRange {
    int units;
    int c;
    __device__ __forceinline__ int begin(int r) const { return r * units / c; }
    // the last rank whose range starts at or before u (every rank has units,
    // so this is the rank whose range holds u)
    __device__ __forceinline__ int owner(int u) const {
        int r = u * c / units;
        while (r + 1 < c && begin(r + 1) <= u) ++r;
        while (r > 0 && begin(r) > u) --r;
        return r;
    }
};

// Walks a rank's units in processing order without divisions: the range
// [a, b) (cluster-local units) is taken as [f, b) then [a, f), f the first
// tile boundary at or after a (or b), so the whole tiles come first and the
// one or two tiles the range shares with its neighbours come last; their
// accumulators are then held until the cluster adds them up.  `tile` is the
// global tile index.
struct UnitCursor {
    int it;
    int tile, kb, nkb;
    int u, a, f, b;
    int a_tile, a_kb;  // tile and k-block of unit a
    __device__ __forceinline__ void next() {
        ++it;
        ++u;
        if (u == b && f > a) {
            u = a;
            tile = a_tile;
            kb = a_kb;
            return;
        }
        if (++kb == nkb) {
            kb = 0;
            ++tile;
        }
    }
    // units left in the current segment (the current tile within the run)
    __device__ __forceinline__ int seg_left() const {
        const int left = (u >= f ? b : f) - u;
        return left < nkb - kb ? left : nkb - kb;
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

// A cluster rank's fp32 partial, read after the cluster barrier that made it
// visible (no compiler memory clobber, so loads of several ranks and tokens
// can be in flight together; volatile keeps them after the barrier).
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// One tile this rank shares with others of its cluster, as the finish sees
// it from one epilogue thread: the thread adds up channel `col` (or none)
// for tokens tok0, tok0 + tstep, ... over contributors r_lo .. r_lo + J - 1;
// lo_slot is the staging slot of contributor r_lo's partial (the others'
// is 0: the tile holds their first unit).
struct SharedTile {
    int64_t col;
    int r_lo, J, tok0, tstep, lo_slot;
    float sc, b;
};

// The scale forms (kMode):
//  kModeRow      scales[n], applied in the epilogue.
//  kModeMxFold   E8M0 scale bytes e8[n, k / 32] (bf16 activations, k % 128
//                == 0); they enter the dequantised weight, and the epilogue
//                adds only the bias.
//  kModeGrouped  one scale per run of gsz = 32, 64 or 128 codes of a row:
//                fp32 scales[n, k / gsz], or E8M0 bytes e8[n, k / 32] (gsz
//                32).  Page "B04 Precision & Quantization", section
//                "Post-training quantization versus quantization-aware
//                training", the granularity table's per-group row: each group's sum is
//                its own product, scaled before it joins the row's total.
//                The MMAs of a group go to their own TMEM accumulator (a ring
//                of kGAcc); the epilogue drains each one, multiplies it by
//                the group's scale and adds it to the tile's fp32 total in
//                registers (at most 32 tokens a launch, and at most one
//                shared tile a CTA).  kGpu = 128 / gsz groups a unit is a
//                compile-time constant (one kernel per group size: with it
//                known the hand-off loops unroll), and where the ring holds
//                the groups of two units or more the hand-off goes once a
//                unit rather than once a group.
template <int NT, bool kBf16, int kMode = kModeRow, int kGpu = 1>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x,
                  const float* __restrict__ scales, const uint8_t* __restrict__ e8, const float* __restrict__ bias,
                  uint16_t* __restrict__ y, int m_rows, int m_row0, int64_t n, int64_t k, int cl, int tpc,
                  int early, int gsz) {
    constexpr bool kMx = kMode == kModeMxFold;
    constexpr bool kGrp = kMode == kModeGrouped;
    static_assert(!kMx || kBf16, "MX-style scales fold into bf16 weights only");
    static_assert(!kGrp || NT <= 32, "per-group totals are held in registers: at most 32 tokens");
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
    constexpr int kGAcc = L::kGAcc;
    auto gfull = [&](int b) { return bar0 + 8u * (L::kGBar0 + b); };
    auto gfree = [&](int b) { return bar0 + 8u * (L::kGBar0 + kGAcc + b); };
    // groups a unit, and MMAs (k = 16) a group (grouped form)
    constexpr int gpu = kGrp ? kGpu : 1;                 // gsz == kBlockK / kGpu
    constexpr int mpg = kBlockK / 16 / gpu;
    // unit v's MMAs are done (v < 0: nothing to wait for)
    auto done_bar = [&](int v) { return udone(v % kDone); };
    auto done_parity = [&](int v) { return static_cast<uint32_t>((v / kDone) & 1); };
    auto code_smem = [&](int g, int s) { return L::kCodesOff + (g * kCS + s) * kCodeStageBytes; };
    auto x_smem = [&](int s) { return L::kXOff + s * L::kXStageBytes; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
    volatile int* ep_abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 12);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles = (n + kTileN - 1) / kTileN;
    const int64_t nkb = (k + kBlockK - 1) / kBlockK;
    // cluster g (cl CTAs) takes tiles [g * tpc, min((g + 1) * tpc, tiles));
    // its rank an even, contiguous share of their units (global unit index =
    // tile * nkb + k-block)
    const int g = static_cast<int>(blockIdx.x) / cl;
    const int rank = static_cast<int>(blockIdx.x) - g * cl;
    const int gt0 = g * tpc;  // the cluster's first tile
    const int gtiles = static_cast<int>(tiles - gt0 < tpc ? tiles - gt0 : tpc);
    const int nkb32 = static_cast<int>(nkb);
    const ClusterRange cr{gtiles * nkb32, cl};
    // this rank's cluster-local units [ua, ub); uf: the first tile boundary at
    // or after ua, capped at ub
    const int ua = cr.begin(rank), ub = cr.begin(rank + 1);
    const int iters = ub - ua;
    const int ua_tile = ua / nkb32, ua_kb = ua - ua_tile * nkb32;
    const int ua_up = ua_kb == 0 ? ua : ua + (nkb32 - ua_kb);
    const int uf = ua_up < ub ? ua_up : ub;
    auto cursor0 = [=]() {
        UnitCursor cu;
        cu.it = 0;
        cu.nkb = nkb32;
        cu.a = ua;
        cu.f = uf;
        cu.b = ub;
        cu.a_tile = gt0 + ua_tile;
        cu.a_kb = ua_kb;
        if (uf < ub) {
            cu.u = uf;
            cu.tile = gt0 + uf / nkb32;
            cu.kb = 0;
        } else {
            cu.u = ua;
            cu.tile = cu.a_tile;
            cu.kb = ua_kb;
        }
        return cu;
    };

    // Start-up: warp 0 sets up the code slots' barriers, warp 1 the
    // activation ring's; each then arrives at the start-up barrier without
    // waiting and begins streaming.  The MMA warp sets up the rest (used only
    // by warps that wait at that barrier) before it joins them there, so no
    // one warp spends ~1300 cycles on all of them while the stream waits.
    if (warp <= kXWarp) {
        // warp 1 sets up udone and xfull, [xb0, xb1): it is the first to wait on udone
        const uint32_t xb0 = static_cast<uint32_t>(L::kLaneBars + kAS);
        const uint32_t xb1 = xb0 + static_cast<uint32_t>(kDone + kXS);
        if (warp == 0) {
            // the code slots' barriers (the MMA warp sets up the others that
            // neither producer uses before the start-up barrier)
            for (uint32_t i = lane; i < L::kLaneBars; i += 32) mbar_init(bar0 + 8 * i, L::arrivals(i));
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
        if (warp == kMmaWarp) {
            // TMEM first (it waits for nothing here: one CTA per SM), then the
            // barriers
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
            const uint32_t xb0 = static_cast<uint32_t>(L::kLaneBars + kAS);
            const uint32_t xb1 = xb0 + static_cast<uint32_t>(kDone + kXS);
            for (uint32_t i = L::kLaneBars + lane; i < L::kNumBars; i += 32)
                if (i < xb0 || i >= xb1) mbar_init(bar0 + 8 * i, L::arrivals(i));
            fence_mbar_init();
        }
        asm volatile("bar.sync %0, %1;" ::"n"(kBarStart), "n"(kThreads) : "memory");
    }
    // let the next kernel in the stream start launching; its CTAs wait for
    // this grid to complete before they read or write global memory
    pdl_launch_dependents();
    // TMEM was allocated by the MMA warp during start-up; the warps that use
    // it meet the MMA warp at a named barrier first.
    uint32_t tmem = 0;
    if (warp >= kMmaWarp) {
        tc_fence_before();
        asm volatile("bar.sync %0, %1;" ::"n"(kBarTmem), "n"(kThreads - 32 * kMmaWarp) : "memory");
        tc_fence_after();
        tmem = *tmem_slot;
    }

    // the tiles this rank shares, as its epilogue thread finishes them (set
    // by the epilogue warps, used after every role is done)
    // (two named entries: an array indexed at run time would live in local memory)
    SharedTile sh0{-1, 0, 0, 0, 0, 1, 0.0f, 0.0f}, sh1{-1, 0, 0, 0, 0, 1, 0.0f, 0.0f};
    int nshared = 0;

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
        // Per-group form: a warp waits for an accumulator's previous group to
        // be drained by phase parity, which cannot tell that phase from the
        // one before it; with two warps taking alternate units, a warp's
        // waits stay within one phase only if the ring holds the groups of
        // two units (kGAcc >= 2 gpu).  Otherwise warp 2 alone issues every
        // unit, and its waits come in order.
        const int w = warp - kMmaWarp;
        constexpr int nw = (kGrp && kGAcc < 2 * gpu) ? 1 : kMmaWarps;  // issuing warps
        // per-group form with several groups a unit: one hand-off a unit where
        // the ring holds the groups of two units or more (g_per units)
        constexpr int g_per = kGrp ? kGAcc / gpu : 1;
        constexpr bool g_unit = kGrp && gpu > 1 && g_per >= 2;
        constexpr uint32_t idesc = idesc_f16(kBf16, NT);
        UnitCursor cu = cursor0();
        int seg = 0, jj = 0;
        int seg_len = iters > 0 ? cu.seg_left() : 0;
        int ra = w, rx = w;          // slots of this warp's next unit: A (unit % 6), activation (unit % kXS)
        uint32_t pa = 0, px = 0;     // their phase parities
        bool mine_in_seg = false;    // this warp has issued into the segment's accumulator
        bool failed = false;
        if (w < nw && w < iters &&
            (!mbar_wait_warp(aready(ra), pa, abort_flag) || !mbar_wait_warp(xfull(rx), px, abort_flag))) {
            if (lane == 0) record_error(kErrWaitDequant, abort_flag, aready(ra), bar0);
            failed = true;
        }
        for (int it = 0; it < iters && !failed; ++it) {
            const int d = seg % L::kDBuf;
            if (!kGrp && jj == 0 &&
                !mbar_wait_warp(dfree(d), static_cast<uint32_t>(((seg / L::kDBuf) & 1) ^ 1), abort_flag)) {
                // the epilogue has not drained this accumulator (two segments ago)
                if (lane == 0) record_error(kErrWaitMma, abort_flag, dfree(d), bar0);
                break;
            }
            if (nw == 1 ? w == 0 : (it & 1) == w) {
                // test this warp's next unit (it + nw) now; the answer is used
                // after this unit's MMAs, which hide the tests' latency
                const int ran = ra + nw >= kAS ? ra + nw - kAS : ra + nw;
                const int rxn = rx + nw >= kXS ? rx + nw - kXS : rx + nw;
                const uint32_t pan = ran < ra ? pa ^ 1u : pa;
                const uint32_t pxn = rxn < rx ? px ^ 1u : px;
                const bool more = it + nw < iters;
                const bool next_a = !more || mbar_test_wait(aready(ran), pan);
                const bool next_x = !more || mbar_test_wait(xfull(rxn), pxn);
                tc_fence_after();
                const uint32_t xs = sbase + x_smem(rx);
                const uint32_t a_tmem = tmem + ra * kAColsPerSlot;  // slot ra = (group ra % 3, A slot ra / 3)
                if constexpr (kGrp) {
                    // group G = it * gpu + q / mpg of the unit goes to accumulator
                    // G % kGAcc, once the epilogue has drained its previous group
                    uint32_t g_tmem = 0;
                    int gb = 0;
                    if constexpr (g_unit) {
                        // one hand-off a unit: the accumulator of the unit's last
                        // group (the epilogue drains in order, so the unit's other
                        // accumulators are free as well), one commit after its MMAs
                        const int bl = (it * gpu + gpu - 1) & (kGAcc - 1);
                        if (!mbar_wait_warp(gfree(bl), static_cast<uint32_t>(((it / g_per) & 1) ^ 1), abort_flag)) {
                            if (lane == 0) record_error(kErrWaitMma, abort_flag, gfree(bl), bar0);
                            failed = true;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int q = 0; q < kBlockK / 16; ++q) {
                            const int qg = q & (mpg - 1);
                            const uint64_t b_desc = smem_desc_sw128_kmajor(xs + (q >> 2) * L::kXBoxBytes + (q & 3) * 32);
                            mma_f16_ts_warp(tmem + kDCol0 + ((it * gpu + q / mpg) & (kGAcc - 1)) * NT, a_tmem + q * 8,
                                            b_desc, idesc, qg != 0);
                        }
                        tc_commit_warp(gfull(bl));
                    } else
#pragma unroll
                    for (int q = 0; q < kBlockK / 16; ++q) {
                        const int qg = q & (mpg - 1);
                        if (qg == 0) {
                            const int G = it * gpu + q / mpg;
                            gb = G & (kGAcc - 1);
                            if (!mbar_wait_warp(gfree(gb), static_cast<uint32_t>(((G / kGAcc) & 1) ^ 1), abort_flag)) {
                                if (lane == 0) record_error(kErrWaitMma, abort_flag, gfree(gb), bar0);
                                failed = true;
                                break;
                            }
                            tc_fence_after();
                            g_tmem = tmem + kDCol0 + gb * NT;
                        }
                        const uint64_t b_desc = smem_desc_sw128_kmajor(xs + (q >> 2) * L::kXBoxBytes + (q & 3) * 32);
                        mma_f16_ts_warp(g_tmem, a_tmem + q * 8, b_desc, idesc, qg != 0);
                        if (qg == mpg - 1) tc_commit_warp(gfull(gb));
                    }
                    if (failed) break;
                } else {
                    const uint32_t d_tmem = tmem + kDCol0 + (w * L::kDBuf + d) * NT;
#pragma unroll
                    for (int q = 0; q < kBlockK / 16; ++q) {
                        const uint64_t b_desc = smem_desc_sw128_kmajor(xs + (q >> 2) * L::kXBoxBytes + (q & 3) * 32);
                        mma_f16_ts_warp(d_tmem, a_tmem + q * 8, b_desc, idesc, mine_in_seg || q > 0);
                    }
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
            if (kGrp) continue;  // the epilogue follows the group accumulators
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
                if (it + 1 < iters) seg_len = cu.seg_left();
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
        pdl_wait();  // y may still be in use by the previous grid
        // The finish of the tiles this rank shares (the tiles of its first and
        // last units, when it does not cover them whole): their contributors
        // r_lo .. r_hi split each tile's channels into contiguous blocks,
        // contributor j taking the j-th; this thread takes one channel of the
        // block for a stride of tokens (a warp reads and writes consecutive
        // channels).  Worked out now, and its scale and bias read now, while
        // the MMAs run: at the end those reads would wait behind the weight
        // stream of the other CTAs.
        // (The per-group form works it out after its loop instead: its
        // registers hold the totals, and its finish reads no scale.)
        auto plan_shared = [&]() {
            const int etid = r;  // 0..127
            const int ub_tile = (ub - 1) / nkb32;
            for (int side = 0; side < 2; ++side) {
                const int tl = side == 0 ? ua_tile : ub_tile;
                if (side == 1 && tl == ua_tile) break;
                const int t_lo = tl * nkb32, t_hi = t_lo + nkb32;
                if (ua <= t_lo && ub >= t_hi) continue;  // covered whole
                SharedTile& st = nshared++ == 0 ? sh0 : sh1;
                st.r_lo = cr.owner(t_lo);
                st.J = cr.owner(t_hi - 1) - st.r_lo + 1;
                st.lo_slot = cr.begin(st.r_lo) == t_lo ? 0 : 1;
                const int j = rank - st.r_lo;
                const int c0 = j * kTileN / st.J, c1 = (j + 1) * kTileN / st.J;
                const int my_nch = c1 - c0;
                st.tstep = kTileN / my_nch;
                st.tok0 = etid / my_nch;
                const int ci = etid - st.tok0 * my_nch;
                st.col = -1;
                st.sc = 0.0f;
                st.b = 0.0f;
                if (st.tok0 < st.tstep) {
                    const int64_t col = static_cast<int64_t>(gt0 + tl) * kTileN + c0 + ci;
                    if (col < n) {
                        st.col = col;
                        st.sc = (kMx || kGrp) ? 1.0f : scales[col];
                        st.b = bias ? bias[col] : 0.0f;
                    }
                }
            }
        };
        if (!kGrp && cl > 1 && iters > 0) plan_shared();
        if constexpr (kGrp) {
            // Per-group scales: for each unit in processing order, each of its
            // groups' accumulators is drained as soon as its MMAs are done and
            // added to this channel's fp32 totals times the group's scale.
            const int64_t nsc = e8 ? (k >> 5) : k / gsz;  // scales a row
            const int gpr = static_cast<int>(nsc);
            auto scale_at = [&](int64_t col, int j) -> float {
                if (col >= n || j >= gpr) return 0.0f;  // rows past n, groups past k: zero codes
                return e8 ? e8m0_to_f32(__ldg(e8 + col * nsc + j)) : __ldg(scales + col * nsc + j);
            };
            // the totals as fp32 pairs (packed FMAs); tot(t) is token t's
            uint64_t tot2[NT / 2];
#pragma unroll
            for (int t = 0; t < NT / 2; ++t) tot2[t] = 0ull;
            auto tot = [&](int t) { return __uint_as_float(static_cast<uint32_t>(tot2[t >> 1] >> (32 * (t & 1)))); };
            // the scales of the unit after the current one, loaded a unit ahead
            float sn[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            UnitCursor cu = cursor0();
            if (iters > 0) {
#pragma unroll
                for (int sg = 0; sg < 4; ++sg)
                    if (sg < gpu) sn[sg] = scale_at(static_cast<int64_t>(cu.tile) * kTileN + r, cu.kb * gpu + sg);
            }
            bool held = false;
            int G = 0;
            // one hand-off a unit where the MMA warps make one (the same rule)
            constexpr int g_per_e = kGAcc / gpu;
            constexpr bool g_unit_e = gpu > 1 && g_per_e >= 2;
            bool ok = true;
            for (int it = 0; it < iters && ok;) {
                const int seg_len = cu.seg_left();
                const int64_t col = static_cast<int64_t>(cu.tile) * kTileN + r;
                const bool whole = cu.kb == 0 && seg_len == cu.nkb;
                for (int jj = 0; jj < seg_len; ++jj, ++it) {
                    float sc[4];
#pragma unroll
                    for (int sg = 0; sg < 4; ++sg) sc[sg] = sn[sg];
                    cu.next();
                    if (it + 1 < iters) {
#pragma unroll
                        for (int sg = 0; sg < 4; ++sg)
                            if (sg < gpu) sn[sg] = scale_at(static_cast<int64_t>(cu.tile) * kTileN + r, cu.kb * gpu + sg);
                    }
                    if constexpr (g_unit_e) {
                        // one hand-off a unit (the MMA warps commit once, on the
                        // barrier of the unit's last group's accumulator)
                        const int u = G / gpu;
                        const int bl = (G + gpu - 1) & (kGAcc - 1);
                        if (!mbar_wait_warp(gfull(bl), static_cast<uint32_t>((u / g_per_e) & 1), abort_flag)) {
                            if (lane == 0) *ep_abort = 1;
                            record_error(kErrWaitMma, abort_flag, gfull(bl), bar0);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int sg = 0; sg < 4; ++sg) {
                            if (sg >= gpu) break;
                            const int gb = (G + sg) & (kGAcc - 1);
#pragma unroll
                            for (int h = 0; h < NT / 16; ++h) {
                                if (h * 16 >= m_rows) break;
                                uint32_t v[16];
                                tmem_ld_x16_sync(lane_addr + kDCol0 + gb * NT + h * 16, v);
                                ffma2_x16(tot2 + h * 8, v, pack2(sc[sg], sc[sg]));
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(gfree(bl));
                        G += gpu;
                        continue;
                    }
#pragma unroll
                    for (int sg = 0; sg < 4; ++sg) {
                        if (sg >= gpu) break;
                        const int gb = G & (kGAcc - 1);
                        if (!mbar_wait_warp(gfull(gb), static_cast<uint32_t>((G / kGAcc) & 1), abort_flag)) {
                            if (lane == 0) *ep_abort = 1;
                            record_error(kErrWaitMma, abort_flag, gfull(gb), bar0);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // 16 tokens at a time (registers: the totals stay resident)
#pragma unroll
                        for (int h = 0; h < NT / 16; ++h) {
                            if (h * 16 >= m_rows) break;
                            uint32_t v[16];
                            tmem_ld_x16_sync(lane_addr + kDCol0 + gb * NT + h * 16, v);
                            ffma2_x16(tot2 + h * 8, v, pack2(sc[sg], sc[sg]));
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(gfree(gb));
                        ++G;
                    }
                    if (!ok) break;
                }
                if (!ok) break;
                if (!whole) {
                    // the one tile this rank shares (clusters split single tiles
                    // in this form): its totals are staged after the loop
                    held = true;
                    continue;
                }
                if (col < n) {
                    const float b = bias ? bias[col] : 0.0f;
#pragma unroll
                    for (int t = 0; t < NT; ++t)
                        if (t < m_rows) y[static_cast<int64_t>(t) * n + col] = round_out<kBf16>(tot(t) + b);
                }
#pragma unroll
                for (int t = 0; t < NT / 2; ++t) tot2[t] = 0ull;
            }
            if (held && !*ep_abort) {
                float* pt = reinterpret_cast<float*>(smem + L::kCodesOff);
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    if (t < m_rows) pt[t * kTileN + r] = tot(t);
            }
            if (cl > 1 && iters > 0) plan_shared();
        } else {
            // tokens [16h, 16h + 16) of the accumulators of buffer d, warp 0's
            // first; a warp with no unit in the segment (a one-unit segment)
            // wrote nothing there
            auto load_acc = [&](int d, int h, int it0, int seg_len, float (&acc)[16]) {
    #pragma unroll
                for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
    #pragma unroll
                for (int w = 0; w < kMmaWarps; ++w) {
                    if (seg_len < kMmaWarps && ((it0 + kMmaWarps - w) % kMmaWarps) >= seg_len) continue;
                    uint32_t v[16];
                    tmem_ld_x16_sync(lane_addr + kDCol0 + (w * L::kDBuf + d) * NT + h * 16, v);
    #pragma unroll
                    for (int q = 0; q < 16; ++q) acc[q] += __uint_as_float(v[q]);
                }
            };
            // a tile this rank shares with others stays in its accumulator until
            // every unit is done (such tiles are processed last): buffer, first
            // unit, length and staging slot (0: the tile of the rank's first unit)
            // (two entries in registers: the arrays would live in local memory)
            int hd0 = 0, hit0 = 0, hlen0 = 0, hslot0 = 0, hd1 = 0, hit1 = 0, hlen1 = 0, hslot1 = 0;
            int nheld = 0;
            int seg = 0;
            UnitCursor cu = cursor0();
            for (int it = 0; it < iters; ++seg) {
                // segment: the units of one tile, contiguous in processing order
                const int seg_len = cu.seg_left();
                const int64_t tile = cu.tile;
                const bool whole = cu.kb == 0 && seg_len == cu.nkb;
                const int it0 = it;
                it += seg_len;
                for (int jj = 0; jj < seg_len; ++jj) cu.next();
                const int d = seg % L::kDBuf;
                bool ok = true;
                for (int w = 0; w < kMmaWarps; ++w)
                    ok = mbar_wait_warp(dready(w, d), static_cast<uint32_t>((seg / L::kDBuf) & 1), abort_flag) && ok;
                if (!ok) {
                    if (lane == 0) *ep_abort = 1;
                    record_error(kErrWaitMma, abort_flag);
                }
                // the four epilogue warps leave together (ep_abort is written only
                // by them, before this barrier), so their named barriers stay matched
                epilogue_bar();
                if (*ep_abort) break;
                tc_fence_after();
                if (!whole) {
                    const int slot = tile == gt0 + ua_tile ? 0 : 1;
                    if (nheld == 0) {
                        hd0 = d, hit0 = it0, hlen0 = seg_len, hslot0 = slot;
                    } else {
                        hd1 = d, hit1 = it0, hlen1 = seg_len, hslot1 = slot;
                    }
                    ++nheld;
                    continue;
                }
                const int64_t col = tile * kTileN + r;
                const float sc = kMx ? 1.0f : col < n ? scales[col] : 0.0f;
                const float b = (bias && col < n) ? bias[col] : 0.0f;
                // 16 tokens at a time, only as many as there are rows
    #pragma unroll 1
                for (int h = 0; h < NT / 16 && h * 16 < m_rows; ++h) {
                    float acc[16];
                    load_acc(d, h, it0, seg_len, acc);
                    if (col < n) {
    #pragma unroll
                        for (int q = 0; q < 16; ++q)
                            if (h * 16 + q < m_rows)
                                y[static_cast<int64_t>(h * 16 + q) * n + col] = round_out<kBf16>(fmaf(acc[q], sc, b));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dfree(d));
            }
            // every unit is done, so the code ring is idle: the held partial
            // tiles go there, token-major, for the cluster to add up
            if (!*ep_abort) {
    #pragma unroll 1
                for (int i = 0; i < nheld && i < kMaxHeld; ++i) {
                    const int hd = i == 0 ? hd0 : hd1, hit = i == 0 ? hit0 : hit1, hlen = i == 0 ? hlen0 : hlen1;
                    float* pt = reinterpret_cast<float*>(smem + L::kCodesOff) + (i == 0 ? hslot0 : hslot1) * (kTileN * NT);
    #pragma unroll 1
                    for (int h = 0; h < NT / 16 && h * 16 < m_rows; ++h) {
                        float acc[16];
                        load_acc(hd, h, hit, hlen, acc);
    #pragma unroll
                        for (int q = 0; q < 16; ++q)
                            if (h * 16 + q < m_rows) pt[(h * 16 + q) * kTileN + r] = acc[q];
                    }
                }
            }
        }
    } else {
        // ------------------------------- dequantising warpgroups (8-19) --
        const int group = (warp - kFirstDequantWarp) >> 2;
        // MX: this thread's row's four scale bytes of a unit (one word), loaded
        // a unit ahead; mcu walks this group's units one ahead of the loop
        UnitCursor mcu = cursor0();
        uint32_t mx_next = 0x7F7F7F7Fu;
        auto mx_load = [&](int64_t tile, int kb) -> uint32_t {
            const int64_t row = tile * kTileN + (warp & 3) * 32 + lane;
            // rows past n hold zero codes (the copy's fill): any scale does
            return row < n ? __ldg(reinterpret_cast<const uint32_t*>(e8 + row * (k >> 5) + kb * 4)) : 0x7F7F7F7Fu;
        };
        if constexpr (kMx) {
            if (!early) pdl_wait();  // the scales may come from the previous kernel
            for (int i = 0; i < group; ++i) mcu.next();
            if (group < iters) mx_next = mx_load(mcu.tile, mcu.kb);
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
                for (int i = 0; i < kLanes; ++i) mcu.next();
                if (it + kLanes < iters) mx_next = mx_load(mcu.tile, mcu.kb);
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
    if (cl > 1) {
        // Every rank's held partials are in its shared memory.  For each tile
        // this rank shares (the tiles of its first and last units, when it
        // does not cover them whole), its contributors r_lo..r_hi split the
        // tile's outputs: contributor j adds up channels j, j + J, ... over all
        // contributors in rank order (so in k order) and writes y.  Every
        // thread of the CTA takes part; kRedBatch outputs' remote loads are
        // issued before any sum, so their round trips overlap.
        cluster_sync_all();
        const bool epi = warp >= kFirstEpilogueWarp && warp < kFirstDequantWarp;
        if (epi && !*ep_abort) {
#pragma unroll 1
            for (int i = 0; i < nshared && i < kMaxHeld; ++i) {
                const SharedTile& st = i == 0 ? sh0 : sh1;
                if (st.col < 0) continue;
                const int ch = static_cast<int>(st.col % kTileN);
                // contributors' partials of this tile, 8 ranks at a time, added
                // in rank order; a contributor's staging slot is 0 if the tile
                // holds its first unit
                for (int tk0 = st.tok0; tk0 < m_rows; tk0 += kRedBatch * st.tstep) {
                    float t[kRedBatch];
#pragma unroll
                    for (int e = 0; e < kRedBatch; ++e) t[e] = 0.0f;
                    for (int rg = 0; rg < st.J; rg += kRankGroup) {
                        float v[kRedBatch][kRankGroup];
#pragma unroll
                        for (int rr = 0; rr < kRankGroup; ++rr) {
                            if (rg + rr >= st.J) break;
                            const int rk = st.r_lo + rg + rr;
                            const int slot = rg + rr == 0 ? st.lo_slot : 0;
                            const uint32_t src = mapa_shared(
                                sbase + L::kCodesOff + static_cast<uint32_t>((slot * kTileN * NT + ch) * 4), rk);
#pragma unroll
                            for (int e = 0; e < kRedBatch; ++e) {
                                const int tk = tk0 + e * st.tstep;
                                if (tk < m_rows) v[e][rr] = ld_dsmem_f32(src + static_cast<uint32_t>(tk * kTileN * 4));
                            }
                        }
#pragma unroll
                        for (int rr = 0; rr < kRankGroup; ++rr) {
                            if (rg + rr >= st.J) break;
#pragma unroll
                            for (int e = 0; e < kRedBatch; ++e) t[e] += v[e][rr];
                        }
                    }
#pragma unroll
                    for (int e = 0; e < kRedBatch; ++e) {
                        const int tk = tk0 + e * st.tstep;
                        if (tk < m_rows) y[static_cast<int64_t>(tk) * n + st.col] = round_out<kBf16>(fmaf(t[e], st.sc, st.b));
                    }
                }
            }
        }
        // no rank leaves while its partials may still be read
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

bool encode_3d_blocks(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k, uint32_t box_rows,
                      uint32_t box_blocks) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn || k % 128 != 0) return false;
    // byte (r, kb, c) of the [rows, k] matrix is at r * k + kb * 128 + c
    const cuuint64_t dims[3] = {128, rows, k / 128};
    const cuuint64_t strides[2] = {k, 128};
    const cuuint32_t box[3] = {128, box_rows, box_blocks};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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

// Launch shape: clusters of `cl` CTAs, each cluster taking `tpc`
// consecutive tiles (the last cluster may take fewer).  A CTA's time is its
// units times the per-unit loop, so the shape with the fewest units per CTA
// wins among those whose clusters all run at once: active[cl] is how many
// clusters of cl CTAs the device holds at a time (a cluster lives in one GPC,
// so a GPC whose SM count cl does not divide leaves SMs idle; active[1] is
// the SM count).  Sharing tiles costs a fixed finish, counted in units
// (measured on GB300 against whole tiles at a ~0.38 us unit): about 2 us
// when a cluster splits one tile (kSplitUnits; [22, 1024] x [1024, 4096]
// fp16, 8 k-blocks a tile: 5.1 us as 32 whole tiles, 5.9 us split over
// clusters of 2), about 3.3 us when its ranks hold two shared tiles each
// (kSharedUnits: both partials wait for the end, and a cluster starts only
// when all its SMs are free).  Each rank gets at least kMinUnitsPerCta
// units (and at least one of every cluster's, so cl <= nkb).  A 64-token launch keeps
// one accumulator per MMA warp, and the per-group form keeps a tile's totals
// in registers, so their CTAs may share at most one tile: tpc == 1 when
// cl > 1.
constexpr int kMinUnitsPerCta = 4;
constexpr int kSplitUnits = 6;
constexpr int kSharedUnits = 9;
constexpr int64_t kMaxClusterUnits = 1 << 24;  // cluster-local unit indices are 32-bit

SkinnyShape skinny_shape(int64_t n, int64_t k, const int* active, int nt, bool grouped) {
    const int64_t tiles = (n + kTileN - 1) / kTileN;
    const int64_t nkb = (k + kBlockK - 1) / kBlockK;
    SkinnyShape best{1, (tiles + active[1] - 1) / active[1]};
    int64_t best_cost = best.tpc * nkb;
    for (int cl = 2; cl <= kMaxCluster && cl <= nkb; ++cl) {
        const int64_t clusters_max = active[cl];
        if (clusters_max < 1) continue;
        const int64_t tpc = (tiles + clusters_max - 1) / clusters_max;
        if ((nt > 32 || grouped) && tpc > 1) continue;
        if (tpc * nkb >= kMaxClusterUnits) continue;
        const int64_t per_cta = (tpc * nkb + cl - 1) / cl;
        if (per_cta < kMinUnitsPerCta) continue;
        const int64_t cost = per_cta + (tpc == 1 ? kSplitUnits : kSharedUnits);
        if (cost < best_cost) {
            best_cost = cost;
            best = {cl, tpc};
        }
    }
    return best;
}

bool skinny_shape_valid(const SkinnyShape& sh, int64_t m, int64_t k, bool grouped) {
    const int64_t nkb = (k + kBlockK - 1) / kBlockK;
    const int nt = m <= 16 ? 16 : m <= 32 ? 32 : 64;
    return sh.cl >= 1 && sh.cl <= kMaxCluster && sh.tpc >= 1 && sh.cl <= nkb && sh.tpc * nkb < kMaxClusterUnits &&
           (sh.cl == 1 || (nt <= 32 && !grouped) || sh.tpc == 1);
}

template <int NT, bool kBf16, int kMode = kModeRow, int kGpu = 1>
static cudaError_t launch_nt(const LinearArgs& a, const SkinnyShape* forced, cudaStream_t st) {
    using L = SkinnySmem<NT>;
    constexpr bool kMx = kMode == kModeMxFold;
    constexpr bool kGrp = kMode == kModeGrouped;
    auto kern = skinny_kernel<NT, kBf16, kMode, kGpu>;
    // per device, once: the kernel's attributes, and how many clusters of
    // each size the device holds at a time (0 where a size cannot launch)
    static std::once_flag attr_once[64];
    static int active[64][kMaxCluster + 1];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = 0;
    e = device_sm_count(sms);
    if (e != cudaSuccess) return e;
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev], [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
        if (attr_err != cudaSuccess) return;
        const bool nonportable =
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        active[dev][1] = sms;
        for (int cl = 2; cl <= kMaxCluster; ++cl) {
            active[dev][cl] = 0;
            if (cl > 8 && !nonportable) continue;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = static_cast<unsigned>(cl);
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            cudaLaunchConfig_t qc = {};
            qc.gridDim = dim3(static_cast<unsigned>(cl * sms));
            qc.blockDim = dim3(kThreads);
            qc.dynamicSmemBytes = L::kAlloc;
            qc.attrs = qa;
            qc.numAttrs = 1;
            int num = 0;
            if (cudaOccupancyMaxActiveClusters(&num, kern, &qc) == cudaSuccess) active[dev][cl] = num;
            else (void)cudaGetLastError();  // an unsupported size: leave it out
        }
    });
    if (attr_err != cudaSuccess) return attr_err;

    CUtensorMap map_codes, map_x;
    if (!encode_2d(&map_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, static_cast<uint64_t>(a.k),
                   static_cast<uint64_t>(a.n), static_cast<uint64_t>(a.k), kBlockK, kTileN))
        return cudaErrorInvalidValue;
    if (!encode_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.x, static_cast<uint64_t>(a.k),
                   static_cast<uint64_t>(a.m), static_cast<uint64_t>(a.k) * 2, 64, NT))
        return cudaErrorInvalidValue;

    const SkinnyShape shape = forced ? *forced : skinny_shape(a.n, a.k, active[dev], NT, kGrp);
    const int64_t tiles = (a.n + kTileN - 1) / kTileN;
    const int64_t clusters = (tiles + shape.tpc - 1) / shape.tpc;
    // programmatic dependent launch: this grid's prologue (barrier set-up,
    // TMEM allocation) overlaps the tail of the previous kernel in the
    // stream; every role waits for that kernel before touching global memory
    // (the code producer too, unless the caller states the weights were
    // complete before it)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(shape.cl);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * shape.cl));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = shape.cl > 1 ? 2 : 1;
    uint16_t* yp = static_cast<uint16_t*>(a.y);
    for (int64_t m0 = 0; m0 < a.m; m0 += NT) {
        const int rows = static_cast<int>(a.m - m0 < NT ? a.m - m0 : NT);
        const bool bytes = kMx || (kGrp && a.e8m0);
        const float* sc = bytes ? nullptr : a.scales;
        const uint8_t* e8 = bytes ? reinterpret_cast<const uint8_t*>(a.scales) : nullptr;
        e = cudaLaunchKernelEx(&cfg, kern, map_codes, map_x, sc, e8, a.bias, yp + m0 * a.n, rows,
                               static_cast<int>(m0), a.n, a.k, shape.cl, static_cast<int>(shape.tpc),
                               a.early ? 1 : 0, kGrp ? static_cast<int>(a.group) : 0);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_skinny(const LinearArgs& a, const SkinnyShape* forced, cudaStream_t st) {
    const bool bf16 = a.act == 1;
    // per-group scales (fp32, or E8M0 bytes with fp16 activations): the
    // per-group form, 16 or 32 tokens a launch (32-row slabs beyond)
    const bool grouped = a.group != 0 && (!a.e8m0 || !bf16);
    if (forced && !skinny_shape_valid(*forced, a.m, a.k, grouped)) return cudaErrorInvalidConfiguration;
    if (grouped) {
        if (a.k % a.group != 0 || (a.group != 32 && a.group != 64 && a.group != 128) || (a.e8m0 && a.group != 32))
            return cudaErrorInvalidValue;
        // one kernel per group count a unit (1, 2 or 4 groups of 128, 64 or 32)
        auto by_groups = [&](auto gpu_tag) -> cudaError_t {
            constexpr int kG = decltype(gpu_tag)::value;
            if (a.m <= 16)
                return bf16 ? launch_nt<16, true, kModeGrouped, kG>(a, forced, st)
                            : launch_nt<16, false, kModeGrouped, kG>(a, forced, st);
            return bf16 ? launch_nt<32, true, kModeGrouped, kG>(a, forced, st)
                        : launch_nt<32, false, kModeGrouped, kG>(a, forced, st);
        };
        if (a.group == 128) return by_groups(std::integral_constant<int, 1>{});
        if (a.group == 64) return by_groups(std::integral_constant<int, 2>{});
        return by_groups(std::integral_constant<int, 4>{});
    }
    if (a.e8m0) {
        // MX-style scales: bf16 activations, k % 128 == 0 (checked by the caller)
        if (!bf16 || a.group != 32 || a.k % 128 != 0) return cudaErrorInvalidValue;
        if (a.m <= 16) return launch_nt<16, true, kModeMxFold>(a, forced, st);
        if (a.m <= 32) return launch_nt<32, true, kModeMxFold>(a, forced, st);
        return launch_nt<64, true, kModeMxFold>(a, forced, st);
    }
    if (a.m <= 16) return bf16 ? launch_nt<16, true>(a, forced, st) : launch_nt<16, false>(a, forced, st);
    if (a.m <= 32) return bf16 ? launch_nt<32, true>(a, forced, st) : launch_nt<32, false>(a, forced, st);
    // 64 tokens a launch (slabs of 64 beyond): each weight tile is dequantised
    // once for all of them
    return bf16 ? launch_nt<64, true>(a, forced, st) : launch_nt<64, false>(a, forced, st);
}

int read_skinny_device_error() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_skinny_error, sizeof v) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_skinny_error, &zero, sizeof zero);
    return v;
}

}  // namespace fp8w
