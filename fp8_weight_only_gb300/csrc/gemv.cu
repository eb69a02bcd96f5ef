// gemv.cu -- kernel K2: the M = 1 linear layer (GEMV) on CUDA cores.
//
// Page "kadirnar/kernel-agent fp8-weights", section "Dequantise in
// registers": the codes are streamed once past L1, converted in registers
// (exactly), multiplied by x with fp32 accumulation, reduced across a warp
// with shuffles, and scale (and bias) are applied once per output in the
// epilogue.
//
// GB300 layout of the work:
//  * The weight is cut into row blocks of R whole rows (up to 64 KB), one
//    per CTA of the grid; a CTA does its own block and then, through the
//    grid scheduler's cluster launch control, cancels CTAs that have not
//    started yet and does their blocks (one request in flight).  SMs that
//    free up early take more of the weight, so the launch ends evenly, and
//    a CTA allowed to start before the previous kernel finishes (weights
//    ready) streams its own block meanwhile; it asks for more only once
//    that kernel is done.  Nothing outside the launch keeps count.
//  * The last warp moves a block (R*K contiguous bytes) per 1-D TMA bulk
//    copy into a ring of slots.  A bulk copy costs the SM's TMA unit a fixed
//    ~0.27 us whatever its size (measured: 4 KB copies stream 15 GB/s per
//    SM, 64 KB copies 218 GB/s), so copies are large (32 and 48 KB blocks
//    measured slower on the 58.7 MB weights).
//  * A slot's rows are dealt round-robin to groups of G compute warps (16
//    warps; G = 1 when a slot holds many rows, more for long rows, so that
//    two slots keep every warp busy); lane l of the group's warp w takes the
//    16-code chunks (32w + l) + 32G*j of its rows, and a group of several
//    warps reduces through shared memory.  Every warp waits for every slot in order
//    and arrives once on its "empty" barrier after its rows there (none, if
//    the slot has fewer rows than warps): a warp whose next row lay several
//    slots ahead would otherwise wait on a slot a full ring cycle early and
//    pass on the previous phase of the same parity.
//  * x is staged once in shared memory (widened to fp32 for rows up to 8192
//    codes, as 16-bit values beyond); a row's scale and bias are read when
//    its sum is done.
//  * Codes are converted exactly by the hardware e4m3x2 -> f16x2 conversion
//    and widened to fp32, and products go two at a time through the packed
//    fma.rn.f32x2.  A warp computes two rows at once, so each activation it
//    reads serves both: x is read as fp32 straight from shared memory for
//    rows up to 8192 codes (about 2.4 instructions a code), and widened from
//    its 16-bit pairs for longer rows.
//  * A row's partial sums are reduced with a shuffle tree; one lane applies
//    fmaf(acc, scale, bias) and rounds once.
// HBM bytes per output channel: K (codes) + 4 (scale) + 4 (bias) + 2 (y).
#include <mutex>

#include "fp8w_device.cuh"
#include "fp8w_internal.h"

namespace fp8w {

static __device__ int g_gemv_error;

constexpr int kGemvWarps = 16;                       // compute warps
constexpr int kGemvThreads = 32 * (kGemvWarps + 1);  // + the producer warp
constexpr int kGemvMaxSlots = 8;
constexpr uint32_t kGemvSlotTarget = 64 * 1024;      // bytes per bulk copy, up to
constexpr uint32_t kGemvSmemBudget = 224 * 1024;
// Largest K the GEMV takes: x (2 bytes a value) and two 64 KB slots fit
// beside the staged scales.
constexpr int64_t kGemvMaxK = 32768;

struct GemvGeom {
    int rows;         // rows per slot (R)
    int slots;        // slots in the ring (S)
    int g;            // warps per row group (1, 2, 4, 8 or 16)
    uint32_t slot_bytes;
    uint32_t ring_bytes;   // code slots, then (per-group scales) scale slots
    uint32_t sslot_bytes;  // per-group scales: a slot's rows of scales (0 otherwise)
    int ngroups;           // per-group scales: groups a row (k / group)
    int gshift;            // per-group scales: log2 of 16-code chunks a group
    int early;             // the weights were complete before the preceding
                           // kernel started: stream them without waiting for it
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// Blackwell cluster launch control: ask the grid scheduler to cancel a CTA
// of this grid that has not started yet, so that this CTA does its work
// instead.  The 16-byte answer lands at `resp` (shared, 16-byte aligned) and
// completes `bar` (expecting 16 bytes of transaction).
__device__ __forceinline__ void cancel_request(uint32_t resp, uint32_t bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(resp),
        "r"(bar)
        : "memory");
}
// The answer: the x index of the cancelled CTA, or -1 if none was left.
__device__ __forceinline__ int64_t cancel_answer(uint32_t resp) {
    uint32_t ok, id;
    asm volatile(
        "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t.reg .b64 lo, hi;\n\t"
        "ld.shared.v2.b64 {lo, hi}, [%2];\n\t"
        "mov.b128 r, {lo, hi};\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(ok), "=r"(id)
        : "r"(resp)
        : "memory");
    return ok ? static_cast<int64_t>(id) : -1;
}

// f16x2 -> two fp32 (the halves selected in the register, no extraction).
__device__ __forceinline__ void f16x2_to_f32x2(uint32_t h, float& lo, float& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
}

// A 16-bit pair of x widened to an fp32 pair.
template <bool kBf16>
__device__ __forceinline__ uint64_t widen_x(uint32_t w) {
    if constexpr (kBf16) {
        return static_cast<uint64_t>(w << 16) | (static_cast<uint64_t>(w & 0xFFFF0000u) << 32);
    } else {
        float lo, hi;
        f16x2_to_f32x2(w, lo, hi);
        return pack2(lo, hi);
    }
}
// Four codes (one word) widened to two fp32 pairs, exactly.
__device__ __forceinline__ void widen_codes(uint32_t w, uint64_t& p01, uint64_t& p23) {
    uint32_t h01, h23;
    e4m3x4_to_f16x2(w, h01, h23);
    float v0, v1, v2, v3;
    f16x2_to_f32x2(h01, v0, v1);
    f16x2_to_f32x2(h23, v2, v3);
    p01 = pack2(v0, v1);
    p23 = pack2(v2, v3);
}

// RP rows' 16-code chunks against the same 16 activations: acc[r] is a pair
// of partial sums (even, odd positions) of row r.
template <int RP, bool kBf16>
__device__ __forceinline__ void dot_chunk(const uint4 (&c)[RP], const uint4 xa, const uint4 xb, uint64_t (&acc)[RP]) {
    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint64_t x01 = widen_x<kBf16>(xw[2 * q]), x23 = widen_x<kBf16>(xw[2 * q + 1]);
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const uint32_t w = q == 0 ? c[r].x : q == 1 ? c[r].y : q == 2 ? c[r].z : c[r].w;
            uint64_t p01, p23;
            widen_codes(w, p01, p23);
            ffma2(acc[r], x01, p01);
            ffma2(acc[r], x23, p23);
        }
    }
}

// RP rows' 16-code chunks against 16 fp32 activations (4 x 16 bytes).
template <int RP>
__device__ __forceinline__ void dot_chunk_f32(const uint4 (&c)[RP], const uint4 (&xf)[4], uint64_t (&acc)[RP]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint64_t x01 = static_cast<uint64_t>(q == 0 ? xf[0].x : q == 1 ? xf[1].x : q == 2 ? xf[2].x : xf[3].x) |
                             (static_cast<uint64_t>(q == 0 ? xf[0].y : q == 1 ? xf[1].y : q == 2 ? xf[2].y : xf[3].y) << 32);
        const uint64_t x23 = static_cast<uint64_t>(q == 0 ? xf[0].z : q == 1 ? xf[1].z : q == 2 ? xf[2].z : xf[3].z) |
                             (static_cast<uint64_t>(q == 0 ? xf[0].w : q == 1 ? xf[1].w : q == 2 ? xf[2].w : xf[3].w) << 32);
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const uint32_t w = q == 0 ? c[r].x : q == 1 ? c[r].y : q == 2 ? c[r].z : c[r].w;
            uint64_t p01, p23;
            widen_codes(w, p01, p23);
            ffma2(acc[r], x01, p01);
            ffma2(acc[r], x23, p23);
        }
    }
}

// kF32X: x is staged in shared memory as fp32 (else as 16-bit values).
// kGrouped: scales[n, k / group], one per run of `group` codes of a row (page
// "B04 Precision & Quantization", section "Post-training quantization versus
// quantization-aware training", the per-group row): the producer brings each
// slot's rows of scales with its codes, and every 16-code chunk's partial
// sums enter the row's sums times their group's scale (one packed FMA), so
// the epilogue adds only the bias.
// kGS: 0 one fp32 scale a row; 1 fp32 scales per group (kGrouped); 2 the
// MX-style form (page "11. Inference with NVFP4/MXFP8", section
// "MXFP8-Style FP8"): one E8M0 byte per 32 codes, worth 2^(b - 127), which
// scales the partials exactly like an fp32 group scale.
template <int RP, bool kBf16, bool kF32X, int kGS>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                const float* __restrict__ bias, uint16_t* __restrict__ y, int64_t n, int64_t k, GemvGeom geo) {
    constexpr bool kGrouped = kGS != 0;
    constexpr bool kE8 = kGS == 2;
    constexpr int kScaleBytes = kE8 ? 1 : 4;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t ring = smem_u32(smem);
    const int S = geo.slots, R = geo.rows;
    // layout: ring (codes [S], then group scales [S]) | x [k] | full, empty [kGemvMaxSlots] |
    // group partial sums [kGemvWarps][2][kGemvWarps][RP] | abort flag | slot blocks [kGemvMaxSlots] |
    // cancel answers [2] (16 B each) | their barriers [2]
    const uint32_t x_bytes = static_cast<uint32_t>(((k * (kF32X ? 4 : 2) + 127) / 128) * 128);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + geo.ring_bytes);
    const uint32_t bar_full = smem_u32(smem + geo.ring_bytes + x_bytes);
    const uint32_t bar_empty = bar_full + 8 * kGemvMaxSlots;
    auto full = [&](int s) { return bar_full + 8u * s; };
    auto empty = [&](int s) { return bar_empty + 8u * s; };
    float* red = reinterpret_cast<float*>(smem + geo.ring_bytes + x_bytes + 16 * kGemvMaxSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + kGemvWarps * 2 * kGemvWarps * RP);
    // the row block of each slot (first row; rows, 0 = no more work)
    int* slot_row0 = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(red + kGemvWarps * 2 * kGemvWarps * RP) + 16);
    int* slot_rows = slot_row0 + kGemvMaxSlots;
    const uint32_t resp0 = smem_u32(slot_rows + kGemvMaxSlots);  // 16-byte aligned (see the layout sizes)
    auto resp = [&](int i) { return resp0 + 16u * i; };
    auto cbar = [&](int i) { return resp0 + 32u + 8u * i; };
    const int G = geo.g, groups = kGemvWarps / G;
    const uint32_t sring = ring + static_cast<uint32_t>(S) * geo.slot_bytes;  // group scale slots

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kGemvWarps) {
        for (int i = lane; i < S; i += 32) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), kGemvWarps);  // one arrival per compute warp
        }
        if (lane < 2) mbar_init(cbar(lane), 1);
        if (lane == 0) *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the next kernel in the stream may start its set-up; it waits for this
    // grid before touching global memory
    pdl_launch_dependents();

    if (warp == kGemvWarps) {
        // ---------------------------------------------------- producer --
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // the codes (and group scales) may come from the previous kernel,
            // unless the caller states that they were complete before it
            if (!geo.early) pdl_wait();
            bool waited = !geo.early;
            // Work: the row blocks of R rows, one per CTA of the grid.  This
            // CTA does its own block, then cancels CTAs that have not started
            // yet and does theirs (one request in flight at a time, answers
            // alternating between two buffers), so SMs that free up early take
            // more of the weight and the launch ends evenly.  It asks only
            // once the previous grid is done: a CTA that starts early (while
            // the previous kernel drains) would otherwise take over blocks it
            // cannot compute yet, which CTAs starting later would have done.
            int64_t blk = blockIdx.x;
            int nreq = 0;             // cancel requests issued
            bool pending = false;     // one is in flight
            auto request = [&]() {
                mbar_arrive_expect_tx(cbar(nreq & 1), 16u);
                cancel_request(resp(nreq & 1), cbar(nreq & 1));
                ++nreq;
                pending = true;
            };
            int64_t issued = 0;
            int s = 0;
            uint32_t ph = 0;
            for (;;) {
                if (!mbar_wait(empty(s), ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    atomicCAS(&g_gemv_error, 0, kErrWaitSlot);
                    break;
                }
                if (blk < 0) {
                    // no block left: the compute warps stop at this slot
                    slot_rows[s] = 0;
                    mbar_arrive(full(s));
                    break;
                }
                const int64_t r0 = blk * R;
                const int64_t rows = (n - r0) < R ? (n - r0) : R;
                slot_row0[s] = static_cast<int>(r0);
                slot_rows[s] = static_cast<int>(rows);
                const uint32_t bytes = static_cast<uint32_t>(rows * k);
                if constexpr (kGrouped) {
                    const uint32_t sbytes = static_cast<uint32_t>(rows * geo.ngroups * kScaleBytes);
                    mbar_arrive_expect_tx(full(s), bytes + sbytes);
                    bulk_load(sring + s * geo.sslot_bytes,
                              reinterpret_cast<const uint8_t*>(scales) + r0 * geo.ngroups * kScaleBytes, sbytes,
                              full(s), pol);
                } else {
                    mbar_arrive_expect_tx(full(s), bytes);
                }
                bulk_load(ring + s * geo.slot_bytes, codes + r0 * k, bytes, full(s), pol);
                ++issued;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
                if (!waited) {
                    pdl_wait();
                    waited = true;
                }
                if (nreq == 0) request();
                // the next block: the answer to the request in flight
                blk = -1;
                if (pending) {
                    const int q = nreq - 1;
                    if (!mbar_wait(cbar(q & 1), static_cast<uint32_t>((q >> 1) & 1), abort_flag)) {
                        *abort_flag = 1;
                        atomicCAS(&g_gemv_error, 0, kErrWaitSlot);
                        break;
                    }
                    pending = false;
                    blk = cancel_answer(resp(q & 1));
                    if (blk >= 0) request();
                }
            }
            if (*abort_flag) {
                // let the copies and the cancel answer in flight land before the CTA exits
                for (int64_t j = (issued > S ? issued - S : 0); j < issued; ++j)
                    if (!mbar_wait_drain(full(static_cast<int>(j % S)), static_cast<uint32_t>((j / S) & 1)))
                        atomicCAS(&g_gemv_error, 0, kErrWaitDrain);
                if (pending && !mbar_wait_drain(cbar((nreq - 1) & 1), static_cast<uint32_t>(((nreq - 1) >> 1) & 1)))
                    atomicCAS(&g_gemv_error, 0, kErrWaitDrain);
            }
        }
        return;
    }

    // -------------------------------------------------------- compute --
    pdl_wait();  // x, scales and bias may come from the previous kernel, y may still be read by it
    const int64_t nchunks = k >> 4;
    // x is staged piece-major: the j-th 16-byte piece of every 16-activation
    // chunk together, so the 32 lanes (32 consecutive chunks) read 32
    // consecutive pieces, free of bank conflicts
    {
        const uint4* xg = reinterpret_cast<const uint4*>(x);
        uint4* xd = reinterpret_cast<uint4*>(xs);
        for (int64_t i = threadIdx.x; i < nchunks * 2; i += 32 * kGemvWarps) {
            const uint4 v = __ldg(xg + i);
            if constexpr (kF32X) {
                // 8 activations -> 8 fp32
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                float f[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (kBf16) {
                        f[2 * e] = bf16_lo_to_f32(wv[e]);
                        f[2 * e + 1] = bf16_hi_to_f32(wv[e]);
                    } else {
                        f16x2_to_f32x2(wv[e], f[2 * e], f[2 * e + 1]);
                    }
                }
                // half h of chunk ch holds pieces 2h and 2h+1
                const int64_t ch = i >> 1, pc = 2 * (i & 1);
                xd[pc * nchunks + ch] =
                    make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
                xd[(pc + 1) * nchunks + ch] =
                    make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]), __float_as_uint(f[7]));
            } else {
                xd[(i & 1) * nchunks + (i >> 1)] = v;
            }
        }
    }
    // the staged x is visible to every compute warp
    asm volatile("bar.sync %0, %1;" ::"n"(15), "n"(32 * kGemvWarps) : "memory");  // ids 1..8: row groups

    const uint32_t xv = smem_u32(xs);
    const uint32_t xpiece = static_cast<uint32_t>(nchunks * 16);  // bytes from one piece of x to the next
    const int grp = warp / G, wg = warp % G;
    int s = 0;
    uint32_t ph = 0;
    int parity = 0;
    for (int64_t sl = 0;; ++sl) {
        bool ok = mbar_wait_warp(full(s), ph, abort_flag);
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicCAS(&g_gemv_error, 0, kErrWaitTma);
        }
        // a group of several warps leaves together, so none is left waiting
        // at the group's barrier below
        if (G > 1) ok = !bar_red_or(1 + grp, 32 * G, !ok);
        if (!ok) break;
        // the slot's row block (no rows: no more work)
        const int rows = slot_rows[s];
        if (rows == 0) break;
        const int64_t row0 = slot_row0[s];
        // items of RP consecutive rows, item index (sl * R / RP + r / RP)
        // dealt round-robin: this group takes the items with index % groups
        // == grp
        const int64_t gbase = sl * R / RP;
        for (int r = static_cast<int>((grp - gbase % groups + groups) % groups) * RP; r < rows; r += groups * RP) {
            const int nr = rows - r < RP ? rows - r : RP;  // rows in this item (the slot's last may be short)
            const uint32_t rowp = ring + s * geo.slot_bytes + static_cast<uint32_t>(r * k);
            // per-group scales of the item's rows
            const uint8_t* gsb = smem + (sring - ring) + s * geo.sslot_bytes +
                                 static_cast<int64_t>(r) * geo.ngroups * kScaleBytes;
            uint64_t acc[RP];
#pragma unroll
            for (int q = 0; q < RP; ++q) acc[q] = 0ull;
            const int nch = static_cast<int>(nchunks);
            const uint32_t kk = static_cast<uint32_t>(k);
#pragma unroll 4
            for (int ch = wg * 32 + lane; ch < nch; ch += 32 * G) {
                uint4 cw[RP];
#pragma unroll
                for (int q = 0; q < RP; ++q)
                    cw[q] = q < nr ? lds128(rowp + q * kk + static_cast<uint32_t>(ch) * 16u)
                                   : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t xa = xv + static_cast<uint32_t>(ch) * 16u;
                uint64_t part[RP];
#pragma unroll
                for (int q = 0; q < RP; ++q) part[q] = 0ull;
                uint64_t (&dst)[RP] = kGrouped ? part : acc;
                if constexpr (kF32X) {
                    const uint4 xf[4] = {lds128(xa), lds128(xa + xpiece), lds128(xa + 2 * xpiece),
                                         lds128(xa + 3 * xpiece)};
                    dot_chunk_f32<RP>(cw, xf, dst);
                } else {
                    dot_chunk<RP, kBf16>(cw, lds128(xa), lds128(xa + xpiece), dst);
                }
                if constexpr (kGrouped) {
#pragma unroll
                    for (int q = 0; q < RP; ++q) {
                        const int gi = q * geo.ngroups + (ch >> geo.gshift);
                        float g;
                        if constexpr (kE8) {
                            // 2^(b - 127) is the fp32 pattern b << 23, except b = 0
                            // (the subnormal 2^-127, 0x00400000) and b = 0xFF (NaN,
                            // 0x7FC00000): both gain the bit 0x00400000, and they are
                            // the two bytes with (b + 1) & 0xFE == 0
                            const uint32_t b = gsb[gi];
                            g = __uint_as_float((b << 23) | (((b + 1u) & 0xFEu) == 0u ? 0x00400000u : 0u));
                        } else {
                            g = reinterpret_cast<const float*>(gsb)[gi];
                        }
                        ffma2(acc[q], part[q], pack2(g, g));
                    }
                }
            }
            float sum[RP];
#pragma unroll
            for (int q = 0; q < RP; ++q) {
                sum[q] = __uint_as_float(static_cast<uint32_t>(acc[q])) + __uint_as_float(static_cast<uint32_t>(acc[q] >> 32));
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) sum[q] += __shfl_xor_sync(0xffffffffu, sum[q], off);
            }
            if (G > 1) {
                // the group's warps add their sums in a fixed order
                float* rd = red + ((grp * 2 + parity) * kGemvWarps) * RP;
                if (lane == 0)
#pragma unroll
                    for (int q = 0; q < RP; ++q) rd[wg * RP + q] = sum[q];
                asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(32 * G) : "memory");
                if (wg == 0 && lane == 0)
#pragma unroll
                    for (int q = 0; q < RP; ++q) {
                        float t = 0.0f;
                        for (int w2 = 0; w2 < G; ++w2) t += rd[w2 * RP + q];
                        sum[q] = t;
                    }
                // the other parity's sums are rewritten only after the next
                // item's barrier, which warp 0 reaches after reading these
                parity ^= 1;
            }
            if (wg == 0 && lane == 0)
#pragma unroll
                for (int q = 0; q < RP; ++q) {
                    if (q >= nr) break;
                    const int64_t i = row0 + r + q;
                    const float bi = bias ? bias[i] : 0.0f;
                    if constexpr (kGrouped) {
                        y[i] = round_out<kBf16>(sum[q] + bi);  // the scales are applied already
                    } else {
                        y[i] = round_out<kBf16>(fmaf(sum[q], scales[i], bi));
                    }
                }
        }
        // this warp has read its rows of the slot
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// Shared memory beside the ring: x, the slot barriers, the row groups'
// partial sums, the abort flag (16), the slots' row blocks (8 per slot), two
// cancel answers (16 each) and their barriers (8 each), and 128 of slack
// for the alignment of the base.
static uint32_t gemv_fixed_bytes(int64_t k, bool f32x) {
    return static_cast<uint32_t>(((k * (f32x ? 4 : 2) + 127) / 128) * 128) + 16 * kGemvMaxSlots +
           4 * kGemvWarps * 2 * kGemvWarps * 2 + 16 + 8 * kGemvMaxSlots + 32 + 16 + 128;
}

template <bool kBf16>
static cudaError_t launch_dt(const LinearArgs& a, cudaStream_t st) {
    const bool grouped = a.group > 0;
    const int sbytes = a.e8m0 ? 1 : 4;
    int sms = 0;
    cudaError_t e = device_sm_count(sms);
    if (e != cudaSuccess) return e;
    if (a.k > kGemvMaxK) return cudaErrorNotSupported;
    GemvGeom geo;
    // a slot holds one row block: whole rows, up to kGemvSlotTarget bytes,
    // and no more than the rows an SM would get if every SM took the same
    // share (so that small matrices still spread over the GPU); rows are
    // computed in pairs, so blocks hold an even number (x is staged as fp32
    // for rows up to 8192 codes, as 16-bit values beyond).  The grid has one
    // CTA per block; running CTAs take over the blocks of CTAs that have not
    // started (cluster launch control).
    const int rp = 2;
    const bool f32x = a.k <= 8192;
    int64_t rows = kGemvSlotTarget / a.k;
    const int64_t share = (a.n + sms - 1) / sms;
    if (rows > share) rows = share + (share & 1);
    rows -= rows % rp;
    if (rows < rp) rows = rp;
    const int64_t grid = (a.n + rows - 1) / rows;
    geo.rows = static_cast<int>(rows);
    geo.slot_bytes = static_cast<uint32_t>(((rows * a.k + 127) / 128) * 128);
    // per-group scales: a slot's rows of scales beside its codes
    geo.ngroups = grouped ? static_cast<int>(a.k / a.group) : 0;
    geo.gshift = 0;
    while (grouped && (16 << geo.gshift) < a.group) ++geo.gshift;
    geo.sslot_bytes = static_cast<uint32_t>(((rows * geo.ngroups * sbytes + 127) / 128) * 128);
    int64_t slots = (kGemvSmemBudget - gemv_fixed_bytes(a.k, f32x)) / (geo.slot_bytes + geo.sslot_bytes);
    if (slots > kGemvMaxSlots) slots = kGemvMaxSlots;
    if (slots < 2) return cudaErrorNotSupported;
    geo.slots = static_cast<int>(slots);
    geo.ring_bytes = geo.slots * (geo.slot_bytes + geo.sslot_bytes);
    // warps per row group: enough that two slots' items keep all warps busy
    const int64_t items = (rows + rp - 1) / rp;
    geo.g = 1;
    while (geo.g < kGemvWarps && items * geo.g * 2 < kGemvWarps) geo.g *= 2;
    geo.early = a.early ? 1 : 0;
    const uint32_t smem = geo.ring_bytes + gemv_fixed_bytes(a.k, f32x);

    const int kind = !grouped ? 0 : a.e8m0 ? 2 : 1;
    decltype(&gemv_kernel<2, kBf16, false, 0>) all[6] = {
        gemv_kernel<2, kBf16, false, 0>, gemv_kernel<2, kBf16, true, 0>, gemv_kernel<2, kBf16, false, 1>,
        gemv_kernel<2, kBf16, true, 1>,  gemv_kernel<2, kBf16, false, 2>, gemv_kernel<2, kBf16, true, 2>};
    auto kern = all[2 * kind + (f32x ? 1 : 0)];
    static std::once_flag attr_once[64];
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        for (auto f : all)
            if (attr_err == cudaSuccess)
                attr_err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmemBudget);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // programmatic dependent launch: set-up overlaps the previous kernel's tail
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint16_t*>(a.x), a.codes, a.scales, a.bias,
                              static_cast<uint16_t*>(a.y), a.n, a.k, geo);
}

bool gemv_supports(int64_t k) { return k <= kGemvMaxK; }

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
