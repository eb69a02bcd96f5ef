// fp8w_device.cuh -- device-side building blocks shared by the libfp8w kernels
// (sm_103a only): streaming loads, e4m3 decoding, mbarrier waits with a time
// limit, TMA tensor loads, tcgen05 (TMEM / tensor core) wrappers and cluster
// shared-memory access.  Every wrapper is a single PTX instruction or a short
// fixed sequence written out here.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "libfp8w is built for sm_103a only"
#endif

namespace fp8w {

// Bounded waits: a wait that has not succeeded after this many SM cycles
// (about 2 s at 2 GHz) gives up, records an error code and lets the kernel
// wind down instead of hanging.  Measured on the SM's own cycle counter,
// which only moves forward with the SM clock.
constexpr long long kWaitLimitCycles = 4000000000ll;

enum DeviceError : int {
    kErrNone = 0,
    kErrWaitTma = 1,      // consumer gave up waiting for a TMA stage
    kErrWaitMma = 2,      // waiting for tensor-core completion
    kErrWaitDequant = 3,  // MMA issuer gave up waiting for a dequantised stage
    kErrWaitSlot = 4,     // producer gave up waiting for a free stage
    kErrWaitDrain = 5     // giving up on in-flight copies at exit
};

// ---------------------------------------------------------------- loads --

// 16 bytes, read-only, not kept in L1 (the codes are streamed exactly once).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ldg_stream_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ long long cycles() { return clock64(); }

// ------------------------------------------------------------ e4m3 codec --

// Two e4m3 codes (low byte = first) -> f16x2 (first code in the low half),
// hardware conversion, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
    return h;
}

// Four codes (byte i = code i) -> two f16x2 words (codes 0,1 and 2,3).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& p01, uint32_t& p23) {
    p01 = e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xFFFFu));
    p23 = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
}

// Four codes (byte i = code i) -> two bf16x2 words, exact, by integer moves:
// the byte S.EEEE.MMM is laid out as the bf16 pattern S.0000EEEE.MMM0000,
// whose value is the e4m3 value times 2^-120 (e4m3 subnormals become bf16
// subnormals), then one packed bf16 multiply by 2^120 restores the value.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

constexpr uint32_t kBf16x2Pow2_120 = 0x7B807B80u;  // bf16 2^120 in both halves

// Four e4m3 codes -> their values times mul / 2^120 as bf16 pairs: the byte
// moves place the code's exponent and mantissa bits in a bf16, which reads
// as value * 2^-120 exactly (e4m3 subnormals become bf16 subnormals); one
// bf16 multiply by mul (2^120 restores the value) rounds the product once.
__device__ __forceinline__ void e4m3x4_to_bf16x2_mul(uint32_t w, uint32_t& p01, uint32_t& p23, uint32_t mul) {
    const uint32_t lo = (w << 4) & 0xF0F0F0F0u;                         // E0 M2 M1 M0 0000
    const uint32_t hi = ((w >> 4) & 0x07070707u) | (w & 0x80808080u);  // S 0000 E3 E2 E1
    p01 = bf16x2_mul(__byte_perm(lo, hi, 0x5140), mul);
    p23 = bf16x2_mul(__byte_perm(lo, hi, 0x7362), mul);
}

// MX-style scales folded into a dequantised bf16 weight: an E8M0 byte b is
// worth 2^e, e = b - 127.  With the byte moves above (value * 2^-120), one
// multiply by 2^(120 + e) gives value * 2^e rounded once; that multiplier is
// a bf16 number for b <= 134.  Larger bytes take 2^120 first and then this
// second factor, 2^e itself as bf16 pairs (b = 0: the subnormal 2^-127; 0xFF:
// NaN), which rounds the same product once.
__device__ __forceinline__ uint32_t mx_first_mul(uint32_t b) {
    const uint32_t h = (b + 120u) << 7;
    return h | (h << 16);
}
__device__ __forceinline__ uint32_t mx_second_mul(uint32_t b) {
    const uint32_t h = b == 255u ? 0x7FC0u : b == 0u ? 0x0040u : b << 7;
    return h | (h << 16);
}

__device__ __forceinline__ void e4m3x4_to_bf16x2(uint32_t w, uint32_t& p01, uint32_t& p23) {
    e4m3x4_to_bf16x2_mul(w, p01, p23, kBf16x2Pow2_120);
}

// Two fp32 values -> two saturating, round-to-nearest-even e4m3 codes
// (first argument in the low byte).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float first, float second) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
    return r;
}

__device__ __forceinline__ float f16_lo_to_f32(uint32_t h2) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi_to_f32(uint32_t h2) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}
__device__ __forceinline__ float bf16_lo_to_f32(uint32_t b2) { return __uint_as_float(b2 << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t b2) { return __uint_as_float(b2 & 0xFFFF0000u); }

// ------------------------------------------------------------- mbarrier --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the same condition (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if the
// CTA-wide abort flag is raised meanwhile or the time limit passes.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = cycles();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (cycles() - t0 > kWaitLimitCycles) return false;
        }
    }
}

// Wait with a time limit only (used while winding down after an abort).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const long long t0 = cycles();
    while (!mbar_try_wait(bar, parity)) {
        if (cycles() - t0 > kWaitLimitCycles) return false;
    }
    return true;
}

// Warp-uniform wait: every lane waits, and the warp proceeds only if all
// lanes saw the phase complete (so warp-collective instructions that follow
// are never reached by part of a warp).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
    const bool ok = mbar_wait(bar, parity, abort_flag);
    return __all_sync(0xffffffffu, ok);
}

// Named barrier `id` over `count` threads that also returns, to every
// participant, whether any of them passed `pred` = true (a group-uniform
// decision, e.g. to leave a loop together).
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Strong gpu-scope load with acquire semantics (a flag published by another CTA).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// 16-byte shared-memory load by 32-bit shared address (a plain pointer into
// dynamic shared memory can be compiled to a generic load, which goes
// through the L1/texture path and waits like a global one).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// ------------------------------------------------------------------ TMA --

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at (x = inner coordinate, y = row) into shared
// memory; completion is counted in bytes on `bar`.  `policy` is an L2 cache
// policy from createpolicy.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// The same for a 3-D tensor map (x innermost).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// -------------------------------------------------------------- tcgen05 --

// TMEM allocation (executed by one full warp): writes the base address to
// shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The scale forms of the tensor-core kernels: one fp32 scale a row; E8M0
// bytes per 32 codes folded into the dequantised bf16 weight; per-group
// scales (fp32, or E8M0 bytes) applied to each group's own accumulator.
constexpr int kModeRow = 0, kModeMxFold = 1, kModeGrouped = 2;

// E8M0 byte -> fp32: 2^(b - 127); 0 is the subnormal 2^-127, 0xFF NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    return b == 0xFFu ? __uint_as_float(0x7FC00000u) : b == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// Two fp32 values in one 64-bit register pair (low word = first).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
// acc2 += a2 * b2, lane-wise on fp32 pairs (one packed FMA, each lane an
// IEEE fma rounded to nearest: the same bits as two fmaf).
__device__ __forceinline__ void ffma2(uint64_t& acc2, uint64_t a2, uint64_t b2) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2) : "l"(a2), "l"(b2));
}
// tot2[i] += s * (v[2i], v[2i + 1]) for the 16 fp32 values v of a TMEM load.
__device__ __forceinline__ void ffma2_x16(uint64_t* tot2, const uint32_t (&v)[16], uint64_t s2) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        ffma2(tot2[i], static_cast<uint64_t>(v[2 * i]) | (static_cast<uint64_t>(v[2 * i + 1]) << 32), s2);
}

// Each thread of the warp writes 8 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// The same followed by tcgen05.wait::ld in one statement: the registers are
// defined only once the load has landed, so no use of them can be scheduled
// ahead of the wait (a separate wait statement orders memory, not registers).
__device__ __forceinline__ void tmem_ld_x16_sync(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Two such loads in flight, then the wait, in one statement.
__device__ __forceinline__ void tmem_ld2_x16_sync(uint32_t a0, uint32_t a1, uint32_t (&r)[16], uint32_t (&q)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
        "[%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]),
          "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]),
          "=r"(q[14]), "=r"(q[15])
        : "r"(a0), "r"(a1)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: M = 128 rows of A (one per TMEM lane), N
// and the operand types from the instruction descriptor, K = 16.  Issued by
// one thread.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// The same MMA issued by a whole, converged warp: every lane passes the same
// operands and elect.sync picks one lane (always the lowest, lane 0, in a full
// warp) to issue.  Issuing from a converged warp keeps the operands in the
// uniform datapath; a tcgen05.mma issued from a one-lane branch costs its
// thread about three times as long.
__device__ __forceinline__ void mma_f16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem], both operands by descriptor (M = 128, N
// and types from the instruction descriptor, K = 16), issued by one elected
// lane of a converged warp.
__device__ __forceinline__ void mma_f16_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Shared-memory writes of this thread become visible to the async proxy
// (the tensor core's operand reads) once a barrier orders them after this.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// tcgen05.commit from the lane elect.sync picks, i.e. the lane that issued
// the MMAs above (a commit tracks its own thread's operations only).
__device__ __forceinline__ void tc_commit_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand in the
// 128-byte swizzled canonical layout -- rows of 128 bytes, 8-row atoms of
// 1024 bytes (SBO), 16-byte chunk c of row r stored at chunk c ^ (r % 8).
// `addr` is the shared address of the first element used (the atom must be
// 1024-byte aligned; advancing along K inside the atom adds bytes here).
__device__ __forceinline__ uint64_t smem_desc_sw128_kmajor(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);    // start address
    d |= static_cast<uint64_t>(1u) << 16;                  // LBO (unused for swizzled K-major)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;          // SBO: 8 rows x 128 B
    d |= static_cast<uint64_t>(1u) << 46;                  // descriptor version (tcgen05)
    d |= static_cast<uint64_t>(2u) << 61;                  // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, A and B both bf16
// (bf16 = true) or both fp16, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, uint32_t n) {
    return (1u << 4)                          // D format: f32
           | ((bf16 ? 1u : 0u) << 7)          // A format
           | ((bf16 ? 1u : 0u) << 10)         // B format
           | ((n >> 3) << 17)                 // N / 8
           | ((128u >> 4) << 24);             // M / 16
}

// -------------------------------------------------------------- cluster --

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------- programmatic dependent launch --

// Wait until the preceding grid in the stream has completed and its memory
// operations are visible (no-op when launched without the PDL attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid in the stream to begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- epilogue --

template <bool kBf16>
__device__ __forceinline__ uint16_t round_out(float v) {
    if constexpr (kBf16) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    } else {
        return __half_as_ushort(__float2half_rn(v));
    }
}

}  // namespace fp8w
