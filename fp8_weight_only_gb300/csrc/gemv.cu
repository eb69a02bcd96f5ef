// gemv.cu -- kernel K2: the M = 1 linear layer (GEMV) on CUDA cores.
//
// Page "kadirnar/kernel-agent fp8-weights", section "Dequantise in
// registers": the codes are streamed once past L1, converted in registers
// (exactly), multiplied by x with fp32 accumulation, reduced across a warp
// with shuffles, and scale (and bias) are applied once per output in the
// epilogue.
//
// GB300 layout of the work:
//  * Persistent grid, one CTA per SM; CTA c owns the contiguous rows
//    [c*N/P, (c+1)*N/P), so every SM streams the same bytes (+-1 row).
//  * The last warp moves a slot of R whole rows (R*K contiguous bytes, up
//    to 64 KB) per 1-D TMA bulk copy into a ring of slots.  A bulk copy costs
//    the SM's TMA unit a fixed ~0.27 us whatever its size (measured: 4 KB
//    copies stream 15 GB/s per SM, 64 KB copies 218 GB/s), so copies are
//    large.
//  * The CTA's rows are dealt round-robin to the 16 compute warps; a warp
//    computes its row whole (lane l takes 16-code chunks l, l+32, ...), so
//    no reduction crosses warps.  Every warp waits for every slot in order
//    and arrives once on its "empty" barrier after its rows there (none, if
//    the slot has fewer rows than warps): a warp whose next row lay several
//    slots ahead would otherwise wait on a slot a full ring cycle early and
//    pass on the previous phase of the same parity.
//  * x is staged once in shared memory (as 16-bit values), and so are the
//    CTA's scales and bias: after start-up the codes are the only stream.
//  * Codes are converted exactly by the hardware e4m3x2 -> f16x2 conversion
//    and widened to fp32, x is widened from its 16-bit pair, and each product
//    is an fp32 FMA.
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
constexpr int kGemvStagedRows = 2048;                // rows whose scale and bias are staged
constexpr uint32_t kGemvSmemBudget = 224 * 1024;
// Largest K the GEMV takes: x (2 bytes a value) and two 64 KB slots fit
// beside the staged scales.
constexpr int64_t kGemvMaxK = 32768;

struct GemvGeom {
    int rows;         // rows per slot (R)
    int slots;        // slots in the ring (S)
    uint32_t slot_bytes;
    uint32_t ring_bytes;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// f16x2 -> two fp32 (the halves selected in the register, no extraction).
__device__ __forceinline__ void f16x2_to_f32x2(uint32_t h, float& lo, float& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
}

// One 16-code chunk against its 16 activations (8 packed 16-bit pairs),
// into two accumulators for instruction-level parallelism.
template <bool kBf16>
__device__ __forceinline__ void dot_chunk(const uint4 c, const uint4 xa, const uint4 xb, float& a0, float& a1) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h01, h23;
        e4m3x4_to_f16x2(w[q], h01, h23);
        float v0, v1, v2, v3;
        f16x2_to_f32x2(h01, v0, v1);
        f16x2_to_f32x2(h23, v2, v3);
        float x0, x1, x2, x3;
        if constexpr (kBf16) {
            x0 = bf16_lo_to_f32(xw[2 * q]);
            x1 = bf16_hi_to_f32(xw[2 * q]);
            x2 = bf16_lo_to_f32(xw[2 * q + 1]);
            x3 = bf16_hi_to_f32(xw[2 * q + 1]);
        } else {
            f16x2_to_f32x2(xw[2 * q], x0, x1);
            f16x2_to_f32x2(xw[2 * q + 1], x2, x3);
        }
        a0 = fmaf(x0, v0, a0);
        a1 = fmaf(x1, v1, a1);
        a0 = fmaf(x2, v2, a0);
        a1 = fmaf(x3, v3, a1);
    }
}

template <bool kBf16>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                const float* __restrict__ bias, uint16_t* __restrict__ y, int64_t n, int64_t k, GemvGeom geo) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t ring = smem_u32(smem);
    const int S = geo.slots, R = geo.rows;
    // layout: ring | x [k] | scales, bias [kGemvStagedRows] | full, empty [kGemvMaxSlots] | abort flag
    const uint32_t x_bytes = static_cast<uint32_t>(((k * 2 + 127) / 128) * 128);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + geo.ring_bytes);
    float* sc_s = reinterpret_cast<float*>(smem + geo.ring_bytes + x_bytes);
    float* bi_s = sc_s + kGemvStagedRows;
    const uint32_t bar_full = smem_u32(bi_s + kGemvStagedRows);
    const uint32_t bar_empty = bar_full + 8 * kGemvMaxSlots;
    auto full = [&](int s) { return bar_full + 8u * s; };
    auto empty = [&](int s) { return bar_empty + 8u * s; };
    volatile int* abort_flag =
        reinterpret_cast<volatile int*>(smem + geo.ring_bytes + x_bytes + 8 * kGemvStagedRows + 16 * kGemvMaxSlots);

    const int64_t P = gridDim.x;
    const int64_t row0 = blockIdx.x * n / P, row1 = (blockIdx.x + 1) * n / P;
    const int64_t nrows = row1 - row0;
    const int64_t nslots = (nrows + R - 1) / R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kGemvWarps) {
        for (int i = lane; i < S; i += 32) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), kGemvWarps);  // one arrival per compute warp
        }
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
            pdl_wait();  // the codes may come from the previous kernel
            int64_t issued = 0;
            int s = 0;
            uint32_t ph = 0;
            for (int64_t sl = 0; sl < nslots; ++sl) {
                if (!mbar_wait(empty(s), ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    atomicCAS(&g_gemv_error, 0, kErrWaitSlot);
                    break;
                }
                const int64_t r0 = row0 + sl * R;
                const int64_t rows = (row1 - r0) < R ? (row1 - r0) : R;
                const uint32_t bytes = static_cast<uint32_t>(rows * k);
                mbar_arrive_expect_tx(full(s), bytes);
                bulk_load(ring + s * geo.slot_bytes, codes + r0 * k, bytes, full(s), pol);
                ++issued;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag) {
                // let the copies in flight land before the CTA exits
                for (int64_t j = (issued > S ? issued - S : 0); j < issued; ++j)
                    if (!mbar_wait_drain(full(static_cast<int>(j % S)), static_cast<uint32_t>((j / S) & 1)))
                        atomicCAS(&g_gemv_error, 0, kErrWaitDrain);
            }
        }
        return;
    }

    // -------------------------------------------------------- compute --
    pdl_wait();  // x, scales and bias may come from the previous kernel, y may still be read by it
    const int64_t nchunks = k >> 4;
    {
        const uint4* xg = reinterpret_cast<const uint4*>(x);
        uint4* xd = reinterpret_cast<uint4*>(xs);
        for (int64_t i = threadIdx.x; i < nchunks * 2; i += 32 * kGemvWarps) xd[i] = __ldg(xg + i);
    }
    const bool staged = nrows <= kGemvStagedRows;
    if (staged) {
        for (int64_t i = threadIdx.x; i < nrows; i += 32 * kGemvWarps) {
            sc_s[i] = scales[row0 + i];
            bi_s[i] = bias ? bias[row0 + i] : 0.0f;
        }
    }
    // the staged x, scales and bias are visible to every compute warp
    asm volatile("bar.sync %0, %1;" ::"n"(1), "n"(32 * kGemvWarps) : "memory");

    const uint4* xv = reinterpret_cast<const uint4*>(xs);
    int s = 0;
    uint32_t ph = 0;
    for (int64_t sl = 0; sl < nslots; ++sl) {
        if (!mbar_wait_warp(full(s), ph, abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1;
                atomicCAS(&g_gemv_error, 0, kErrWaitTma);
            }
            break;
        }
        const int64_t base = sl * R;  // CTA-local index of the slot's first row
        const int rows = static_cast<int>((nrows - base) < R ? (nrows - base) : R);
        // rows i = base + r with i % kGemvWarps == warp
        for (int r = static_cast<int>((warp - base % kGemvWarps + kGemvWarps) % kGemvWarps); r < rows;
             r += kGemvWarps) {
            const int64_t i = base + r;
            const int64_t row = row0 + i;
            float sc = 0.0f, bi = 0.0f;
            if (lane == 0) {
                if (staged) {
                    sc = sc_s[i];
                    bi = bi_s[i];
                } else {
                    sc = scales[row];
                    bi = bias ? bias[row] : 0.0f;
                }
            }
            const uint8_t* rowp = smem + s * geo.slot_bytes + static_cast<int64_t>(r) * k;
            float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 4
            for (int64_t ch = lane; ch < nchunks; ch += 32)
                dot_chunk<kBf16>(*reinterpret_cast<const uint4*>(rowp + ch * 16), xv[2 * ch], xv[2 * ch + 1], a0, a1);
            float acc = a0 + a1;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) y[row] = round_out<kBf16>(fmaf(acc, sc, bi));
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

static uint32_t gemv_fixed_bytes(int64_t k) {
    return static_cast<uint32_t>(((k * 2 + 127) / 128) * 128) + 8 * kGemvStagedRows + 16 * kGemvMaxSlots + 16 + 128;
}

template <bool kBf16>
static cudaError_t launch_dt(const LinearArgs& a, cudaStream_t st) {
    int sms = 0;
    cudaError_t e = device_sm_count(sms);
    if (e != cudaSuccess) return e;
    if (a.k > kGemvMaxK) return cudaErrorNotSupported;
    GemvGeom geo;
    // a slot holds whole rows, up to kGemvSlotTarget bytes
    int64_t rows = kGemvSlotTarget / a.k;
    if (rows < 1) rows = 1;
    geo.rows = static_cast<int>(rows);
    geo.slot_bytes = static_cast<uint32_t>(((rows * a.k + 127) / 128) * 128);
    int64_t slots = (kGemvSmemBudget - gemv_fixed_bytes(a.k)) / geo.slot_bytes;
    if (slots > kGemvMaxSlots) slots = kGemvMaxSlots;
    if (slots < 2) return cudaErrorNotSupported;
    geo.slots = static_cast<int>(slots);
    geo.ring_bytes = geo.slots * geo.slot_bytes;
    const uint32_t smem = geo.ring_bytes + gemv_fixed_bytes(a.k);

    auto kern = gemv_kernel<kBf16>;
    static std::once_flag attr_once[64];
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmemBudget);
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
