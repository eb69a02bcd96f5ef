// fp8w_internal.h -- launch functions shared between the kernels' translation
// units and the C ABI layer (api.cu).  Host-side only.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8w {

struct LinearArgs {
    const void* x;
    int act;  // FP8W_BF16 / FP8W_F16
    int64_t m, k, n;
    const uint8_t* codes;
    const float* scales;
    const float* bias;  // may be null
    void* y;
    int64_t group = 0;  // 0: scales[n]; else scales[n, k / group]
    bool e8m0 = false;  // with group 32: scales are E8M0 bytes, not fp32
    bool early = false; // the weights were complete before the preceding kernel
                        // started: their copies may begin before it finishes
};

// K1: codes/scales from fp32 weights.
cudaError_t launch_quantize(const float* w, int64_t n, int64_t k, uint8_t* codes, float* scales,
                            cudaStream_t st);

// K1 for 16-bit weights (bf16 or fp16), widened exactly to fp32.
cudaError_t launch_quantize_16(const uint16_t* w, bool bf16, int64_t n, int64_t k, uint8_t* codes, float* scales,
                               cudaStream_t st);

// Per-group scales: scales[n, k / group], group 32, 64 or 128, k % group == 0.
cudaError_t launch_quantize_grouped(const float* w, int64_t n, int64_t k, int group, uint8_t* codes, float* scales,
                                    cudaStream_t st);

// MX-style: codes and E8M0 scales[n, k / 32], k % 32 == 0.
cudaError_t launch_quantize_mx(const float* w, int64_t n, int64_t k, uint8_t* codes, uint8_t* scales,
                               cudaStream_t st);

// The dequantised weight, rounded once to fp32 (out_dtype 0), bf16 (1) or fp16 (2).
cudaError_t launch_dequantize(const uint8_t* codes, const float* scales, int64_t n, int64_t k, int out_dtype,
                              void* w, cudaStream_t st);

// The same with per-group scales: fp32 scales[n, k / group] (group 32, 64 or
// 128), or E8M0 bytes[n, k / 32] (e8m0, group 32).
cudaError_t launch_dequantize_grouped(const uint8_t* codes, const void* scales, bool e8m0, int group, int64_t n,
                                      int64_t k, int out_dtype, void* w, cudaStream_t st);

// K2: m == 1, k <= 32768 (gemv_supports).
cudaError_t launch_gemv(const LinearArgs& a, cudaStream_t st);
bool gemv_supports(int64_t k);

// K3: any m (16-, 32- or 64-token launches, 64-row slabs beyond; the
// per-group form 16 or 32, 32-row slabs beyond); no workspace.  Launch shape: clusters of `cl` CTAs (1..16), each taking `tpc`
// consecutive 128-channel tiles; forced == nullptr picks it from the shape.
struct SkinnyShape {
    int cl;
    int64_t tpc;
};
cudaError_t launch_skinny(const LinearArgs& a, const SkinnyShape* forced, cudaStream_t st);
// grouped: the per-group form (a CTA shares at most one tile)
SkinnyShape skinny_shape(int64_t n, int64_t k, const int* active, int nt, bool grouped = false);
bool skinny_shape_valid(const SkinnyShape& sh, int64_t m, int64_t k, bool grouped = false);
cudaError_t device_sm_count(int& sms);
// 2-D tiled tensor map with 128-byte swizzle: `inner` x `outer` elements,
// rows of `row_bytes`, boxes of box_inner x box_outer.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// 3-D tensor map over a [rows, k] byte matrix (k % 128 == 0) seen as
// (128 bytes of a k-block, row, k-block), 128-byte swizzle: a box of
// box_rows rows and box_blocks consecutive k-blocks lands as box_blocks
// tiles of box_rows x 128 bytes, one after the other.
bool encode_3d_blocks(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k, uint32_t box_rows,
                      uint32_t box_blocks);

// K4: m > 64 (prefill shapes), per-row scales; one launch, no workspace.
cudaError_t launch_prefill(const LinearArgs& a, cudaStream_t st);
int read_prefill_device_error();

// K5: W8A8, e4m3 activation codes x_codes[m, k] with per-token scales
// x_scales[m] times e4m3 weight codes w_codes[n, k] with per-channel scales
// w_scales[n]; y[m, n] in bf16 (out 1) or fp16 (out 2).  early: the weights
// were complete before the preceding kernel started (their copies may begin
// before it finishes).
struct W8A8Args {
    const uint8_t* x_codes;
    const float* x_scales;
    int64_t m, k, n;
    const uint8_t* w_codes;
    const float* w_scales;
    const float* bias;  // may be null
    void* y;
    int out;
    bool early;
};
cudaError_t launch_w8a8(const W8A8Args& a, cudaStream_t st);
int read_w8a8_device_error();

// Kernel-recorded wait failures (0 = none); reading clears them.
int read_skinny_device_error();
int read_gemv_device_error();

}  // namespace fp8w
