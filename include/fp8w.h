/*
 * fp8w.h -- C ABI of libfp8w, the FP8 weight-only linear layer for one
 * GB300 (sm_103a).
 *
 * The operation (page "kadirnar/kernel-agent fp8-weights", section "The
 * contract"):
 *
 *   quantise once, per output channel n of a weight W[N,K] (nn.Linear
 *   [out, in], row-major):
 *     scale[n] = amax_k |W[n,k]| / 448          (fp32 division; 1.0 if 0)
 *     q[n,k]   = e4m3( W[n,k] / scale[n] )      (OCP e4m3fn, round to nearest
 *                                                even, saturated to +-448)
 *   then, per call, with activations x[M,K] in bf16 or fp16:
 *     y[m,n]   = round_act( scale[n] * sum_k x[m,k] * q[n,k] + bias[n] )
 *   accumulated in fp32; scale and bias applied in fp32 with one rounding
 *   to the activation dtype.
 *
 * Conventions shared by every entry point:
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The
 *    library allocates no device memory, needs no scratch, keeps no state
 *    between calls, frees nothing and never synchronises: it enqueues
 *    kernels on `stream` (a cudaStream_t; NULL is the legacy default stream)
 *    and returns.  Calls can be captured in a CUDA graph, and calls on
 *    different streams may run at the same time.
 *  - Arguments are checked on the host before any launch; on an error the
 *    outputs are untouched and no work is enqueued.  FP8W_ERR_CUDA means a
 *    CUDA runtime call failed (fp8w_last_cuda_error() names it).  Faults
 *    inside a kernel surface on the caller's next synchronisation.
 *  - A kernel that gives up a bounded wait (it never should) records a
 *    nonzero code that fp8w_device_error() returns.
 *  - On its first use on a device the library sets each kernel's
 *    shared-memory attribute and reads the device's SM count and cluster
 *    capacity, and keeps them for the process (the "state" above is about
 *    calls, not this).  A cudaDeviceReset discards the attributes: a process
 *    that resets the device must not call the library afterwards.
 *  - All matrices are row-major and densely packed (row stride = columns).
 */
#ifndef FP8W_H
#define FP8W_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8W_ABI_VERSION 12

#if defined(__GNUC__)
#define FP8W_API __attribute__((visibility("default")))
#else
#define FP8W_API
#endif

typedef enum fp8w_status {
    FP8W_OK = 0,
    FP8W_ERR_NULL = 1,      /* a required pointer is NULL */
    FP8W_ERR_SHAPE = 2,     /* m, n or k out of range, or k % 16 != 0 */
    FP8W_ERR_ALIGN = 3,     /* a pointer breaks its alignment rule */
    FP8W_ERR_DTYPE = 4,     /* activation dtype is not FP8W_BF16 / FP8W_F16 */
    FP8W_ERR_CUDA = 5,      /* a CUDA runtime/driver call failed */
    FP8W_ERR_CONFIG = 6     /* an explicit launch configuration is invalid */
} fp8w_status;

/* Activation / output dtypes (FP8W_F32: fp8w_dequantize's output and
 * fp8w_quantize_ex's weights only). */
enum { FP8W_BF16 = 1, FP8W_F16 = 2, FP8W_F32 = 3 };

/* Largest supported reduction length and row count. */
#define FP8W_MAX_K 65536
#define FP8W_MAX_DIM 2147483647LL

/*
 * fp8w_quantize -- steps "row amax", "scale" and "encode" of the contract
 * (page "kadirnar/kernel-agent fp8-weights", "The contract"; the saturating
 * conversion is page "tensormux Write an FP8 kernel", step 4).
 *
 *   w      [n, k] fp32, device, 16-byte aligned; values must be finite
 *          (non-finite weights are a precondition violation, not checked).
 *   codes  [n, k] uint8 OCP e4m3fn bytes, device, 16-byte aligned (output).
 *   scales [n] fp32, device, 4-byte aligned (output).
 *   1 <= n <= FP8W_MAX_DIM, 16 <= k <= FP8W_MAX_K, k % 16 == 0.
 *
 * Codes and scales are exact functions of w: scale = fp32(amax / 448), or
 * 1.0 when that quotient is 0; code = nearest-even e4m3 of fp32(w / scale).
 */
FP8W_API fp8w_status fp8w_quantize(const float *w, int64_t n, int64_t k,
                          uint8_t *codes, float *scales, void *stream);

/*
 * fp8w_quantize_ex -- fp8w_quantize for weights stored as fp32, bf16 or fp16
 * (w_dtype FP8W_F32, FP8W_BF16 or FP8W_F16; any other is FP8W_ERR_DTYPE).
 * A 16-bit weight is widened to fp32, which is exact, and then quantised by
 * the same rule, so its codes and scales equal fp8w_quantize's on the
 * widened matrix.  w is [n, k] of w_dtype, device, 16-byte aligned; other
 * arguments and checks as fp8w_quantize.
 */
FP8W_API fp8w_status fp8w_quantize_ex(const void *w, int w_dtype, int64_t n, int64_t k,
                             uint8_t *codes, float *scales, void *stream);

/*
 * fp8w_quantize_grouped -- the quantiser with one scale per run of `group`
 * weights of a row instead of one per row (page "B04 Precision &
 * Quantization", section "Post-training quantization versus
 * quantization-aware training", the granularity table's per-group row).
 *
 *   w      [n, k] fp32, device, 16-byte aligned, finite.
 *   group  32, 64 or 128; k % group == 0.
 *   codes  [n, k] uint8, device, 16-byte aligned (output).
 *   scales [n, k / group] fp32 row-major, device, 4-byte aligned (output).
 *
 * Each group takes fp8w_quantize's rule on its own weights: scale =
 * fp32(amax / 448), 1.0 when that is 0; code = nearest-even e4m3 of the fp32
 * quotient.
 */
FP8W_API fp8w_status fp8w_quantize_grouped(const float *w, int64_t n, int64_t k, int group,
                                  uint8_t *codes, float *scales, void *stream);

/*
 * fp8w_linear_grouped -- fp8w_linear for codes with per-group scales:
 *   y[i, r] = round_act( sum_j scales[r, j] * sum_{c in group j} x[i, c] * e4m3(codes[r, c]) + bias[r] ).
 *
 * group 32, 64 or 128 with k % group == 0; scales [n, k / group] fp32,
 * 16-byte aligned.  Other arguments as fp8w_linear.  fp32 accumulation, each
 * group's partial sum times its scale, bias added once, one rounding:
 *  - m == 1 with k % (4 * group) == 0 and k <= 32768: the GEMV (a slot's
 *    rows of scales are bulk-copied beside its codes; each 16-code partial
 *    sum is scaled by its group's scale);
 *  - otherwise the tensor-core kernels' per-group form (the skinny kernel up
 *    to m = 64 in launches of 16 or 32 tokens, the prefill GEMM beyond):
 *    each group's products go to their own fp32 accumulator in tensor
 *    memory, which is multiplied by the group's scale and added to the
 *    output's fp32 total.
 */
FP8W_API fp8w_status fp8w_linear_grouped(const void *x, int act_dtype, int64_t m, int64_t k,
                                const uint8_t *codes, const float *scales, int group,
                                const float *bias, int64_t n, void *y, void *stream);

/*
 * fp8w_quantize_mx -- the MX-style weight-only quantiser (page "11.
 * Inference with NVFP4/MXFP8", section "MXFP8-Style FP8": e4m3 codes
 * [n, k] and one E8M0 ("f8e8m0fnu") scale byte per 32 codes along k).
 *
 *   w      [n, k] fp32, device, 16-byte aligned; k % 32 == 0.
 *   codes  [n, k] uint8, device, 16-byte aligned (output).
 *   scales [n, k / 32] uint8 row-major, device, any alignment (output).
 *
 * A byte b stands for 2^(b - 127) (0xFF is NaN).  Each block of 32 takes
 * the smallest power of two 2^e >= amax / 448, e clamped to [-127, 127], so
 * its largest weight is never clipped; an all-zero block takes 2^0.  Codes
 * are the nearest-even e4m3 of fp32(w / 2^e).  A block with an infinite
 * weight gets the NaN byte 0xFF and NaN codes (0x7F).
 */
FP8W_API fp8w_status fp8w_quantize_mx(const float *w, int64_t n, int64_t k,
                             uint8_t *codes, uint8_t *scales, void *stream);

/*
 * fp8w_linear_mx -- fp8w_linear for codes with E8M0 scale bytes (group 32):
 *   y[i, r] = round_act( sum_j 2^(scales[r, j] - 127) * sum_{c in block j} x[i, c] * e4m3(codes[r, c]) + bias[r] ).
 *
 *   scales [n, k / 32] uint8, device, 16-byte aligned; k % 128 == 0.
 *   Other arguments as fp8w_linear.
 *
 * m == 1 with k % 512 == 0 and k <= 32768 runs the GEMV: a slot's rows of
 * scale bytes are bulk-copied beside its codes, and each 16-code fp32 partial
 * sum is scaled by its block's power of two, which adds no rounding (short
 * of over- or underflow); bias added once, one rounding.  Any other shape
 * runs a tensor-core kernel (the skinny one up to m = 64, the prefill GEMM
 * beyond).  With bf16 activations the scale is folded into the dequantised
 * bf16 weight, e4m3(q) * 2^(b - 127), which is exact wherever that product
 * is a bf16 number (anything but products below 2^-130 or beyond the bf16
 * range).  With fp16 activations it is fp8w_linear_grouped's per-group form
 * at group 32 with each byte decoded to its fp32 power of two (2^-127 for
 * 0, NaN for 0xFF), which gives the same bits as that call on the decoded
 * scales.  fp32 accumulation, bias added once, one rounding.
 */
FP8W_API fp8w_status fp8w_linear_mx(const void *x, int act_dtype, int64_t m, int64_t k,
                           const uint8_t *codes, const uint8_t *scales,
                           const float *bias, int64_t n, void *y, void *stream);

/*
 * fp8w_dequantize -- the dequantised weight, the pages' fallback form
 * (page "kadirnar/kernel-agent fp8-weights", section "The contract": the
 * codes decoded and multiplied by their row's scale).
 *
 *   codes  [n, k] e4m3 bytes, device, 16-byte aligned.
 *   scales [n] fp32, device, 4-byte aligned.
 *   out_dtype FP8W_F32, FP8W_BF16 or FP8W_F16.
 *   w      [n, k] of out_dtype, device, 16-byte aligned (output).
 *   1 <= n <= FP8W_MAX_DIM, 16 <= k <= FP8W_MAX_K, k % 16 == 0.
 *
 * w[r, c] = e4m3(codes[r, c]) * scales[r], the exact product rounded once to
 * out_dtype (nearest even).  For bf16 the rounding is exact while the
 * product is an fp32 normal number (|product| >= 2^-126); below that, a bf16
 * tie may be broken to even where the exact value lies off it.  NaN codes
 * give NaN.
 */
FP8W_API fp8w_status fp8w_dequantize(const uint8_t *codes, const float *scales, int64_t n,
                            int64_t k, int out_dtype, void *w, void *stream);

/*
 * fp8w_dequantize_grouped / fp8w_dequantize_mx -- fp8w_dequantize for codes
 * with per-group fp32 scales [n, k / group] (group 32, 64 or 128, k % group
 * == 0; 4-byte aligned) or E8M0 scale bytes [n, k / 32] (each 2^(b - 127),
 * 0xFF NaN; any alignment).  w[r, c] is the exact product of the decoded
 * code and its group's scale, rounded once to out_dtype.  An E8M0 product is
 * exact in fp32 (the smallest is 2^-136), so every output type gets the one
 * rounding of the exact value; fp32 group scales have fp8w_dequantize's bf16
 * limit below 2^-126.  Other arguments, checks and errors as
 * fp8w_dequantize.
 */
FP8W_API fp8w_status fp8w_dequantize_grouped(const uint8_t *codes, const float *scales, int group,
                                    int64_t n, int64_t k, int out_dtype, void *w, void *stream);
FP8W_API fp8w_status fp8w_dequantize_mx(const uint8_t *codes, const uint8_t *scales, int64_t n,
                               int64_t k, int out_dtype, void *w, void *stream);

/*
 * fp8w_linear -- steps "stream codes", "decode", "contract", "epilogue" and
 * "dispatch" of the contract (page "kadirnar/kernel-agent fp8-weights",
 * sections "The contract" and "Dequantise in registers": GEMV for M = 1,
 * a tensor-core kernel from M = 2).
 *
 *   x      [m, k] bf16 or fp16 bits (act_dtype), device, 16-byte aligned.
 *   codes  [n, k] e4m3 bytes from fp8w_quantize, device, 16-byte aligned.
 *   scales [n] fp32, device, 4-byte aligned.
 *   bias   [n] fp32, device, 4-byte aligned, or NULL for no bias.
 *   y      [m, n] in act_dtype, device, 2-byte aligned (output).
 *   1 <= m <= FP8W_MAX_DIM, 1 <= n <= FP8W_MAX_DIM, 16 <= k <= FP8W_MAX_K,
 *   k % 16 == 0.  x and y must not overlap codes, scales or bias.
 *
 * m == 1 with k <= 32768 runs the GEMV kernel; 2 <= m <= 64 the
 * tensor-core kernel for few tokens (one launch of 16, 32 or 64 token
 * columns; thread-block clusters of CTAs share 128-channel tiles and add up
 * their fp32 partials in distributed shared memory); m > 64 the prefill
 * GEMM, which dequantises each 128-row weight tile into shared memory once
 * and multiplies it by 128- or 256-token tiles.  Every path is one launch
 * and needs no workspace.
 */
FP8W_API fp8w_status fp8w_linear(const void *x, int act_dtype, int64_t m, int64_t k,
                        const uint8_t *codes, const float *scales,
                        const float *bias, int64_t n, void *y, void *stream);

/* Explicit kernel choice, for tests and tuning; fp8w_linear uses
 * FP8W_KERNEL_AUTO. */
enum { FP8W_KERNEL_AUTO = 0, FP8W_KERNEL_GEMV = 1, FP8W_KERNEL_SKINNY = 2, FP8W_KERNEL_PREFILL = 3 };

/*
 * FP8W_FLAG_WEIGHTS_READY (fp8w_linear_config.flags, fp8w_linear_w8a8's
 * flags): every write to the weight operands (codes and scales) completed
 * before this call was enqueued -- no kernel or copy that writes them is
 * still pending on any stream, as with weights quantised at load time and
 * followed by a synchronisation.  The linear kernels then start streaming
 * the codes while the preceding kernel in the stream is still finishing,
 * instead of first waiting for it; x, bias and y are still ordered after
 * that kernel.  Without the flag every global access waits for it.
 */
#define FP8W_FLAG_WEIGHTS_READY 1

typedef struct fp8w_linear_config {
    int kernel;   /* FP8W_KERNEL_*; GEMV requires m == 1 and k <= 32768 */
    int cluster;  /* FP8W_KERNEL_SKINNY only: CTAs per thread-block cluster,
                     1..16 (beyond 8 only where the device allows
                     non-portable clusters, else FP8W_ERR_CUDA) and at most
                     ceil(k / 128); beyond 32 tokens only 1 unless
                     tiles == 1; 0 (with tiles 0) chooses from the shape;
                     must be 0 for the other kernels */
    int tiles;    /* with cluster: 128-channel tiles each cluster shares
                     (its ranks split their units evenly), >= 1 */
    int flags;    /* 0 or FP8W_FLAG_WEIGHTS_READY */
    int reserved[4];  /* must be 0 */
} fp8w_linear_config;

/* fp8w_linear with an explicit configuration (NULL = automatic). */
FP8W_API fp8w_status fp8w_linear_ex(const void *x, int act_dtype, int64_t m, int64_t k,
                           const uint8_t *codes, const float *scales,
                           const float *bias, int64_t n, void *y,
                           const fp8w_linear_config *config, void *stream);

/*
 * fp8w_linear_noalloc -- the same call as fp8w_linear, kept for callers
 * that cannot allocate device memory while they run (a serving loop with a
 * fixed memory budget, where cudaMalloc could also synchronise the device,
 * or a host program whose device pointers come from another runtime).  No
 * path of the library uses scratch memory any more, so fp8w_linear itself
 * serves them: arguments, checks, kernels and results are identical.  The
 * pages have no counterpart.
 */
FP8W_API fp8w_status fp8w_linear_noalloc(const void *x, int act_dtype, int64_t m, int64_t k,
                                const uint8_t *codes, const float *scales,
                                const float *bias, int64_t n, void *y, void *stream);

/*
 * W8A8: the activations are quantised too (page "tensormux Write an FP8
 * kernel", "Required reasoning process", steps 2, 4 and 5: per-token
 * activation scales and per-channel weight scales, both amax / 448, a
 * saturating e4m3 conversion, and an epilogue that multiplies the fp32
 * accumulator by both scales; page "kadirnar/kernel-agent fp8-weights",
 * section "Tensor cores and libraries on sm_120", names the e4m3 x e4m3
 * tensor-core MMA as this separate target).  Two calls: fp8w_quantize_act
 * once per activation matrix, then fp8w_linear_w8a8 for every weight that
 * reads it.  The caller owns the activation codes and scales in between.
 */

/*
 * fp8w_quantize_act -- per-token activation codes and scales: row i of x,
 * widened exactly to fp32, takes fp8w_quantize's rule:
 *   x_scales[i]   = fp32(amax_k |x[i, k]| / 448), 1.0 when that is 0
 *   x_codes[i, k] = nearest-even, saturated e4m3 of fp32(x[i, k] / x_scales[i])
 *   x        [m, k] bf16 or fp16 bits (act_dtype), device, 16-byte aligned.
 *   x_codes  [m, k] uint8, device, 16-byte aligned (output).
 *   x_scales [m] fp32, device, 4-byte aligned (output).
 *   1 <= m <= FP8W_MAX_DIM, 16 <= k <= FP8W_MAX_K, k % 16 == 0.
 * It runs fp8w_quantize_ex's kernel: codes and scales equal that call's on
 * the same matrix.  Errors as fp8w_quantize_ex (FP8W_ERR_DTYPE for any
 * act_dtype but FP8W_BF16 / FP8W_F16).
 */
FP8W_API fp8w_status fp8w_quantize_act(const void *x, int act_dtype, int64_t m, int64_t k,
                              uint8_t *x_codes, float *x_scales, void *stream);

/*
 * fp8w_linear_w8a8 --
 *   y[i, r] = round_out( x_scales[i] * w_scales[r]
 *                        * sum_c e4m3(x_codes[i, c]) * e4m3(w_codes[r, c]) + bias[r] )
 * on the tensor cores (tcgen05.mma kind::f8f6f4: every product of two e4m3
 * values is exact, fp32 accumulation); in fp32 the accumulator is multiplied
 * by x_scales[i], then fused-multiplied by w_scales[r] with bias[r] added,
 * and rounded once to out_dtype.
 *   x_codes  [m, k] uint8 from fp8w_quantize_act, device, 16-byte aligned.
 *   x_scales [m] fp32, device, 4-byte aligned.
 *   w_codes  [n, k] uint8 from fp8w_quantize, device, 16-byte aligned.
 *   w_scales [n] fp32, device, 4-byte aligned.
 *   bias     [n] fp32, device, 4-byte aligned, or NULL for no bias.
 *   y        [m, n] of out_dtype (FP8W_BF16 or FP8W_F16), device, 2-byte
 *            aligned (output); it must not overlap the inputs.
 *   flags    0 or FP8W_FLAG_WEIGHTS_READY (for w_codes and w_scales).
 *   1 <= m, n <= FP8W_MAX_DIM, 16 <= k <= FP8W_MAX_K, k % 16 == 0.
 * One launch, no workspace.  Errors: FP8W_ERR_NULL, FP8W_ERR_SHAPE,
 * FP8W_ERR_ALIGN, FP8W_ERR_DTYPE (out_dtype), FP8W_ERR_CONFIG (unknown
 * flags), FP8W_ERR_CUDA.
 */
FP8W_API fp8w_status fp8w_linear_w8a8(const uint8_t *x_codes, const float *x_scales, int64_t m, int64_t k,
                             const uint8_t *w_codes, const float *w_scales, const float *bias, int64_t n,
                             void *y, int out_dtype, int flags, void *stream);

/* Human-readable name of a status code (static string). */
FP8W_API const char *fp8w_status_string(int status);

/* Name of the last failing CUDA call in this thread ("" if none). */
FP8W_API const char *fp8w_last_cuda_error(void);

/* Code recorded by a kernel that gave up a bounded wait on the current
 * device (0 = none), and clears it.  Synchronises the device first. */
FP8W_API int fp8w_device_error(void);

/* FP8W_ABI_VERSION of the loaded library. */
FP8W_API int fp8w_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8W_H */
