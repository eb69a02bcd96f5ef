// api.cu -- the C ABI of libfp8w (declared in include/fp8w.h): argument
// checks on the host, then dispatch to the kernels.  Nothing here allocates
// device memory or synchronises (except fp8w_device_error, which says so).
#include <cstdint>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/fp8w.h"
#include "fp8w_internal.h"

namespace {

thread_local char g_last_cuda_error[256] = "";

fp8w_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return FP8W_OK;
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s (%d)", what, cudaGetErrorString(e),
                  static_cast<int>(e));
    return FP8W_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_k(int64_t k) { return k >= 16 && k <= FP8W_MAX_K && (k % 16) == 0; }

fp8w_status check_linear(const void* x, int act, int64_t m, int64_t k, const uint8_t* codes,
                         const float* scales, const float* bias, int64_t n, const void* y) {
    if (!x || !codes || !scales || !y) return FP8W_ERR_NULL;
    if (act != FP8W_BF16 && act != FP8W_F16) return FP8W_ERR_DTYPE;
    if (m < 1 || n < 1 || m > FP8W_MAX_DIM || n > FP8W_MAX_DIM || !valid_k(k)) return FP8W_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4) || (bias && !aligned(bias, 4)) ||
        !aligned(y, 2))
        return FP8W_ERR_ALIGN;
    return FP8W_OK;
}

}  // namespace

extern "C" {

fp8w_status fp8w_quantize(const float* w, int64_t n, int64_t k, uint8_t* codes, float* scales, void* stream) {
    if (!w || !codes || !scales) return FP8W_ERR_NULL;
    if (n < 1 || n > FP8W_MAX_DIM || !valid_k(k)) return FP8W_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return FP8W_ERR_ALIGN;
    return cuda_status(fp8w::launch_quantize(w, n, k, codes, scales, static_cast<cudaStream_t>(stream)),
                       "fp8w_quantize launch");
}

fp8w_status fp8w_quantize_ex(const void* w, int w_dtype, int64_t n, int64_t k, uint8_t* codes, float* scales,
                             void* stream) {
    if (w_dtype == FP8W_F32) return fp8w_quantize(static_cast<const float*>(w), n, k, codes, scales, stream);
    if (!w || !codes || !scales) return FP8W_ERR_NULL;
    if (w_dtype != FP8W_BF16 && w_dtype != FP8W_F16) return FP8W_ERR_DTYPE;
    if (n < 1 || n > FP8W_MAX_DIM || !valid_k(k)) return FP8W_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return FP8W_ERR_ALIGN;
    return cuda_status(fp8w::launch_quantize_16(static_cast<const uint16_t*>(w), w_dtype == FP8W_BF16, n, k, codes,
                                                scales, static_cast<cudaStream_t>(stream)),
                       "fp8w_quantize_ex launch");
}

// m > 64 runs the prefill GEMM.
static bool use_prefill(int64_t m) { return m > 64; }

static bool valid_group(int group) { return group == 32 || group == 64 || group == 128; }

fp8w_status fp8w_quantize_grouped(const float* w, int64_t n, int64_t k, int group, uint8_t* codes, float* scales,
                                  void* stream) {
    if (!w || !codes || !scales) return FP8W_ERR_NULL;
    if (n < 1 || n > FP8W_MAX_DIM || !valid_k(k) || !valid_group(group) || k % group != 0) return FP8W_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return FP8W_ERR_ALIGN;
    return cuda_status(fp8w::launch_quantize_grouped(w, n, k, group, codes, scales, static_cast<cudaStream_t>(stream)),
                       "fp8w_quantize_grouped launch");
}

fp8w_status fp8w_linear_grouped(const void* x, int act_dtype, int64_t m, int64_t k, const uint8_t* codes,
                                const float* scales, int group, const float* bias, int64_t n, void* y, void* stream) {
    fp8w_status st = check_linear(x, act_dtype, m, k, codes, scales, bias, n, y);
    if (st != FP8W_OK) return st;
    if (!valid_group(group) || k % group != 0) return FP8W_ERR_SHAPE;
    if (!aligned(scales, 16)) return FP8W_ERR_ALIGN;
    fp8w::LinearArgs a{x, act_dtype, m, k, n, codes, scales, bias, y, group};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // m == 1: the GEMV, which bulk-copies each row's scales beside its codes
    // (k % (4 * group) == 0); otherwise the tensor-core kernels' per-group
    // form: the prefill GEMM beyond 64 tokens, the skinny kernel below
    if (m == 1 && k % (4 * group) == 0 && fp8w::gemv_supports(k))
        return cuda_status(fp8w::launch_gemv(a, s), "fp8w_linear_grouped gemv launch");
    if (use_prefill(m)) return cuda_status(fp8w::launch_prefill(a, s), "fp8w_linear_grouped prefill launch");
    return cuda_status(fp8w::launch_skinny(a, nullptr, s), "fp8w_linear_grouped tensor-core launch");
}

fp8w_status fp8w_quantize_mx(const float* w, int64_t n, int64_t k, uint8_t* codes, uint8_t* scales, void* stream) {
    if (!w || !codes || !scales) return FP8W_ERR_NULL;
    if (n < 1 || n > FP8W_MAX_DIM || !valid_k(k) || k % 32 != 0) return FP8W_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(codes, 16)) return FP8W_ERR_ALIGN;
    return cuda_status(fp8w::launch_quantize_mx(w, n, k, codes, scales, static_cast<cudaStream_t>(stream)),
                       "fp8w_quantize_mx launch");
}

fp8w_status fp8w_linear_mx(const void* x, int act_dtype, int64_t m, int64_t k, const uint8_t* codes,
                           const uint8_t* scales, const float* bias, int64_t n, void* y, void* stream) {
    const float* sp = reinterpret_cast<const float*>(scales);  // E8M0 bytes, passed through
    fp8w_status st = check_linear(x, act_dtype, m, k, codes, sp, bias, n, y);
    if (st != FP8W_OK) return st;
    // a unit's 128 codes take one 4-byte word of scale bytes a row
    if (k % 128 != 0) return FP8W_ERR_SHAPE;
    if (!aligned(scales, 16)) return FP8W_ERR_ALIGN;
    fp8w::LinearArgs a{x, act_dtype, m, k, n, codes, sp, bias, y, 32, true};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // m == 1: the GEMV, which bulk-copies a row's k / 32 scale bytes with its
    // codes (16-byte pieces: k % 512 == 0)
    if (m == 1 && k % 512 == 0 && fp8w::gemv_supports(k))
        return cuda_status(fp8w::launch_gemv(a, s), "fp8w_linear_mx gemv launch");
    // otherwise a tensor-core kernel (the prefill GEMM beyond 64 tokens, the
    // skinny kernel below): with bf16 activations the scales fold into the
    // bf16 weights; with fp16, the per-group form decodes each byte to fp32
    if (use_prefill(m)) return cuda_status(fp8w::launch_prefill(a, s), "fp8w_linear_mx prefill launch");
    return cuda_status(fp8w::launch_skinny(a, nullptr, s), "fp8w_linear_mx tensor-core launch");
}

fp8w_status fp8w_dequantize(const uint8_t* codes, const float* scales, int64_t n, int64_t k, int out_dtype,
                            void* w, void* stream) {
    if (!codes || !scales || !w) return FP8W_ERR_NULL;
    if (n < 1 || n > FP8W_MAX_DIM || !valid_k(k)) return FP8W_ERR_SHAPE;
    if (out_dtype != FP8W_F32 && out_dtype != FP8W_BF16 && out_dtype != FP8W_F16) return FP8W_ERR_DTYPE;
    if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(w, 16)) return FP8W_ERR_ALIGN;
    const int kind = out_dtype == FP8W_BF16 ? 1 : out_dtype == FP8W_F16 ? 2 : 0;
    return cuda_status(fp8w::launch_dequantize(codes, scales, n, k, kind, w, static_cast<cudaStream_t>(stream)),
                       "fp8w_dequantize launch");
}

static fp8w_status dequant_grouped(const uint8_t* codes, const void* scales, bool e8m0, int group, int64_t n,
                                   int64_t k, int out_dtype, void* w, void* stream, const char* what) {
    if (!codes || !scales || !w) return FP8W_ERR_NULL;
    if (n < 1 || n > FP8W_MAX_DIM || !valid_k(k) || !valid_group(group) || k % group != 0) return FP8W_ERR_SHAPE;
    if (out_dtype != FP8W_F32 && out_dtype != FP8W_BF16 && out_dtype != FP8W_F16) return FP8W_ERR_DTYPE;
    if (!aligned(codes, 16) || !aligned(scales, e8m0 ? 1 : 4) || !aligned(w, 16)) return FP8W_ERR_ALIGN;
    const int kind = out_dtype == FP8W_BF16 ? 1 : out_dtype == FP8W_F16 ? 2 : 0;
    return cuda_status(fp8w::launch_dequantize_grouped(codes, scales, e8m0, group, n, k, kind, w,
                                                       static_cast<cudaStream_t>(stream)),
                       what);
}

fp8w_status fp8w_dequantize_grouped(const uint8_t* codes, const float* scales, int group, int64_t n, int64_t k,
                                    int out_dtype, void* w, void* stream) {
    return dequant_grouped(codes, scales, false, group, n, k, out_dtype, w, stream, "fp8w_dequantize_grouped launch");
}

fp8w_status fp8w_dequantize_mx(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, int out_dtype,
                               void* w, void* stream) {
    return dequant_grouped(codes, scales, true, 32, n, k, out_dtype, w, stream, "fp8w_dequantize_mx launch");
}

// m == 1 runs the GEMV unless its x does not fit in shared memory.
static bool use_gemv(int64_t m, int64_t k) { return m == 1 && fp8w::gemv_supports(k); }

fp8w_status fp8w_linear_ex(const void* x, int act_dtype, int64_t m, int64_t k, const uint8_t* codes,
                           const float* scales, const float* bias, int64_t n, void* y,
                           const fp8w_linear_config* config, void* stream) {
    fp8w_status st = check_linear(x, act_dtype, m, k, codes, scales, bias, n, y);
    if (st != FP8W_OK) return st;
    int kernel = config ? config->kernel : FP8W_KERNEL_AUTO;
    if (kernel == FP8W_KERNEL_AUTO)
        kernel = use_gemv(m, k) ? FP8W_KERNEL_GEMV : use_prefill(m) ? FP8W_KERNEL_PREFILL : FP8W_KERNEL_SKINNY;
    if (kernel == FP8W_KERNEL_GEMV && !use_gemv(m, k)) return FP8W_ERR_CONFIG;
    if (kernel != FP8W_KERNEL_GEMV && kernel != FP8W_KERNEL_SKINNY && kernel != FP8W_KERNEL_PREFILL)
        return FP8W_ERR_CONFIG;
    const int cluster = config ? config->cluster : 0, tiles = config ? config->tiles : 0;
    if ((cluster == 0) != (tiles == 0) || cluster < 0 || tiles < 0) return FP8W_ERR_CONFIG;
    if (cluster != 0 && kernel != FP8W_KERNEL_SKINNY) return FP8W_ERR_CONFIG;
    const int flags = config ? config->flags : 0;
    if (flags & ~FP8W_FLAG_WEIGHTS_READY) return FP8W_ERR_CONFIG;
    if (config)
        for (int r : config->reserved)
            if (r != 0) return FP8W_ERR_CONFIG;
    fp8w::LinearArgs a{x, act_dtype, m, k, n, codes, scales, bias, y};
    a.early = (flags & FP8W_FLAG_WEIGHTS_READY) != 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kernel == FP8W_KERNEL_GEMV) return cuda_status(fp8w::launch_gemv(a, s), "fp8w_linear gemv launch");
    if (kernel == FP8W_KERNEL_PREFILL) return cuda_status(fp8w::launch_prefill(a, s), "fp8w_linear prefill launch");
    if (cluster != 0) {
        const fp8w::SkinnyShape shape{cluster, tiles};
        if (!fp8w::skinny_shape_valid(shape, m, k)) return FP8W_ERR_CONFIG;
        return cuda_status(fp8w::launch_skinny(a, &shape, s), "fp8w_linear tensor-core launch");
    }
    return cuda_status(fp8w::launch_skinny(a, nullptr, s), "fp8w_linear tensor-core launch");
}

fp8w_status fp8w_linear(const void* x, int act_dtype, int64_t m, int64_t k, const uint8_t* codes,
                        const float* scales, const float* bias, int64_t n, void* y, void* stream) {
    return fp8w_linear_ex(x, act_dtype, m, k, codes, scales, bias, n, y, nullptr, stream);
}

fp8w_status fp8w_linear_noalloc(const void* x, int act_dtype, int64_t m, int64_t k, const uint8_t* codes,
                                const float* scales, const float* bias, int64_t n, void* y, void* stream) {
    return fp8w_linear_ex(x, act_dtype, m, k, codes, scales, bias, n, y, nullptr, stream);
}

fp8w_status fp8w_quantize_act(const void* x, int act_dtype, int64_t m, int64_t k, uint8_t* x_codes, float* x_scales,
                              void* stream) {
    if (act_dtype != FP8W_BF16 && act_dtype != FP8W_F16) return FP8W_ERR_DTYPE;
    return fp8w_quantize_ex(x, act_dtype, m, k, x_codes, x_scales, stream);
}

fp8w_status fp8w_linear_w8a8(const uint8_t* x_codes, const float* x_scales, int64_t m, int64_t k,
                             const uint8_t* w_codes, const float* w_scales, const float* bias, int64_t n, void* y,
                             int out_dtype, int flags, void* stream) {
    if (!x_codes || !x_scales || !w_codes || !w_scales || !y) return FP8W_ERR_NULL;
    if (out_dtype != FP8W_BF16 && out_dtype != FP8W_F16) return FP8W_ERR_DTYPE;
    if (m < 1 || n < 1 || m > FP8W_MAX_DIM || n > FP8W_MAX_DIM || !valid_k(k)) return FP8W_ERR_SHAPE;
    if (!aligned(x_codes, 16) || !aligned(w_codes, 16) || !aligned(x_scales, 4) || !aligned(w_scales, 4) ||
        (bias && !aligned(bias, 4)) || !aligned(y, 2))
        return FP8W_ERR_ALIGN;
    if (flags & ~FP8W_FLAG_WEIGHTS_READY) return FP8W_ERR_CONFIG;
    fp8w::W8A8Args a{x_codes, x_scales, m, k, n, w_codes, w_scales, bias, y, out_dtype,
                     (flags & FP8W_FLAG_WEIGHTS_READY) != 0};
    return cuda_status(fp8w::launch_w8a8(a, static_cast<cudaStream_t>(stream)), "fp8w_linear_w8a8 launch");
}

const char* fp8w_status_string(int status) {
    switch (status) {
        case FP8W_OK: return "ok";
        case FP8W_ERR_NULL: return "a required pointer is NULL";
        case FP8W_ERR_SHAPE: return "shape out of range (need m,n >= 1, 16 <= k <= 65536, k % 16 == 0)";
        case FP8W_ERR_ALIGN: return "pointer misaligned (x, codes, w: 16 B; scales, bias: 4 B; y: 2 B)";
        case FP8W_ERR_DTYPE: return "activation dtype must be FP8W_BF16 or FP8W_F16";
        case FP8W_ERR_CUDA: return "CUDA call failed (see fp8w_last_cuda_error)";
        case FP8W_ERR_CONFIG: return "invalid explicit launch configuration";
        default: return "unknown status";
    }
}

const char* fp8w_last_cuda_error(void) { return g_last_cuda_error; }

int fp8w_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    const int a = fp8w::read_skinny_device_error();
    const int b = fp8w::read_gemv_device_error();
    const int c = fp8w::read_prefill_device_error();
    const int d = fp8w::read_w8a8_device_error();
    return a ? a : b ? b : c ? c : d;
}

int fp8w_abi_version(void) { return FP8W_ABI_VERSION; }

}  // extern "C"
