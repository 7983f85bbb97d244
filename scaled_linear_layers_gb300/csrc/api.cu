// C-ABI entry points: host-side validation, then launches on the caller's
// stream.  Nothing here allocates device memory; nothing synchronises except
// fp8_check_device_status and the meta checkpoint's save and load.  The
// delayed-scaling step also uses a second stream the library owns (created
// once per host thread and device), forked from and joined back into the
// caller's stream with events.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace fp8 {

extern std::atomic<uint64_t> g_wait_limit_ns;

namespace {

thread_local char g_err[512] = "";

fp8_status fail(fp8_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

fp8_status cuda_status(cudaError_t e, const char *where, const char *why = nullptr) {
    if (e == cudaSuccess) return FP8_OK;
    return fail(FP8_ERR_CUDA, "%s: %s%s%s", where, cudaGetErrorString(e), why ? " — " : "",
                why ? why : "");
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

thread_local int tl_fail_launches = 0;

namespace {

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
int g_arch_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other

fp8_status check_device(const char *who) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, who);
    if (dev < 0 || dev >= kMaxDevices) return fail(FP8_ERR_UNSUPPORTED, "%s: device %d", who, dev);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = sms > 0 ? sms : 1;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        if (g_arch_ok[dev] < 0)
            snprintf(g_err, sizeof g_err, "device %d is sm_%d%d", dev, major, minor);
    }
    if (g_arch_ok[dev] < 0)
        return fail(FP8_ERR_UNSUPPORTED, "%s: this library runs on sm_103 (GB300) only", who);
    return FP8_OK;
}

fp8_status check_dim16(const char *who, const char *name, int64_t v, int64_t mult) {
    if (v % mult != 0)
        return fail(FP8_ERR_ALIGNMENT, "%s: Expected %s to be divisible by %lld, but got %s=%lld",
                    who, name, (long long)mult, name, (long long)v);
    return FP8_OK;
}

#define FP8_TRY(expr)                   \
    do {                                \
        fp8_status _st = (expr);        \
        if (_st != FP8_OK) return _st;  \
    } while (0)

#define FP8_NEED(ptr, who)                                                       \
    do {                                                                         \
        if ((ptr) == nullptr) return fail(FP8_ERR_NULL, "%s: %s is NULL", who, #ptr); \
    } while (0)

#define FP8_ALIGN(ptr, who)                                                                   \
    do {                                                                                      \
        if ((ptr) != nullptr && !aligned16(ptr))                                              \
            return fail(FP8_ERR_ALIGNMENT, "%s: %s is not 16-byte aligned", who, #ptr);       \
    } while (0)

}  // namespace

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace fp8

using namespace fp8;

extern "C" {

const char *fp8_last_error(void) { return g_err; }

const char *fp8_version(void) { return "fp8linear 0.1 sm_103a"; }

fp8_status fp8_amax(const uint16_t *x, int64_t n, float *amax_out, cudaStream_t s) {
    const char *who = "fp8_amax";
    if (n < 0) return fail(FP8_ERR_SHAPE, "%s: n=%lld < 0", who, (long long)n);
    FP8_NEED(amax_out, who);
    if (n > 0) FP8_NEED(x, who);
    FP8_ALIGN(x, who);
    FP8_TRY(check_device(who));
    return cuda_status(launch_amax(x, n, amax_out, s), who);
}

fp8_status fp8_quantize(const uint16_t *x, int64_t rows, int64_t cols, fp8_recipe r, float *scale,
                        float *scale_inv, uint8_t *q, float *amax_out, cudaStream_t s) {
    const char *who = "fp8_quantize";
    if (rows < 0 || cols < 0)
        return fail(FP8_ERR_SHAPE, "%s: negative shape [%lld, %lld]", who, (long long)rows,
                    (long long)cols);
    const int64_t n = rows * cols;
    if (n > 0) {
        FP8_NEED(x, who);
        FP8_NEED(q, who);
    }
    FP8_ALIGN(x, who);
    FP8_ALIGN(q, who);
    switch (r) {
    case FP8_RECIPE_DELAYED:
        FP8_NEED(scale_inv, who);
        FP8_TRY(check_device(who));
        return cuda_status(launch_quantize_tensor(x, n, false, scale, scale_inv, q, amax_out, s), who);
    case FP8_RECIPE_DYNAMIC:
        FP8_NEED(scale, who);
        FP8_NEED(scale_inv, who);
        FP8_NEED(amax_out, who);
        FP8_TRY(check_device(who));
        return cuda_status(launch_quantize_tensor(x, n, true, scale, scale_inv, q, amax_out, s), who);
    case FP8_RECIPE_BLOCK:
        FP8_TRY(check_dim16(who, "cols", cols, 128));
        FP8_NEED(scale, who);
        FP8_NEED(scale_inv, who);
        FP8_TRY(check_device(who));
        return cuda_status(launch_quantize_rowtiles(x, rows, cols, scale, scale_inv, q, amax_out, s),
                           who);
    case FP8_RECIPE_BLOCK_2D:
        FP8_TRY(check_dim16(who, "rows", rows, 128));
        FP8_TRY(check_dim16(who, "cols", cols, 128));
        FP8_NEED(scale, who);
        FP8_NEED(scale_inv, who);
        if (rows > 0x7FFFFFFF || cols > 0x7FFFFFFF)
            return fail(FP8_ERR_SHAPE, "%s: dims must fit in 31 bits", who);
        FP8_TRY(check_device(who));
        // the cast+transpose kernel without its transposed output
        return cuda_status(launch_quantize_transpose(x, rows, cols, 2, scale, scale_inv, q, nullptr,
                                                     nullptr, nullptr, amax_out, s),
                           who);
    }
    return fail(FP8_ERR_SHAPE, "%s: unknown recipe %d", who, (int)r);
}

fp8_status fp8_quantize_transpose(const uint16_t *x, int64_t rows, int64_t cols, fp8_recipe r,
                                  float *scale, float *scale_inv, uint8_t *q, uint8_t *qt,
                                  float *scale_t, float *scale_inv_t, float *amax_out,
                                  cudaStream_t s) {
    const char *who = "fp8_quantize_transpose";
    if (rows < 0 || cols < 0)
        return fail(FP8_ERR_SHAPE, "%s: negative shape [%lld, %lld]", who, (long long)rows,
                    (long long)cols);
    if (rows > 0x7FFFFFFF || cols > 0x7FFFFFFF)
        return fail(FP8_ERR_SHAPE, "%s: dims must fit in 31 bits", who);
    const int64_t mult = (r == FP8_RECIPE_BLOCK || r == FP8_RECIPE_BLOCK_2D) ? 128 : 16;
    FP8_TRY(check_dim16(who, "rows", rows, mult));
    FP8_TRY(check_dim16(who, "cols", cols, mult));
    if (rows * cols > 0) {
        FP8_NEED(x, who);
        FP8_NEED(qt, who);
    }
    FP8_ALIGN(x, who);
    FP8_ALIGN(q, who);
    FP8_ALIGN(qt, who);
    int mode;
    switch (r) {
    case FP8_RECIPE_DELAYED:
        FP8_NEED(scale_inv, who);
        mode = 0;
        break;
    case FP8_RECIPE_DYNAMIC:
        FP8_NEED(scale, who);
        FP8_NEED(scale_inv, who);
        FP8_NEED(amax_out, who);
        mode = 1;
        break;
    case FP8_RECIPE_BLOCK_2D:
        FP8_NEED(scale, who);
        FP8_NEED(scale_inv, who);
        mode = 2;
        break;
    case FP8_RECIPE_BLOCK:
        FP8_NEED(scale_t, who);
        FP8_NEED(scale_inv_t, who);
        if (q != nullptr) {
            FP8_NEED(scale, who);
            FP8_NEED(scale_inv, who);
        }
        mode = 3;
        break;
    default:
        return fail(FP8_ERR_SHAPE, "%s: unknown recipe %d", who, (int)r);
    }
    FP8_TRY(check_device(who));
    return cuda_status(launch_quantize_transpose(x, rows, cols, mode, scale, scale_inv, q, qt,
                                                 scale_t, scale_inv_t, amax_out, s),
                       who);
}

size_t fp8_dbias_workspace_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)((rows + 127) / 128) * (size_t)cols * sizeof(float);
}

fp8_status fp8_quantize_transpose_dbias(const uint16_t *g, int64_t rows, int64_t cols,
                                        fp8_recipe r, float *scale, float *scale_inv, uint8_t *q,
                                        uint8_t *qt, float *amax_out, uint16_t *dbias,
                                        float *workspace, cudaStream_t s) {
    const char *who = "fp8_quantize_transpose_dbias";
    if (r != FP8_RECIPE_DELAYED && r != FP8_RECIPE_DYNAMIC)
        return fail(FP8_ERR_UNSUPPORTED, "%s: tensorwise recipes only (DELAYED, DYNAMIC)", who);
    if (rows * cols > 0) {
        FP8_NEED(dbias, who);
        FP8_NEED(workspace, who);
    }
    FP8_ALIGN(dbias, who);
    FP8_ALIGN(workspace, who);
    // the quantisation's own checks, then the fused launch and the reduction
    if (rows < 0 || cols < 0 || rows > 0x7FFFFFFF || cols > 0x7FFFFFFF)
        return fail(FP8_ERR_SHAPE, "%s: bad shape [%lld, %lld]", who, (long long)rows,
                    (long long)cols);
    FP8_TRY(check_dim16(who, "rows", rows, 16));
    FP8_TRY(check_dim16(who, "cols", cols, 16));
    if (rows * cols > 0) {
        FP8_NEED(g, who);
        FP8_NEED(qt, who);
    }
    FP8_ALIGN(g, who);
    FP8_ALIGN(q, who);
    FP8_ALIGN(qt, who);
    FP8_NEED(scale_inv, who);
    if (r == FP8_RECIPE_DYNAMIC) {
        FP8_NEED(scale, who);
        FP8_NEED(amax_out, who);
    }
    FP8_TRY(check_device(who));
    if (rows * cols == 0) {
        if (cols > 0) FP8_TRY(cuda_status(cudaMemsetAsync(dbias, 0, cols * 2, s), who));
        return cuda_status(launch_quantize_transpose(g, rows, cols, r == FP8_RECIPE_DYNAMIC ? 1 : 0,
                                                     scale, scale_inv, q, qt, nullptr, nullptr,
                                                     amax_out, s),
                           who);
    }
    FP8_TRY(cuda_status(launch_quantize_transpose(g, rows, cols, r == FP8_RECIPE_DYNAMIC ? 1 : 0,
                                                  scale, scale_inv, q, qt, nullptr, nullptr,
                                                  amax_out, s, workspace),
                        who));
    return cuda_status(launch_colsum_reduce(workspace, rows, cols, dbias, s), who);
}

size_t fp8_quantize_fused_workspace_bytes(void) { return kFusedWorkspaceBytes; }

fp8_status fp8_quantize_fused_dynamic(const uint16_t *x, int64_t rows, int64_t cols, float *scale,
                                      float *scale_inv, uint8_t *q, uint8_t *qt, float *amax_out,
                                      void *workspace, cudaStream_t s) {
    const char *who = "fp8_quantize_fused_dynamic";
    if (rows < 0 || cols < 0 || rows > 0x7FFFFFFF || cols > 0x7FFFFFFF)
        return fail(FP8_ERR_SHAPE, "%s: bad shape [%lld, %lld]", who, (long long)rows,
                    (long long)cols);
    if (!fused_tiles_fit(rows, cols))
        return fail(FP8_ERR_SHAPE, "%s: [%lld, %lld] has more 128x128 tiles than 2^31 - 1", who,
                    (long long)rows, (long long)cols);
    FP8_TRY(check_dim16(who, "rows", rows, 16));
    FP8_TRY(check_dim16(who, "cols", cols, 16));
    if (rows * cols > 0) {
        FP8_NEED(x, who);
        if (q == nullptr && qt == nullptr) return fail(FP8_ERR_NULL, "%s: q and qt are both NULL", who);
    }
    FP8_NEED(scale, who);
    FP8_NEED(scale_inv, who);
    FP8_NEED(amax_out, who);
    FP8_NEED(workspace, who);
    FP8_ALIGN(x, who);
    FP8_ALIGN(q, who);
    FP8_ALIGN(qt, who);
    FP8_ALIGN(workspace, who);
    FP8_TRY(check_device(who));
    return cuda_status(launch_quantize_fused_dynamic(x, rows, cols, scale, scale_inv, q, qt, amax_out,
                                                     static_cast<unsigned int *>(workspace), s),
                       who);
}

fp8_status fp8_quantize_fused_dynamic_noalloc(const uint16_t *x, int64_t rows, int64_t cols,
                                              float *scale, float *scale_inv, uint8_t *q,
                                              uint8_t *qt, float *amax_out, cudaStream_t s) {
    const char *who = "fp8_quantize_fused_dynamic_noalloc";
    if (rows < 0 || cols < 0 || rows > 0x7FFFFFFF || cols > 0x7FFFFFFF)
        return fail(FP8_ERR_SHAPE, "%s: bad shape [%lld, %lld]", who, (long long)rows,
                    (long long)cols);
    if (!fused_tiles_fit(rows, cols))
        return fail(FP8_ERR_SHAPE, "%s: [%lld, %lld] has more 128x128 tiles than 2^31 - 1", who,
                    (long long)rows, (long long)cols);
    FP8_TRY(check_dim16(who, "rows", rows, 16));
    FP8_TRY(check_dim16(who, "cols", cols, 16));
    if (rows * cols > 0) {
        FP8_NEED(x, who);
        if (q == nullptr && qt == nullptr) return fail(FP8_ERR_NULL, "%s: q and qt are both NULL", who);
    }
    FP8_NEED(scale, who);
    FP8_NEED(scale_inv, who);
    FP8_NEED(amax_out, who);
    FP8_ALIGN(x, who);
    FP8_ALIGN(q, who);
    FP8_ALIGN(qt, who);
    FP8_TRY(check_device(who));
    const char *why = nullptr;
    cudaError_t e = launch_quantize_fused_dynamic_noalloc(x, rows, cols, scale, scale_inv, q, qt,
                                                          amax_out, s, &why);
    return cuda_status(e, who, why);
}

static fp8_status gemm_common(const char *who, const uint8_t *A, const float *sa, const uint8_t *B,
                              const float *sb, int64_t M, int64_t N, int64_t K, fp8_recipe r,
                              uint16_t *D, const char *mname, const char *nname, const char *kname,
                              bool device_check = true) {
    if (M <= 0 || N <= 0 || K <= 0)
        return fail(FP8_ERR_SHAPE, "%s: empty or negative GEMM [%s=%lld, %s=%lld, %s=%lld]", who,
                    mname, (long long)M, nname, (long long)N, kname, (long long)K);
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF)
        return fail(FP8_ERR_SHAPE, "%s: dims must fit in 31 bits", who);
    const int64_t mult = r == FP8_RECIPE_BLOCK ? 128 : 16;
    FP8_TRY(check_dim16(who, mname, M, mult));
    FP8_TRY(check_dim16(who, nname, N, mult));
    FP8_TRY(check_dim16(who, kname, K, mult));
    FP8_NEED(A, who);
    FP8_NEED(B, who);
    FP8_NEED(sa, who);
    FP8_NEED(sb, who);
    FP8_NEED(D, who);
    FP8_ALIGN(A, who);
    FP8_ALIGN(B, who);
    FP8_ALIGN(D, who);
    if (r == FP8_RECIPE_BLOCK) {
        // the block kernel stages per-row B scales with 16-byte async copies
        if (!aligned16(sa) || !aligned16(sb))
            return fail(FP8_ERR_ALIGNMENT, "%s: block scales are not 16-byte aligned", who);
    }
    if (r != FP8_RECIPE_DELAYED && r != FP8_RECIPE_DYNAMIC && r != FP8_RECIPE_BLOCK)
        return fail(FP8_ERR_SHAPE, "%s: recipe %d is not a GEMM recipe", who, (int)r);
    return device_check ? check_device(who) : FP8_OK;
}

fp8_status fp8_linear_fprop(const uint8_t *xq, const float *x_scale, const uint8_t *wq,
                            const float *w_scale, int64_t M, int64_t N, int64_t K, fp8_recipe r,
                            const uint16_t *bias, uint16_t *y, cudaStream_t s) {
    const char *who = "fp8_linear_fprop";
    FP8_TRY(gemm_common(who, xq, x_scale, wq, w_scale, M, N, K, r, y, "M", "N", "K"));
    const char *why = nullptr;
    if (r == FP8_RECIPE_BLOCK) {
        if (bias != nullptr) return fail(FP8_ERR_UNSUPPORTED, "%s: bias with the block recipe", who);
        // A = Xq [M,K], scales [M, K/128]; B = Wq [N,K], 128x128 grid [N/128, K/128]
        const BlockScales sc{x_scale, K / 128, 1, w_scale, K / 128, 1, 128};
        return cuda_status(launch_gemm_block(xq, wq, M, N, K, sc, y, s, &why), who, why);
    }
    FP8_ALIGN(bias, who);
    return cuda_status(launch_gemm_tensor(xq, wq, M, N, K, x_scale, w_scale, bias, y, s, &why), who,
                       why);
}

fp8_status fp8_linear_dgrad(const uint8_t *gq, const float *g_scale, const uint8_t *wqt,
                            const float *w_scale, int64_t M, int64_t N, int64_t K, fp8_recipe r,
                            uint16_t *dx, cudaStream_t s) {
    const char *who = "fp8_linear_dgrad";
    // dX [M,K]: GEMM rows M, cols K, contraction N
    FP8_TRY(gemm_common(who, gq, g_scale, wqt, w_scale, M, N, K, r, dx, "M", "N", "K"));
    const char *why = nullptr;
    if (r == FP8_RECIPE_BLOCK) {
        // A = Gq [M,N], scales [M, N/128]; B = Wqᵀ [K,N]: the scale of B row k,
        // contraction block nb is W's grid entry [nb, k/128].
        const BlockScales sc{g_scale, N / 128, 1, w_scale, 1, K / 128, 128};
        return cuda_status(launch_gemm_block(gq, wqt, M, K, N, sc, dx, s, &why), who, why);
    }
    return cuda_status(launch_gemm_tensor(gq, wqt, M, K, N, g_scale, w_scale, nullptr, dx, s, &why),
                       who, why);
}

fp8_status fp8_linear_wgrad(const uint8_t *gqt, const float *g_scale, const uint8_t *xqt,
                            const float *x_scale, int64_t M, int64_t N, int64_t K, fp8_recipe r,
                            uint16_t *dw, cudaStream_t s) {
    const char *who = "fp8_linear_wgrad";
    // dW [N,K]: GEMM rows N, cols K, contraction M
    FP8_TRY(gemm_common(who, gqt, g_scale, xqt, x_scale, M, N, K, r, dw, "M", "N", "K"));
    const char *why = nullptr;
    if (r == FP8_RECIPE_BLOCK) {
        // A = Gqᵀ [N,M] and B = Xqᵀ [K,M]; their column-tile scales are
        // [M/128, N] and [M/128, K] (block-major)
        const BlockScales sc{g_scale, 1, N, x_scale, 1, K, 1};
        return cuda_status(launch_gemm_block(gqt, xqt, N, K, M, sc, dw, s, &why), who, why);
    }
    return cuda_status(launch_gemm_tensor(gqt, xqt, N, K, M, g_scale, x_scale, nullptr, dw, s, &why),
                       who, why);
}

fp8_status fp8_linear_dgrad_wgrad(const uint8_t *gq, const uint8_t *gqt, const float *g_scale,
                                  const uint8_t *wqt, const float *w_scale, const uint8_t *xqt,
                                  const float *x_scale, int64_t M, int64_t N, int64_t K,
                                  fp8_recipe r, uint16_t *dx, uint16_t *dw, cudaStream_t s) {
    const char *who = "fp8_linear_dgrad_wgrad";
    if (r == FP8_RECIPE_BLOCK)
        return fail(FP8_ERR_UNSUPPORTED,
                    "%s: the block recipe takes fp8_linear_dgrad and fp8_linear_wgrad", who);
    // both problems' arguments first, then the device
    FP8_TRY(gemm_common(who, gq, g_scale, wqt, w_scale, M, N, K, r, dx, "M", "N", "K", false));
    FP8_TRY(gemm_common(who, gqt, g_scale, xqt, x_scale, M, N, K, r, dw, "M", "N", "K"));
    const char *why = nullptr;
    // dX [M,K] = Gq · (Wqᵀ)ᵀ (contraction N); dW [N,K] = Gqᵀ · (Xqᵀ)ᵀ (contraction M)
    const PairGemm dgrad{gq, wqt, M, K, N, g_scale, w_scale, nullptr, dx};
    const PairGemm wgrad{gqt, xqt, N, K, M, g_scale, x_scale, nullptr, dw};
    return cuda_status(launch_gemm_tensor2(dgrad, wgrad, s, &why), who, why);
}

fp8_status fp8_meta_init(fp8_meta *m, float *dev_block, int32_t interval, cudaStream_t s) {
    const char *who = "fp8_meta_init";
    FP8_NEED(m, who);
    FP8_NEED(dev_block, who);
    FP8_ALIGN(dev_block, who);
    if (interval < 1 || interval > 1024)
        return fail(FP8_ERR_SHAPE, "%s: interval=%d outside 1..1024", who, interval);
    FP8_TRY(check_device(who));
    m->dev = dev_block;
    m->interval = interval;
    m->idx = 0;
    return cuda_status(launch_meta_init(dev_block, interval, s), who);
}

fp8_status fp8_meta_record(fp8_meta *m, fp8_slot which, const float *amax_dev, cudaStream_t s) {
    const char *who = "fp8_meta_record";
    FP8_NEED(m, who);
    FP8_NEED(m->dev, who);
    FP8_NEED(amax_dev, who);
    if (m->interval < 1 || m->idx < 0 || m->idx >= m->interval)
        return fail(FP8_ERR_SHAPE, "%s: corrupt meta (interval=%d idx=%d)", who, m->interval, m->idx);
    FP8_TRY(check_device(who));
    switch (which) {
    case FP8_SLOT_W: {
        fp8_status st = cuda_status(launch_meta_copy(m->dev + FP8_META_HISTORY + m->idx, amax_dev, s), who);
        if (st == FP8_OK) m->idx = (m->idx + 1) % m->interval;
        return st;
    }
    case FP8_SLOT_X:
        return cuda_status(launch_meta_lag(m->dev + FP8_META_X_SCALE, m->dev + FP8_META_X_SCALE_INV,
                                           amax_dev, s),
                           who);
    case FP8_SLOT_G:
        return cuda_status(launch_meta_lag(m->dev + FP8_META_G_SCALE, m->dev + FP8_META_G_SCALE_INV,
                                           amax_dev, s),
                           who);
    }
    return fail(FP8_ERR_SHAPE, "%s: unknown slot %d", who, (int)which);
}

fp8_status fp8_meta_refresh(fp8_meta *m, cudaStream_t s) {
    const char *who = "fp8_meta_refresh";
    FP8_NEED(m, who);
    FP8_NEED(m->dev, who);
    if (m->interval < 1) return fail(FP8_ERR_SHAPE, "%s: corrupt meta", who);
    FP8_TRY(check_device(who));
    return cuda_status(launch_meta_refresh(m->dev, m->interval, s), who);
}

namespace {

// Header of a saved meta state; the device block's floats follow it.
struct MetaBlobHeader {
    uint32_t magic, version;
    int32_t interval, idx;
    int64_t step_count;
};
constexpr uint32_t kMetaBlobMagic = 0x534D3846u;  // "F8MS"
constexpr uint32_t kMetaBlobVersion = 1;

}  // namespace

size_t fp8_meta_state_bytes(int32_t interval) {
    if (interval < 1 || interval > 1024) return 0;
    return sizeof(MetaBlobHeader) + (size_t)FP8_META_FLOATS(interval) * sizeof(float);
}

fp8_status fp8_meta_save(const fp8_meta *m, int64_t step_count, void *host_buf, size_t bytes,
                         cudaStream_t s) {
    const char *who = "fp8_meta_save";
    FP8_NEED(m, who);
    FP8_NEED(m->dev, who);
    FP8_NEED(host_buf, who);
    if (m->interval < 1 || m->interval > 1024 || m->idx < 0 || m->idx >= m->interval)
        return fail(FP8_ERR_SHAPE, "%s: corrupt meta", who);
    const size_t need = fp8_meta_state_bytes(m->interval);
    if (bytes < need)
        return fail(FP8_ERR_SHAPE, "%s: buffer of %zu bytes, %zu needed", who, bytes, need);
    FP8_TRY(check_device(who));
    MetaBlobHeader h{kMetaBlobMagic, kMetaBlobVersion, m->interval, m->idx, step_count};
    std::memcpy(host_buf, &h, sizeof h);
    float *dst = reinterpret_cast<float *>(static_cast<char *>(host_buf) + sizeof h);
    FP8_TRY(cuda_status(cudaMemcpyAsync(dst, m->dev, FP8_META_FLOATS(m->interval) * sizeof(float),
                                        cudaMemcpyDeviceToHost, s),
                        who));
    return cuda_status(cudaStreamSynchronize(s), who);
}

fp8_status fp8_meta_load(fp8_meta *m, float *dev_block, int64_t *step_count, const void *host_buf,
                         size_t bytes, cudaStream_t s) {
    const char *who = "fp8_meta_load";
    FP8_NEED(m, who);
    FP8_NEED(dev_block, who);
    FP8_NEED(host_buf, who);
    FP8_ALIGN(dev_block, who);
    MetaBlobHeader h;
    if (bytes < sizeof h) return fail(FP8_ERR_SHAPE, "%s: buffer shorter than the header", who);
    std::memcpy(&h, host_buf, sizeof h);
    if (h.magic != kMetaBlobMagic || h.version != kMetaBlobVersion)
        return fail(FP8_ERR_SHAPE, "%s: not a saved fp8 meta state (version %u)", who,
                    (unsigned)h.version);
    if (h.interval < 1 || h.interval > 1024 || h.idx < 0 || h.idx >= h.interval)
        return fail(FP8_ERR_SHAPE, "%s: corrupt state (interval %d, idx %d)", who, h.interval,
                    h.idx);
    if (bytes < fp8_meta_state_bytes(h.interval))
        return fail(FP8_ERR_SHAPE, "%s: buffer of %zu bytes, %zu needed", who, bytes,
                    fp8_meta_state_bytes(h.interval));
    FP8_TRY(check_device(who));
    const float *src =
        reinterpret_cast<const float *>(static_cast<const char *>(host_buf) + sizeof h);
    FP8_TRY(cuda_status(cudaMemcpyAsync(dev_block, src,
                                        FP8_META_FLOATS(h.interval) * sizeof(float),
                                        cudaMemcpyHostToDevice, s),
                        who));
    FP8_TRY(cuda_status(cudaStreamSynchronize(s), who));
    m->dev = dev_block;
    m->interval = h.interval;
    m->idx = h.idx;
    if (step_count != nullptr) *step_count = h.step_count;
    return FP8_OK;
}

fp8_status fp8_state_step(int64_t *step_count, int32_t interval, fp8_meta *metas, int32_t n,
                          cudaStream_t s) {
    const char *who = "fp8_state_step";
    FP8_NEED(step_count, who);
    if (interval < 1) return fail(FP8_ERR_SHAPE, "%s: interval=%d", who, interval);
    if (n < 0 || (n > 0 && metas == nullptr)) return fail(FP8_ERR_NULL, "%s: metas", who);
    *step_count += 1;
    if (*step_count % interval != 0) return FP8_OK;
    for (int32_t i = 0; i < n; ++i) FP8_TRY(fp8_meta_refresh(&metas[i], s));
    return FP8_OK;
}

namespace {

// The second stream of fp8_linear_step_delayed and its fork/join events, one
// set per host thread and device (created on first use, kept for the thread's
// lifetime), so concurrent callers never share them.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideStream tl_side[kMaxDevices];

fp8_status side_stream(const char *who, SideStream **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, who);
    SideStream &ss = tl_side[dev];
    if (ss.stream == nullptr) {
        if ((e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_status(e, who, "creating the step's second stream");
    }
    *out = &ss;
    return FP8_OK;
}

}  // namespace

fp8_status fp8_linear_step_delayed(fp8_meta *m, int64_t *step_count, const fp8_linear_step_io *io,
                                   int64_t M, int64_t N, int64_t K, cudaEvent_t *events,
                                   cudaStream_t s) {
    const char *who = "fp8_linear_step_delayed";
    FP8_NEED(m, who);
    FP8_NEED(m->dev, who);
    FP8_NEED(step_count, who);
    FP8_NEED(io, who);
    if (M <= 0 || N <= 0 || K <= 0 || M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF)
        return fail(FP8_ERR_SHAPE, "%s: bad shape [M=%lld, N=%lld, K=%lld]", who, (long long)M,
                    (long long)N, (long long)K);
    FP8_TRY(check_dim16(who, "M", M, 16));
    FP8_TRY(check_dim16(who, "N", N, 16));
    FP8_TRY(check_dim16(who, "K", K, 16));
    if (m->interval < 1 || m->idx < 0 || m->idx >= m->interval)
        return fail(FP8_ERR_SHAPE, "%s: corrupt meta", who);
    const bool bwd = io->g != nullptr;
    FP8_NEED(io->x, who);
    FP8_NEED(io->w, who);
    FP8_NEED(io->xq, who);
    FP8_NEED(io->wq, who);
    FP8_NEED(io->wqt, who);
    FP8_NEED(io->amax, who);
    FP8_NEED(io->y, who);
    if (bwd) {
        FP8_NEED(io->gq, who);
        FP8_NEED(io->gqt, who);
        FP8_NEED(io->xqt, who);
    }
    if (io->dbias != nullptr) {
        if (!bwd) return fail(FP8_ERR_NULL, "%s: dbias needs g", who);
        FP8_NEED(io->dbias_workspace, who);
    }
    if ((io->flags & ~FP8_STEP_SAVE_XQ_FWD) != 0)
        return fail(FP8_ERR_SHAPE, "%s: unknown flags 0x%x", who, (unsigned)io->flags);
    const bool save_x = (io->flags & FP8_STEP_SAVE_XQ_FWD) != 0;
    if (save_x && io->xqt == nullptr)
        return fail(FP8_ERR_NULL, "%s: FP8_STEP_SAVE_XQ_FWD needs xqt", who);
    const void *ptrs[] = {io->x, io->w, io->g, io->bias, io->xq, io->xqt, io->wq, io->wqt,
                          io->gq, io->gqt, io->y, io->dx, io->dw, io->dbias, io->dbias_workspace};
    for (const void *p : ptrs)
        if (p != nullptr && !aligned16(p))
            return fail(FP8_ERR_ALIGNMENT, "%s: a buffer is not 16-byte aligned", who);
    FP8_TRY(check_device(who));
    SideStream *side = nullptr;
    FP8_TRY(side_stream(who, &side));
    // with timing events everything stays on `s`, so consecutive events
    // bracket one kernel each
    const bool overlap = events == nullptr;
    cudaStream_t s2 = overlap ? side->stream : s;

    int ev = 0;
    auto mark = [&](cudaStream_t on) -> fp8_status {
        if (events == nullptr) return FP8_OK;
        return cuda_status(cudaEventRecord(events[ev++], on), who);
    };
    float *d = m->dev;
    FP8_TRY(fp8_state_step(step_count, m->interval, m, 1, s));
    // zeroed by a kernel (programmatic dependent launch), not a memset: a memset
    // between the previous step's last kernel and this step's first would break
    // their launch overlap (measured: 174.2 -> 172.0-172.7 us per 4096^3 step)
    FP8_TRY(cuda_status(launch_zero_f32(io->amax, 3, s), who));
    // forward: X (lagged x scale, q only) and W (q, and qt for a forward-only
    // step) in one launch, which also keeps the x scale fprop must use
    FP8_TRY(mark(s));
    DelayedQuantJob jx{io->x, M, K, d + FP8_META_X_SCALE_INV, io->xq,
                       save_x ? io->xqt : nullptr, io->amax + 0};
    // with a backward, Wqᵀ (only dgrad reads it) comes from the backward
    // launch as the byte transpose of Wq, off the path to fprop: the
    // forward launch then moves 98 MB instead of 117 at 4096^3
    DelayedQuantJob jw{io->w, N, K, d + FP8_META_SCALE_INV, io->wq, bwd ? nullptr : io->wqt,
                       io->amax + 1};
    // W's tiles take the launch's first CTAs and X's (q only) its last, so
    // the partly filled last wave holds the cheaper tiles
    FP8_TRY(cuda_status(launch_quantize_delayed_pair(jw, jx, s, d + FP8_META_X_SCALE,
                                                     d + FP8_META_X_SCALE_FWD),
                        who));
    if (overlap) {  // fork: the state update and the backward quantisation
        FP8_TRY(cuda_status(cudaEventRecord(side->fork, s), who));
        FP8_TRY(cuda_status(cudaStreamWaitEvent(s2, side->fork, 0), who));
    }
    FP8_TRY(mark(s));
    FP8_TRY(fp8_linear_fprop(io->xq, d + FP8_META_X_SCALE_FWD, io->wq, d + FP8_META_SCALE, M, N,
                             K, FP8_RECIPE_DELAYED, io->bias, io->y, s));
    // record(amax_w) and the lag update of the x scale, one launch
    FP8_TRY(mark(s2));
    FP8_TRY(cuda_status(launch_meta_fwd(d, m->idx, io->amax + 0, io->amax + 1, s2), who));
    m->idx = (m->idx + 1) % m->interval;
    if (bwd) {
        // backward: G (q and qt), X again, transposed, with the updated
        // scale, and Wqᵀ from Wq's bytes; the launch keeps the g scale the
        // backward GEMMs must use, so
        // the lag update of the g scale runs right after it, off the GEMMs'
        // critical path
        FP8_TRY(mark(s2));
        DelayedQuantJob jg{io->g, M, N, d + FP8_META_G_SCALE_INV, io->gq, io->gqt, io->amax + 2};
        // X again, transposed, with the just-updated scale (none when the
        // forward kept its Xqᵀ)
        DelayedQuantJob jxt{io->x, save_x ? 0 : M, K, d + FP8_META_X_SCALE_INV, nullptr, io->xqt,
                            nullptr};
        jg.colsum = io->dbias != nullptr ? io->dbias_workspace : nullptr;  // G's column sums
        const ByteTransposeJob wt{io->wq, N, K, io->wqt};  // Wqᵀ for dgrad
        FP8_TRY(cuda_status(launch_quantize_delayed_pair(jg, jxt, s2, d + FP8_META_G_SCALE,
                                                         d + FP8_META_G_SCALE_BWD, &wt),
                            who));
        if (io->dbias != nullptr)
            FP8_TRY(cuda_status(launch_colsum_reduce(io->dbias_workspace, M, N, io->dbias, s2),
                                who));
        FP8_TRY(mark(s2));
        FP8_TRY(fp8_meta_record(m, FP8_SLOT_G, io->amax + 2, s2));
    }
    if (overlap) {  // join
        FP8_TRY(cuda_status(cudaEventRecord(side->join, s2), who));
        FP8_TRY(cuda_status(cudaStreamWaitEvent(s, side->join, 0), who));
    }
    if (bwd) {
        const float *gs = d + FP8_META_G_SCALE_BWD;
        const float *xs = d + (save_x ? FP8_META_X_SCALE_FWD : FP8_META_X_SCALE);
        FP8_TRY(mark(s));
        if (io->dx != nullptr && io->dw != nullptr) {
            // both backward GEMMs in one launch (they share its waves)
            FP8_TRY(fp8_linear_dgrad_wgrad(io->gq, io->gqt, gs, io->wqt, d + FP8_META_SCALE,
                                           io->xqt, xs, M, N, K, FP8_RECIPE_DELAYED, io->dx,
                                           io->dw, s));
            FP8_TRY(mark(s));
        } else {
            if (io->dx != nullptr)
                FP8_TRY(fp8_linear_dgrad(io->gq, gs, io->wqt, d + FP8_META_SCALE, M, N, K,
                                         FP8_RECIPE_DELAYED, io->dx, s));
            FP8_TRY(mark(s));
            if (io->dw != nullptr)
                FP8_TRY(fp8_linear_wgrad(io->gqt, gs, io->xqt, xs, M, N, K, FP8_RECIPE_DELAYED,
                                         io->dw, s));
        }
    }
    while (events != nullptr && ev < FP8_STEP_NEVENTS) FP8_TRY(mark(s));
    return FP8_OK;
}

fp8_status fp8_linear_fprop_dynamic_small(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N,
                                          int64_t K, const uint16_t *bias, float *scales,
                                          float *amax, uint8_t *xq, uint8_t *wq, uint16_t *y,
                                          cudaStream_t s) {
    const char *who = "fp8_linear_fprop_dynamic_small";
    if (M <= 0 || N <= 0 || K <= 0)
        return fail(FP8_ERR_SHAPE, "%s: bad shape [M=%lld, N=%lld, K=%lld]", who, (long long)M,
                    (long long)N, (long long)K);
    FP8_TRY(check_dim16(who, "M", M, 16));
    FP8_TRY(check_dim16(who, "N", N, 16));
    FP8_TRY(check_dim16(who, "K", K, 16));
    if (!linear_small_fits(M, N, K))
        return fail(FP8_ERR_UNSUPPORTED,
                    "%s: [M=%lld, N=%lld, K=%lld] is larger than one tile (M <= 128, N <= 256, "
                    "K <= 512); use the quantisers and fp8_linear_fprop",
                    who, (long long)M, (long long)N, (long long)K);
    FP8_NEED(x, who);
    FP8_NEED(w, who);
    FP8_NEED(scales, who);
    FP8_NEED(y, who);
    FP8_ALIGN(x, who);
    FP8_ALIGN(w, who);
    FP8_ALIGN(xq, who);
    FP8_ALIGN(wq, who);
    FP8_ALIGN(y, who);
    FP8_TRY(check_device(who));
    return cuda_status(
        launch_linear_small_dynamic(x, w, M, N, K, bias, scales, amax, xq, wq, y, s), who);
}

fp8_status fp8_linear_step_dynamic(const fp8_linear_step_io *io, float *scales, void *workspace,
                                   int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    const char *who = "fp8_linear_step_dynamic";
    FP8_NEED(io, who);
    FP8_NEED(scales, who);
    FP8_NEED(workspace, who);
    if (M <= 0 || N <= 0 || K <= 0 || M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF)
        return fail(FP8_ERR_SHAPE, "%s: bad shape [M=%lld, N=%lld, K=%lld]", who, (long long)M,
                    (long long)N, (long long)K);
    FP8_TRY(check_dim16(who, "M", M, 16));
    FP8_TRY(check_dim16(who, "N", N, 16));
    FP8_TRY(check_dim16(who, "K", K, 16));
    const bool bwd = io->g != nullptr;
    FP8_NEED(io->x, who);
    FP8_NEED(io->w, who);
    FP8_NEED(io->xq, who);
    FP8_NEED(io->wq, who);
    FP8_NEED(io->amax, who);
    FP8_NEED(io->y, who);
    if (bwd) {
        FP8_NEED(io->wqt, who);
        FP8_NEED(io->gq, who);
        FP8_NEED(io->gqt, who);
        FP8_NEED(io->xqt, who);
    }
    if (io->dbias != nullptr)
        return fail(FP8_ERR_UNSUPPORTED, "%s: dbias is fused into the delayed-scaling step only",
                    who);
    if (io->flags != 0) return fail(FP8_ERR_SHAPE, "%s: unknown flags 0x%x", who, (unsigned)io->flags);
    const void *ptrs[] = {io->x, io->w, io->g, io->bias, io->xq, io->xqt, io->wq, io->wqt,
                          io->gq, io->gqt, io->y, io->dx, io->dw, workspace};
    for (const void *p : ptrs)
        if (p != nullptr && !aligned16(p))
            return fail(FP8_ERR_ALIGNMENT, "%s: a buffer is not 16-byte aligned", who);
    FP8_TRY(check_device(who));
    unsigned int *ws = static_cast<unsigned int *>(workspace);
    const size_t wsw = kFusedWorkspaceBytes / sizeof(unsigned int);
    // X and W: current scaling, each in one launch (q, and qᵀ for the backward)
    FP8_TRY(cuda_status(launch_quantize_fused_dynamic(io->x, M, K, scales + 0, scales + 1, io->xq,
                                                      bwd ? io->xqt : nullptr, io->amax + 0, ws,
                                                      s),
                        who));
    FP8_TRY(cuda_status(launch_quantize_fused_dynamic(io->w, N, K, scales + 2, scales + 3, io->wq,
                                                      bwd ? io->wqt : nullptr, io->amax + 1,
                                                      ws + wsw, s),
                        who));
    FP8_TRY(fp8_linear_fprop(io->xq, scales + 0, io->wq, scales + 2, M, N, K, FP8_RECIPE_DYNAMIC,
                             io->bias, io->y, s));
    if (!bwd) return FP8_OK;
    FP8_TRY(cuda_status(launch_quantize_fused_dynamic(io->g, M, N, scales + 4, scales + 5, io->gq,
                                                      io->gqt, io->amax + 2, ws + 2 * wsw, s),
                        who));
    if (io->dx != nullptr && io->dw != nullptr)
        return fp8_linear_dgrad_wgrad(io->gq, io->gqt, scales + 4, io->wqt, scales + 2, io->xqt,
                                      scales + 0, M, N, K, FP8_RECIPE_DYNAMIC, io->dx, io->dw, s);
    if (io->dx != nullptr)
        FP8_TRY(fp8_linear_dgrad(io->gq, scales + 4, io->wqt, scales + 2, M, N, K,
                                 FP8_RECIPE_DYNAMIC, io->dx, s));
    if (io->dw != nullptr)
        FP8_TRY(fp8_linear_wgrad(io->gqt, scales + 4, io->xqt, scales + 0, M, N, K,
                                 FP8_RECIPE_DYNAMIC, io->dw, s));
    return FP8_OK;
}

fp8_status fp8_linear_step_block(const fp8_linear_step_io *io, const fp8_block_step_scales *sc,
                                 int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    const char *who = "fp8_linear_step_block";
    FP8_NEED(io, who);
    FP8_NEED(sc, who);
    if (M <= 0 || N <= 0 || K <= 0 || M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF)
        return fail(FP8_ERR_SHAPE, "%s: bad shape [M=%lld, N=%lld, K=%lld]", who, (long long)M,
                    (long long)N, (long long)K);
    FP8_TRY(check_dim16(who, "M", M, 128));
    FP8_TRY(check_dim16(who, "N", N, 128));
    FP8_TRY(check_dim16(who, "K", K, 128));
    const bool bwd = io->g != nullptr;
    FP8_NEED(io->x, who);
    FP8_NEED(io->w, who);
    FP8_NEED(io->xq, who);
    FP8_NEED(io->wq, who);
    FP8_NEED(io->y, who);
    if (bwd) {
        FP8_NEED(io->xqt, who);
        FP8_NEED(io->wqt, who);
        FP8_NEED(io->gq, who);
        FP8_NEED(io->gqt, who);
    }
    if (io->bias != nullptr || io->dbias != nullptr || io->flags != 0)
        return fail(FP8_ERR_UNSUPPORTED, "%s: bias, dbias and flags are not supported", who);
    const float *scs[] = {sc->x_scale, sc->x_scale_inv, sc->x_scale_t, sc->x_scale_inv_t,
                          sc->w_scale, sc->w_scale_inv, sc->g_scale, sc->g_scale_inv,
                          sc->g_scale_t, sc->g_scale_inv_t};
    for (const float *p : scs) {
        if (p == nullptr) return fail(FP8_ERR_NULL, "%s: a scale array is NULL", who);
        if (!aligned16(p))  // the block GEMMs stage scales with 16-byte copies
            return fail(FP8_ERR_ALIGNMENT, "%s: a scale array is not 16-byte aligned", who);
    }
    const void *ptrs[] = {io->x, io->w, io->g, io->xq, io->xqt, io->wq, io->wqt,
                          io->gq, io->gqt, io->y, io->dx, io->dw};
    for (const void *p : ptrs)
        if (p != nullptr && !aligned16(p))
            return fail(FP8_ERR_ALIGNMENT, "%s: a buffer is not 16-byte aligned", who);
    FP8_TRY(check_device(who));
    float *amax = io->amax;
    FP8_TRY(cuda_status(launch_quantize_transpose(io->x, M, K, 3, sc->x_scale, sc->x_scale_inv,
                                                  io->xq, bwd ? io->xqt : nullptr, sc->x_scale_t,
                                                  sc->x_scale_inv_t, amax, s),
                        who));
    FP8_TRY(cuda_status(launch_quantize_transpose(io->w, N, K, 2, sc->w_scale, sc->w_scale_inv,
                                                  io->wq, bwd ? io->wqt : nullptr, nullptr,
                                                  nullptr, amax ? amax + 1 : nullptr, s),
                        who));
    FP8_TRY(fp8_linear_fprop(io->xq, sc->x_scale, io->wq, sc->w_scale, M, N, K,
                             FP8_RECIPE_BLOCK, nullptr, io->y, s));
    if (!bwd) return FP8_OK;
    FP8_TRY(cuda_status(launch_quantize_transpose(io->g, M, N, 3, sc->g_scale, sc->g_scale_inv,
                                                  io->gq, io->gqt, sc->g_scale_t,
                                                  sc->g_scale_inv_t, amax ? amax + 2 : nullptr, s),
                        who));
    if (io->dx != nullptr)
        FP8_TRY(fp8_linear_dgrad(io->gq, sc->g_scale, io->wqt, sc->w_scale, M, N, K,
                                 FP8_RECIPE_BLOCK, io->dx, s));
    if (io->dw != nullptr)
        FP8_TRY(fp8_linear_wgrad(io->gqt, sc->g_scale_t, io->xqt, sc->x_scale_t, M, N, K,
                                 FP8_RECIPE_BLOCK, io->dw, s));
    return FP8_OK;
}

int64_t fp8_pad_multiple(int32_t cp_size, int32_t tp_size) {
    if (cp_size < 1 || tp_size < 1 || (int64_t)cp_size * tp_size > (1 << 20)) return -1;
    return 16 * (int64_t)cp_size * tp_size;
}

int64_t fp8_padded_seq_len(int64_t batch, int64_t seq, int32_t cp_size, int32_t tp_size) {
    if (batch < 1 || seq < 0 || cp_size < 1 || tp_size < 1) return -1;
    const int64_t r = (int64_t)cp_size * tp_size;
    if (r > (1 << 20)) return -1;
    auto gcd = [](int64_t a, int64_t b) {
        while (b) {
            const int64_t t = a % b;
            a = b;
            b = t;
        }
        return a;
    };
    // T' % r == 0 and batch*T' % (16 r) == 0: T' a multiple of lcm(r, 16r / gcd(batch, 16r))
    const int64_t step_b = 16 * r / gcd(batch % (16 * r), 16 * r);
    const int64_t L = r / gcd(r, step_b) * step_b;
    return (seq + L - 1) / L * L;
}

fp8_status fp8_pad_tokens_bshd(const uint16_t *x, int64_t batch, int64_t seq, int64_t hidden,
                               int32_t cp_size, int32_t tp_size, uint16_t *out,
                               int64_t *padded_seq, cudaStream_t s) {
    const char *who = "fp8_pad_tokens_bshd";
    const int64_t tp = fp8_padded_seq_len(batch, seq, cp_size, tp_size);
    if (tp < 0 || hidden < 0)
        return fail(FP8_ERR_SHAPE, "%s: batch=%lld seq=%lld hidden=%lld cp=%d tp=%d", who,
                    (long long)batch, (long long)seq, (long long)hidden, cp_size, tp_size);
    if (hidden % 8 != 0)
        return fail(FP8_ERR_ALIGNMENT, "%s: hidden=%lld must be a multiple of 8", who,
                    (long long)hidden);
    if (padded_seq != nullptr) *padded_seq = tp;
    if (batch * tp * hidden > 0) FP8_NEED(out, who);
    if (batch * seq * hidden > 0) FP8_NEED(x, who);
    FP8_ALIGN(x, who);
    FP8_ALIGN(out, who);
    if (x != nullptr && out != nullptr && batch * seq * hidden > 0) {
        const char *xb = reinterpret_cast<const char *>(x), *ob = reinterpret_cast<const char *>(out);
        if (xb < ob + batch * tp * hidden * 2 && ob < xb + batch * seq * hidden * 2)
            return fail(FP8_ERR_SHAPE, "%s: x and out overlap", who);
    }
    FP8_TRY(check_device(who));
    return cuda_status(launch_pad_bshd(x, batch, seq, hidden, tp, out, s), who);
}

fp8_status fp8_multi_amax_scales(const uint16_t *const *w, const int64_t *numel, int32_t n,
                                 float *amax, float *scale, float *scale_inv, cudaStream_t s) {
    const char *who = "fp8_multi_amax_scales";
    if (n < 0) return fail(FP8_ERR_SHAPE, "%s: n=%d", who, n);
    if (n == 0) return FP8_OK;
    FP8_NEED(w, who);
    FP8_NEED(numel, who);
    FP8_NEED(amax, who);
    FP8_NEED(scale, who);
    FP8_NEED(scale_inv, who);
    for (int32_t i = 0; i < n; ++i) {
        if (numel[i] < 0)
            return fail(FP8_ERR_SHAPE, "%s: numel[%d]=%lld", who, i, (long long)numel[i]);
        if (numel[i] > 0 && w[i] == nullptr)
            return fail(FP8_ERR_NULL, "%s: w[%d] is NULL", who, i);
        if (!aligned16(w[i]))
            return fail(FP8_ERR_ALIGNMENT, "%s: w[%d] is not 16-byte aligned", who, i);
    }
    FP8_TRY(check_device(who));
    return cuda_status(launch_multi_amax_scales(w, numel, n, amax, scale, scale_inv, s), who);
}

int64_t fp8_padded_rows(int64_t rows, int64_t multiple) {
    if (rows < 0 || multiple < 1) return -1;
    return (rows + multiple - 1) / multiple * multiple;
}

fp8_status fp8_pad_tokens(const uint16_t *x, int64_t rows, int64_t cols, int64_t multiple,
                          uint16_t *out, int64_t *padded_rows, cudaStream_t s) {
    const char *who = "fp8_pad_tokens";
    if (rows < 0 || cols < 0 || multiple < 1)
        return fail(FP8_ERR_SHAPE, "%s: rows=%lld cols=%lld multiple=%lld", who, (long long)rows,
                    (long long)cols, (long long)multiple);
    const int64_t padded = fp8_padded_rows(rows, multiple);
    if (padded_rows != nullptr) *padded_rows = padded;
    if (padded * cols > 0) FP8_NEED(out, who);
    if (rows * cols > 0) FP8_NEED(x, who);
    FP8_ALIGN(x, who);
    FP8_ALIGN(out, who);
    if (x != nullptr && out != nullptr && rows * cols > 0) {
        const char *xb = reinterpret_cast<const char *>(x), *ob = reinterpret_cast<const char *>(out);
        if (xb < ob + padded * cols * 2 && ob < xb + rows * cols * 2)
            return fail(FP8_ERR_SHAPE, "%s: x and out overlap", who);
    }
    FP8_TRY(check_device(who));
    return cuda_status(launch_pad_rows(x, rows, cols, padded, out, s), who);
}

fp8_status fp8_inject_launch_failures(int32_t n) {
    if (n < 0) return fail(FP8_ERR_SHAPE, "fp8_inject_launch_failures: n=%d", n);
    tl_fail_launches = n;
    return FP8_OK;
}

fp8_status fp8_check_device_status(cudaStream_t s) {
    const char *who = "fp8_check_device_status";
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e, who);
    unsigned int v = 0;
    e = read_and_clear_device_status(&v);
    if (e != cudaSuccess) return cuda_status(e, who);
    if (v == 0) return FP8_OK;
    return fail(FP8_ERR_TIMEOUT, "%s: a bounded wait ran out (status bits 0x%x: %s%s%s%s%s)", who, v,
                (v & kStatusTimeoutTma) ? "tma " : "", (v & kStatusTimeoutMma) ? "mma " : "",
                (v & kStatusTimeoutEpilogue) ? "epilogue " : "",
                (v & kStatusTimeoutSelftest) ? "selftest " : "",
                (v & kStatusTimeoutBarrier) ? "grid-barrier" : "");
}

uint64_t fp8_set_wait_limit_ns(uint64_t limit_ns) {
    const uint64_t v = limit_ns == 0 ? kDefaultWaitLimitNs : limit_ns;
    return g_wait_limit_ns.exchange(v, std::memory_order_relaxed);
}

fp8_status fp8_selftest_wait_timeout(uint32_t timeout_us, cudaStream_t s) {
    const char *who = "fp8_selftest_wait_timeout";
    if (timeout_us < 1 || timeout_us > 1000000)
        return fail(FP8_ERR_SHAPE, "%s: timeout_us=%u outside 1..1000000", who, timeout_us);
    FP8_TRY(check_device(who));
    return cuda_status(launch_selftest_wait(timeout_us, s), who);
}

}  // extern "C"
