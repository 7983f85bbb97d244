// Delayed-scaling state kernels: one thread each, launched on the caller's
// stream so the host never waits for a scale.  Semantics follow the AstrAI
// page "astrai/extension/fp8_state.py": FP8TensorMeta.__init__ (all ones),
// record (ring push), refresh (window max, skipped when not > 0) and
// _update_delayed_scale (clamp to 1e-12, then amax/448 and 448/amax).
#include "common.cuh"
#include "kernels.h"

namespace fp8 {

namespace {

__device__ unsigned int g_device_status = 0;

__global__ void meta_init_kernel(float *dev, int interval) {
    pdl_wait_prior();
    pdl_allow_next();
    for (int i = threadIdx.x; i < FP8_META_HISTORY + interval; i += blockDim.x)
        dev[i] = (i == 6 || i == 7) ? 0.0f : 1.0f;
}

__global__ void meta_copy_kernel(float *dst, const float *src) {
    pdl_wait_prior();
    pdl_allow_next();
    *dst = *src;
}

__global__ void meta_lag_kernel(float *scale, float *scale_inv, const float *amax) {
    pdl_wait_prior();
    pdl_allow_next();
    float s, si;
    scales_from_amax(*amax, s, si);
    *scale = s;
    *scale_inv = si;
}

__global__ void zero_f32_kernel(float *p, int64_t n) {
    pdl_wait_prior();
    pdl_allow_next();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) p[i] = 0.0f;
}

__global__ void meta_fwd_kernel(float *dev, int idx, const float *amax_x, const float *amax_w) {
    pdl_wait_prior();
    pdl_allow_next();
    dev[FP8_META_HISTORY + idx] = *amax_w;
    float s, si;
    scales_from_amax(*amax_x, s, si);
    dev[FP8_META_X_SCALE] = s;
    dev[FP8_META_X_SCALE_INV] = si;
}

__global__ void meta_refresh_kernel(float *dev, int interval) {
    pdl_wait_prior();
    pdl_allow_next();
    const float *h = dev + FP8_META_HISTORY;
    float m = h[0];
    for (int i = 1; i < interval; ++i) {
        const float v = h[i];
        if (isnan(v) || v > m) m = isnan(m) ? m : v;  // a NaN anywhere stays
    }
    if (m > 0.0f) {  // false for NaN and for 0: keep the old scale
        dev[FP8_META_SCALE] = __fdiv_rn(m, 448.0f);
        dev[FP8_META_SCALE_INV] = __fdiv_rn(448.0f, m);
    }
}

__global__ void selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)  // nothing ever arrives on `bar`
        mbar_wait_bounded(&bar, 0, &abort_flag, limit_ns, kStatusTimeoutSelftest, &g_device_status);
}

}  // namespace

unsigned int *device_status_word() {
    // one address per device, looked up once with that device current
    static unsigned int *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}

cudaError_t read_and_clear_device_status(unsigned int *out) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_device_status, sizeof *out);
    if (e != cudaSuccess || *out == 0) return e;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
}

cudaError_t launch_meta_init(float *dev, int interval, cudaStream_t s) {
    return launch_pdl(meta_init_kernel, 1, 128, 0, s, dev, interval);
}

cudaError_t launch_meta_copy(float *dst, const float *src, cudaStream_t s) {
    return launch_pdl(meta_copy_kernel, 1, 1, 0, s, dst, src);
}

cudaError_t launch_meta_lag(float *scale, float *scale_inv, const float *amax, cudaStream_t s) {
    return launch_pdl(meta_lag_kernel, 1, 1, 0, s, scale, scale_inv, amax);
}

cudaError_t launch_meta_fwd(float *dev, int idx, const float *amax_x, const float *amax_w,
                            cudaStream_t s) {
    return launch_pdl(meta_fwd_kernel, 1, 1, 0, s, dev, idx, amax_x, amax_w);
}

cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int threads = n < 256 ? 32 : 256;
    return launch_pdl(zero_f32_kernel, (unsigned)((n + threads - 1) / threads), threads, 0, s, p, n);
}

cudaError_t launch_meta_refresh(float *dev, int interval, cudaStream_t s) {
    return launch_pdl(meta_refresh_kernel, 1, 1, 0, s, dev, interval);
}

cudaError_t launch_selftest_wait(uint32_t timeout_us, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>((uint64_t)timeout_us * 1000ull);
    return cudaGetLastError();
}

}  // namespace fp8
