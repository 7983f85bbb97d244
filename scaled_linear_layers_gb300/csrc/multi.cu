// Many tensors in one pass: the current-scaling amax and scales of a list of
// weights (run after an optimizer step, before their fp8 casts), and the
// per-sequence token padding of a [B, T, H] batch.
#include "common.cuh"
#include "kernels.h"
#include "qtile.cuh"

namespace fp8 {

namespace {

constexpr int kMultiMax = 64;                   // tensors per launch
constexpr int kMultiThreads = 256;
constexpr int64_t kMultiChunk = kMultiThreads * 8 * 8;  // elements per CTA

struct MultiArgs {
    const uint16_t *w[kMultiMax];
    int64_t numel[kMultiMax];
    int cta_start[kMultiMax + 1];  // CTAs of tensor i: [cta_start[i], cta_start[i+1])
    int n;
    float *amax;                   // [n] (this launch's slice), zero on entry
};

// CTA b takes one 64K-element chunk of one tensor: 16-byte loads for the
// chunk's whole vectors, element loads for a tensor's last few elements,
// |x| reduced on bf16 bit patterns, one atomicMax per CTA.
__global__ void __launch_bounds__(kMultiThreads) multi_amax_kernel(const MultiArgs a) {
    __shared__ uint32_t red[kMultiThreads / 32];
    pdl_wait_prior();
    pdl_allow_next();
    const int b = blockIdx.x;
    int i = 0;
    while (i + 1 < a.n && a.cta_start[i + 1] <= b) ++i;
    const int64_t numel = a.numel[i];
    const int64_t lo = (int64_t)(b - a.cta_start[i]) * kMultiChunk;
    const int64_t hi = min(numel, lo + kMultiChunk);
    const uint16_t *w = a.w[i];
    uint32_t m = 0;
    const int64_t vhi = lo + ((hi - lo) & ~int64_t(7));  // end of whole 8-element vectors
    for (int64_t e = lo + 8 * threadIdx.x; e < vhi; e += 8 * kMultiThreads)
        m = max(m, absmax_bits8(ldg_nc_v4(w + e)));
    for (int64_t e = vhi + threadIdx.x; e < hi; e += kMultiThreads) {
        uint32_t v = w[e] & 0x7FFFu;
        m = max(m, v);
    }
    m = block_max_u32(m, red);
    if (threadIdx.x == 0 && m != 0)
        atomicMax(reinterpret_cast<unsigned int *>(a.amax + i), bf16bits_to_f32bits(m));
}

__global__ void multi_scales_kernel(const float *amax, float *scale, float *scale_inv, int n) {
    pdl_wait_prior();
    pdl_allow_next();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float s, si;
    scales_from_amax(amax[i], s, si);
    scale[i] = s;
    scale_inv[i] = si;
}

// out [B, Tp, H] = x [B, T, H] with rows T..Tp-1 of every sequence zero;
// one 16-byte vector (8 bf16) per thread and step, H a multiple of 8.
__global__ void __launch_bounds__(256) pad_bshd_kernel(const uint4 *__restrict__ x, int64_t T,
                                                       int64_t Tp, int64_t hv, int64_t total,
                                                       uint4 *__restrict__ out) {
    pdl_wait_prior();
    pdl_allow_next();
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t c = v % hv, r = v / hv;  // r = b * Tp + t
        const int64_t t = r % Tp, bb = r / Tp;
        out[v] = t < T ? x[(bb * T + t) * hv + c] : make_uint4(0, 0, 0, 0);
    }
}

}  // namespace

cudaError_t launch_multi_amax_scales(const uint16_t *const *w, const int64_t *numel, int n,
                                     float *amax, float *scale, float *scale_inv,
                                     cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    cudaError_t e = launch_zero_f32(amax, n, s);
    if (e != cudaSuccess) return e;
    for (int base = 0; base < n; base += kMultiMax) {
        MultiArgs a;
        a.n = n - base < kMultiMax ? n - base : kMultiMax;
        a.amax = amax + base;
        int64_t ctas = 0;
        for (int i = 0; i < a.n; ++i) {
            a.w[i] = w[base + i];
            a.numel[i] = numel[base + i];
            a.cta_start[i] = (int)ctas;
            // an empty tensor still owns one CTA (it finds nothing)
            ctas += numel[base + i] > 0 ? (numel[base + i] + kMultiChunk - 1) / kMultiChunk : 1;
        }
        a.cta_start[a.n] = (int)ctas;
        if (ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
        e = launch_pdl(multi_amax_kernel, (int)ctas, kMultiThreads, 0, s, a);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(multi_scales_kernel, (n + 255) / 256, 256, 0, s, (const float *)amax, scale,
                      scale_inv, n);
}

cudaError_t launch_pad_bshd(const uint16_t *x, int64_t B, int64_t T, int64_t H, int64_t Tp,
                            uint16_t *out, cudaStream_t s) {
    const int64_t hv = H / 8, total = B * Tp * hv;
    if (total == 0) return cudaSuccess;
    int64_t grid = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (grid > cap) grid = cap;
    return launch_pdl(pad_bshd_kernel, (int)grid, 256, 0, s, reinterpret_cast<const uint4 *>(x), T,
                      Tp, hv, total, reinterpret_cast<uint4 *>(out));
}

}  // namespace fp8
