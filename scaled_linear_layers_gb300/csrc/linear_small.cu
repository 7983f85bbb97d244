// Current-scaling fprop of a small linear in one launch.
//
// For problems that fit one output tile (M <= 128, N <= 256, K <= 512) the
// work is a few microseconds of device time, and three launches (amax and
// cast of X, the same for W, the GEMM) cost more than the arithmetic.  One
// launch of a cluster of C CTAs (C = 8, 4, 2 or 1: the largest with N/C a
// multiple of 16) does it all, CTA r owning W's rows [r*N/C, (r+1)*N/C) and
// the output columns they give:
//   * every thread loads its 16-element chunks of X and of its CTA's W rows
//     once, all loads issued before the first use (up to kCacheX + kCacheW
//     chunks per thread stay in registers; any further ones are read again
//     for the cast);
//   * each CTA takes the amax of all of X (the same value in every CTA) and
//     of its W rows; the W partial maxima are exchanged through distributed
//     shared memory between two cluster barriers, so every CTA has both
//     amaxes and derives both scale pairs;
//   * the casts go straight into shared memory in the layout the tensor core
//     reads (K-major, 128-byte rows, 16-byte chunks XOR-swizzled by row % 8
//     within 8-row groups of 1024 bytes: what a TMA copy with 128-byte
//     swizzling produces), then a proxy fence;
//   * one thread issues tcgen05.mma kind::f8f6f4 (M = 128, N = N/C, K = 32 per
//     instruction) into TMEM, and the epilogue writes acc * fl32(s_x * s_w)
//     (+ bias) rounded to bf16.
// Rows past M and chunks past K are zero in shared memory, so the MMA shape
// is fixed.  The arithmetic is that of the three-call path (same casts, same
// MMA sequence per 128-byte block, same epilogue), so the outputs agree bit
// for bit.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "qtile.cuh"

namespace fp8 {

extern std::atomic<uint64_t> g_wait_limit_ns;

namespace {

constexpr int kThreads = 512;
constexpr int kCacheX = 4, kCacheW = 4;  // 16-element chunks per thread kept in registers
constexpr int kRowsA = 128, kMaxRowsB = 256;
constexpr int kBoxA = kRowsA * 128;  // bytes of A per 128-byte K box
constexpr int kMaxCluster = 8;

struct SmallArgs {
    const uint16_t *x, *w, *bias;
    int M, N, K;
    float *scales;  // x scale, x scale_inv, w scale, w scale_inv
    float *amax;    // amax of x, of w (nullable)
    uint8_t *xq, *wq;  // nullable
    uint16_t *y;
    uint64_t wait_limit_ns;
    unsigned int *status;
};

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// Row and 16-byte chunk of chunk `id` of a matrix with `cpr` chunks per row;
// the row is floor(id / cpr) as a multiply-high by inv = ceil(2^32 / cpr),
// exact for id < 2^16 and 2 <= cpr <= 32 (the error term id * (inv -
// 2^32/cpr) / 2^32 stays below 2^-16, under the 1/cpr gap to the next
// integer); one chunk per row (inv would be 2^32) is the row itself.
__device__ __forceinline__ void chunk_rc(int id, int cpr, uint32_t inv, int &r, int &c) {
    r = cpr == 1 ? id : (int)__umulhi((uint32_t)id, inv);
    c = id - r * cpr;
}

// Byte offset of 16-byte chunk `c` (of a row's K bytes) of row `r` in the
// swizzled operand layout.
__device__ __forceinline__ uint32_t swz_offset(int r, int c, int box_bytes) {
    return (uint32_t)((c >> 3) * box_bytes + (r >> 3) * 1024 + (r & 7) * 128 +
                      (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void load_chunk(const uint16_t *__restrict__ x, int K, int r, int c,
                                           uint4 (&v)[2]) {
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)r * K + (c << 4));
    v[0] = ldg_nc_v4(src);
    v[1] = ldg_nc_v4(src + 1);
}

// Casts one chunk with scale_inv `si` into the swizzled shared tile (row r of
// the tile) and to global q at row qr (q nullable).
__device__ __forceinline__ void cast_chunk(const uint4 (&v)[2], int K, int r, int c, int qr,
                                           float si, uint8_t *s, int box_bytes,
                                           uint8_t *__restrict__ q) {
    const uint4 o = make_uint4(quant4(v[0].x, v[0].y, si), quant4(v[0].z, v[0].w, si),
                               quant4(v[1].x, v[1].y, si), quant4(v[1].z, v[1].w, si));
    if (q != nullptr) *reinterpret_cast<uint4 *>(q + (int64_t)qr * K + (c << 4)) = o;
    *reinterpret_cast<uint4 *>(s + swz_offset(r, c, box_bytes)) = o;
}

__device__ __forceinline__ uint32_t chunk_absmax(const uint4 (&v)[2]) {
    return max(absmax_bits8(v[0]), absmax_bits8(v[1]));
}

__global__ void __launch_bounds__(kThreads, 1) linear_small_dynamic_kernel(const SmallArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int C = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
    const int nb = p.N / C;          // W rows (output columns) of this CTA, a multiple of 16
    const int w0 = rank * nb;        // first of them
    const int box_b = nb * 128;      // bytes of B per 128-byte K box
    const int nkb = (p.K + 127) / 128;
    uint8_t *sA = smem;
    uint8_t *sB = smem + nkb * kBoxA;
    uint64_t *done = reinterpret_cast<uint64_t *>(sB + nkb * box_b);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    __shared__ uint32_t red[kThreads / 32];
    __shared__ uint32_t w_partial;   // this CTA's W maximum, read by the whole cluster
    __shared__ float s_si[2], s_s[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tmem_cols = nb <= 32 ? 32u : nb <= 64 ? 64u : nb <= 128 ? 128u : 256u;

    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_wait_prior();
    pdl_allow_next();

    // zero both operand tiles (rows past M and chunks past K stay zero)
    {
        uint4 *z = reinterpret_cast<uint4 *>(smem);
        const int n16 = nkb * (kBoxA + box_b) / 16;
        for (int i = threadIdx.x; i < n16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    }

    // every thread's chunks of X and of this CTA's W rows, loads first
    const int cpr = p.K >> 4;  // 16-element chunks per row
    const uint32_t inv = cpr > 1 ? (uint32_t)((0x100000000ull + cpr - 1) / cpr) : 0u;
    const int ux = p.M * cpr, uw = nb * cpr;
    const uint16_t *wsl = p.w + (int64_t)w0 * p.K;
    uint4 xr[kCacheX][2], wr[kCacheW][2];
#pragma unroll
    for (int u = 0; u < kCacheX; ++u) {
        const int id = threadIdx.x + u * kThreads;
        int r, c;
        chunk_rc(id, cpr, inv, r, c);
        if (id < ux) load_chunk(p.x, p.K, r, c, xr[u]);
        else xr[u][0] = xr[u][1] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kCacheW; ++u) {
        const int id = threadIdx.x + u * kThreads;
        int r, c;
        chunk_rc(id, cpr, inv, r, c);
        if (id < uw) load_chunk(wsl, p.K, r, c, wr[u]);
        else wr[u][0] = wr[u][1] = make_uint4(0, 0, 0, 0);
    }
    uint32_t mx = 0, mw = 0;
#pragma unroll
    for (int u = 0; u < kCacheX; ++u) mx = max(mx, chunk_absmax(xr[u]));
#pragma unroll
    for (int u = 0; u < kCacheW; ++u) mw = max(mw, chunk_absmax(wr[u]));
    for (int id = threadIdx.x + kCacheX * kThreads; id < ux; id += kThreads) {
        int r, c;
        chunk_rc(id, cpr, inv, r, c);
        uint4 v[2];
        load_chunk(p.x, p.K, r, c, v);
        mx = max(mx, chunk_absmax(v));
    }
    for (int id = threadIdx.x + kCacheW * kThreads; id < uw; id += kThreads) {
        int r, c;
        chunk_rc(id, cpr, inv, r, c);
        uint4 v[2];
        load_chunk(wsl, p.K, r, c, v);
        mw = max(mw, chunk_absmax(v));
    }
    mx = block_max_u32(mx, red);
    __syncthreads();  // red is reused
    mw = block_max_u32(mw, red);
    if (threadIdx.x == 0) w_partial = mw;
    // every CTA's W maximum is in its shared memory before any CTA reads it
    cluster_sync_all();
    if (threadIdx.x == 0) {
        for (int q = 0; q < C; ++q)
            mw = max(mw, ld_shared_cluster_u32(mapa_shared(smem_u32(&w_partial), (uint32_t)q)));
        const float ax = __uint_as_float(mx << 16), aw = __uint_as_float(mw << 16);
        float sx, six, sw, siw;
        scales_from_amax(ax, sx, six);
        scales_from_amax(aw, sw, siw);
        s_si[0] = six;
        s_si[1] = siw;
        s_s[0] = sx;
        s_s[1] = sw;
        if (rank == 0) {
            p.scales[0] = sx;
            p.scales[1] = six;
            p.scales[2] = sw;
            p.scales[3] = siw;
            if (p.amax != nullptr) {
                p.amax[0] = ax;
                p.amax[1] = aw;
            }
        }
    }
    __syncthreads();  // also orders the zero fill before the casts

    // casts into the swizzled operand tiles: kept chunks from registers, the
    // rest read again (from L2); X's bytes go to global from rank 0 only
    const float six = s_si[0], siw = s_si[1];
    uint8_t *xq = rank == 0 ? p.xq : nullptr;
    uint8_t *wq = p.wq;
#pragma unroll
    for (int u = 0; u < kCacheX; ++u) {
        const int id = threadIdx.x + u * kThreads;
        int r, c;
        chunk_rc(id, cpr, inv, r, c);
        if (id < ux) cast_chunk(xr[u], p.K, r, c, r, six, sA, kBoxA, xq);
    }
#pragma unroll
    for (int u = 0; u < kCacheW; ++u) {
        const int id = threadIdx.x + u * kThreads;
        int r, c;
        chunk_rc(id, cpr, inv, r, c);
        if (id < uw) cast_chunk(wr[u], p.K, r, c, w0 + r, siw, sB, box_b, wq);
    }
    for (int id = threadIdx.x + kCacheX * kThreads; id < ux; id += kThreads) {
        int r, c;
        chunk_rc(id, cpr, inv, r, c);
        uint4 v[2];
        load_chunk(p.x, p.K, r, c, v);
        cast_chunk(v, p.K, r, c, r, six, sA, kBoxA, xq);
    }
    for (int id = threadIdx.x + kCacheW * kThreads; id < uw; id += kThreads) {
        int r, c;
        chunk_rc(id, cpr, inv, r, c);
        uint4 v[2];
        load_chunk(wsl, p.K, r, c, v);
        cast_chunk(v, p.K, r, c, w0 + r, siw, sB, box_b, wq);
    }
    // the tensor core reads shared memory through the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_f8_f32(kRowsA, (uint32_t)nb);
        for (int kb = 0; kb < nkb; ++kb) {
            const uint32_t a0 = smem_u32(sA + kb * kBoxA), b0 = smem_u32(sB + kb * box_b);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_f8(tmem_base, smem_desc_sw128(a0 + 32 * k), smem_desc_sw128(b0 + 32 * k),
                       idesc, (kb | k) != 0);
        }
        mma_commit(done);
    }

    // epilogue: warp w reads TMEM lanes (rows) 32*(w % 4) .. +31 and the
    // 16-column chunks j = w/4, w/4 + 4, ... of this CTA's nb columns; warps
    // whose rows lie wholly past M have nothing to write and skip the loads
    {
        const int quarter = warp & 3, cg = warp >> 2;
        if (quarter * 32 < p.M && cg * 16 < nb) {
            const bool ok = mbar_wait_bounded(done, 0, abort_flag, p.wait_limit_ns,
                                              kStatusTimeoutEpilogue, p.status);
            if (__all_sync(0xFFFFFFFFu, ok)) {
                tc_fence_after();
                const int row = quarter * 32 + lane;
                const float s = __fmul_rn(s_s[0], s_s[1]);
                uint16_t *drow = p.y + (int64_t)row * p.N + w0;
                for (int j = cg; j * 16 < nb; j += kThreads / 128) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(16 * j), r);
                    tmem_ld_wait();
                    if (row < p.M) {
                        const int col = 16 * j;
                        uint32_t packed[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float v0 = __fmul_rn(__uint_as_float(r[2 * e]), s);
                            float v1 = __fmul_rn(__uint_as_float(r[2 * e + 1]), s);
                            if (p.bias != nullptr) {
                                v0 = __fadd_rn(v0, __uint_as_float((uint32_t)p.bias[w0 + col + 2 * e] << 16));
                                v1 = __fadd_rn(v1, __uint_as_float((uint32_t)p.bias[w0 + col + 2 * e + 1] << 16));
                            }
                            packed[e] = pack_bf16x2(v0, v1);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(drow + col);
                        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    }
                }
            }
        }
    }

    if (threadIdx.x == 0) {  // the MMAs have completed before TMEM is freed
        volatile int no_abort = 0;
        mbar_wait_bounded(done, 0, &no_abort, 10000000ull, kStatusTimeoutMma, p.status);
    }
    tc_fence_before();
    // no CTA leaves (its shared memory with it) while another may still read
    // its W maximum
    cluster_sync_all();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base, tmem_cols);
}

// Cluster size: the largest of 8, 4, 2, 1 that leaves each CTA a multiple of
// 16 output columns.
int small_cluster(int64_t N) {
    for (int c = kMaxCluster; c > 1; c >>= 1)
        if ((N / 16) % c == 0) return c;
    return 1;
}

}  // namespace

bool linear_small_fits(int64_t M, int64_t N, int64_t K) {
    return M >= 1 && M <= kRowsA && N >= 1 && N <= kMaxRowsB && K >= 1 && K <= 512;
}

cudaError_t launch_linear_small_dynamic(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N,
                                        int64_t K, const uint16_t *bias, float *scales,
                                        float *amax, uint8_t *xq, uint8_t *wq, uint16_t *y,
                                        cudaStream_t s) {
    if (tl_fail_launches > 0) {
        --tl_fail_launches;
        return cudaErrorLaunchFailure;
    }
    const int C = small_cluster(N);
    const int nkb = (int)((K + 127) / 128);
    const size_t smem = 1024 + (size_t)nkb * (kBoxA + (N / C) * 128) + 64;
    static std::atomic<bool> attr_done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev].load(std::memory_order_relaxed)) {
        // the largest size any call can need, set once per device
        const int most = 1024 + 4 * (kBoxA + kMaxRowsB * 128) + 64;
        e = cudaFuncSetAttribute(linear_small_dynamic_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, most);
        if (e != cudaSuccess) return e;
        attr_done[dev].store(true, std::memory_order_relaxed);
    }
    SmallArgs a;
    a.x = x;
    a.w = w;
    a.bias = bias;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.scales = scales;
    a.amax = amax;
    a.xq = xq;
    a.wq = wq;
    a.y = y;
    a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    a.status = device_status_word();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, linear_small_dynamic_kernel, a);
}

}  // namespace fp8
