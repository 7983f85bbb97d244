// Current (dynamic) tensorwise scaling in one launch.
//
// The two-pass form reads x twice from HBM (amax pass, then the cast).  Here a
// persistent grid (cooperative launch: every CTA resident) sweeps its 128x128
// tiles once for the amax, keeping the last tile in registers, meets at a
// grid-wide barrier, derives the scale from the global amax and casts: first
// the tile still in registers, then its other tiles in reverse order, so the
// re-reads hit the L2 (129 MB) whenever the tensor fits there.  The barrier
// and the per-CTA partial amaxes live in a small caller-owned workspace.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "qtile.cuh"

namespace fp8 {

extern std::atomic<uint64_t> g_wait_limit_ns;

namespace {

// workspace words: [0] arrivals, [1] generation, [kWsHeader + b] partial amax
// (bf16 magnitude bits) of CTA b
constexpr int kWsHeader = 16;
constexpr int kMaxGrid = (int)(kFusedWorkspaceBytes / 4) - kWsHeader;

struct FusedArgs {
    const uint16_t *x;
    int R, C, tiles_x, tiles;
    float *scale, *scale_inv, *amax_out;
    uint8_t *q, *qt;
    unsigned int *ws;
    uint64_t wait_limit_ns;
    unsigned int *status;
};

// Grid-wide barrier (sense by generation).  Thread 0 of each CTA reads the
// generation, publishes its CTA's writes, arrives; the last arrival resets the
// count and advances the generation; the others wait (bounded) for it to move.
// Returns false (in every thread of the CTA) if the wait ran out.
__device__ bool grid_barrier(unsigned int *ws, unsigned int nblocks, uint64_t limit_ns,
                             unsigned int *status, int *flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile unsigned int *gen = ws + 1;
        const unsigned int g = *gen;
        __threadfence();
        int ok = 1;
        if (atomicAdd(ws, 1u) + 1u == nblocks) {
            atomicExch(ws, 0u);
            __threadfence();
            atomicAdd(ws + 1, 1u);
        } else {
            const uint64_t t0 = global_timer_ns();
            while (*gen == g) {
                if (global_timer_ns() - t0 > limit_ns) {
                    ok = 0;
                    atomicOr(status, kStatusTimeoutBarrier);
                    break;
                }
                __nanosleep(100);
            }
        }
        __threadfence();
        *flag = ok;
    }
    __syncthreads();
    return *flag != 0;
}

__global__ void __launch_bounds__(256) quantize_fused_dynamic_kernel(const FusedArgs p) {
    __shared__ uint32_t tile[128 * 32];
    __shared__ uint32_t red[8];
    __shared__ int flag;
    __shared__ float s_si;
    const int G = gridDim.x;

    // phase 1: amax over this CTA's tiles; the last one stays in registers
    uint4 v[8];
    uint32_t m = 0;
    int held = -1;
    for (int t = blockIdx.x; t < p.tiles; t += G) {
        tile_load(p.x, p.R, p.C, (t / p.tiles_x) * 128, (t % p.tiles_x) * 128, v);
        m = max(m, tile_absmax_bits(v));
        held = t;
    }
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) p.ws[kWsHeader + blockIdx.x] = m;
    if (!grid_barrier(p.ws, (unsigned int)G, p.wait_limit_ns, p.status, &flag)) return;

    // global amax from the partials (every CTA reduces the same values)
    uint32_t mm = 0;
    const volatile unsigned int *part = p.ws + kWsHeader;
    for (int i = threadIdx.x; i < G; i += blockDim.x) mm = max(mm, part[i]);
    mm = block_max_u32(mm, red);
    if (threadIdx.x == 0) {
        const float a = __uint_as_float(mm << 16);
        float s, si;
        scales_from_amax(a, s, si);
        s_si = si;
        if (blockIdx.x == 0) {
            *p.amax_out = a;
            *p.scale = s;
            *p.scale_inv = si;
        }
    }
    __syncthreads();
    const float si = s_si;

    // phase 2: the held tile, then the earlier ones, most recently read first
    for (int t = held; t >= 0; t -= G) {
        const int r0 = (t / p.tiles_x) * 128, c0 = (t % p.tiles_x) * 128;
        if (t != held) tile_load(p.x, p.R, p.C, r0, c0, v);
        tile_quant_tensor(v, si, p.q, tile, p.R, p.C, r0, c0);
        if (p.qt != nullptr) {
            __syncthreads();
            tile_transpose_store(tile, p.qt, p.R, p.C, r0, c0);
        }
        __syncthreads();  // the shared tile is refilled next iteration
    }
}

// Scratch of the allocation-free entry point (fp8_quantize_fused_dynamic_noalloc):
// the barrier words and one partial amax for each of at most
// kStaticMaxGrid CTAs, 4 KiB that every GPU loading the library keeps until
// the process exits.  All calls of that entry point share it.
constexpr int kStaticMaxGrid = 1008;
static __device__ __align__(256) unsigned int g_noalloc_scratch[kWsHeader + kStaticMaxGrid];

}  // namespace

// Resident CTAs per SM of the fused kernel on device `dev`, looked up once per
// device.  Host threads may race on the first lookup; they store the same
// value, and the atomic makes the race well defined.
static cudaError_t fused_occupancy(int dev, int *occ) {
    static std::atomic<int> cache[64];
    int v = (dev >= 0 && dev < 64) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (v == 0) {
        cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, quantize_fused_dynamic_kernel, 256, 0);
        if (e != cudaSuccess) return e;
        if (v < 1) return cudaErrorInvalidConfiguration;
        if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
    }
    *occ = v;
    return cudaSuccess;
}

static FusedArgs fused_args(const uint16_t *x, int64_t rows, int64_t cols, float *scale,
                            float *scale_inv, uint8_t *q, uint8_t *qt, float *amax_out,
                            unsigned int *ws) {
    FusedArgs a;
    a.x = x;
    a.R = (int)rows;
    a.C = (int)cols;
    a.tiles_x = (int)((cols + 127) / 128);
    a.tiles = rows * cols == 0 ? 0 : (int)(a.tiles_x * ((rows + 127) / 128));
    a.scale = scale;
    a.scale_inv = scale_inv;
    a.amax_out = amax_out;
    a.q = q;
    a.qt = qt;
    a.ws = ws;
    a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    a.status = device_status_word();
    return a;
}

bool fused_tiles_fit(int64_t rows, int64_t cols) {
    return ((cols + 127) / 128) * ((rows + 127) / 128) <= 0x7FFFFFFF;
}

cudaError_t launch_quantize_fused_dynamic(const uint16_t *x, int64_t rows, int64_t cols,
                                          float *scale, float *scale_inv, uint8_t *q, uint8_t *qt,
                                          float *amax_out, unsigned int *workspace,
                                          cudaStream_t s) {
    int dev = 0, occ = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = fused_occupancy(dev, &occ);
    if (e != cudaSuccess) return e;
    FusedArgs a = fused_args(x, rows, cols, scale, scale_inv, q, qt, amax_out, workspace);
    int64_t grid = (int64_t)num_sms() * occ;
    if (grid > a.tiles) grid = a.tiles;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid < 1) grid = 1;
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(quantize_fused_dynamic_kernel),
                                       dim3((unsigned)grid), dim3(256), args, 0, s);
}

// The same kernel with its scratch in g_noalloc_scratch instead of a caller
// workspace.  In host code the array's name is only a stand-in for the device
// object, so its device address is looked up with cudaGetSymbolAddress once
// per device (with that device current) on the first call there.  The grid is
// clamped to the array's kStaticMaxGrid partial slots (CTAs walk their tiles
// with a grid stride, so fewer CTAs than the GPU could hold give the same
// result), so no tensor size needs more scratch than the array has.
cudaError_t launch_quantize_fused_dynamic_noalloc(const uint16_t *x, int64_t rows, int64_t cols,
                                                  float *scale, float *scale_inv, uint8_t *q,
                                                  uint8_t *qt, float *amax_out, cudaStream_t s,
                                                  const char **why) {
    // per-device address of the array; host threads that race on a device's
    // first call store the same address
    static std::atomic<unsigned int *> scratch_addr[64];
    int dev = 0, occ = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) {
        *why = "device index out of range";
        return cudaErrorInvalidDevice;
    }
    unsigned int *ws = scratch_addr[dev].load(std::memory_order_acquire);
    if (ws == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) {
            *why = "cudaGetSymbolAddress of the static scratch failed";
            return e;
        }
        ws = static_cast<unsigned int *>(ptr);
        scratch_addr[dev].store(ws, std::memory_order_release);
    }
    e = fused_occupancy(dev, &occ);
    if (e != cudaSuccess) return e;
    FusedArgs a = fused_args(x, rows, cols, scale, scale_inv, q, qt, amax_out, ws);
    int64_t grid = (int64_t)num_sms() * occ;
    if (grid > a.tiles) grid = a.tiles;
    if (grid > kStaticMaxGrid) grid = kStaticMaxGrid;
    if (grid < 1) grid = 1;
    // the arrival count must start at zero; a previous call that timed out
    // may have left it otherwise (a memset, not an allocation)
    e = cudaMemsetAsync(a.ws, 0, 2 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(quantize_fused_dynamic_kernel),
                                       dim3((unsigned)grid), dim3(256), args, 0, s);
}

}  // namespace fp8
