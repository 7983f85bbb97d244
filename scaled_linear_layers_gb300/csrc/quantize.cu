// HBM-bound kernels: amax, quantise (tensorwise and 1x128 row tiles), the fused
// quantise + transpose (tensorwise, 128x128 tiles, and 1x128 / 128x1 tiles),
// and token padding.
//
// All of them stream bf16 with 16-byte loads, reduce amax on the bf16 bit
// patterns (|x| of non-negative bf16 orders like the unsigned pattern) with
// warp reductions and one atomicMax per block, and cast with
// cvt.rn.satfinite.e4m3x2.f32 after one IEEE fp32 multiply by scale_inv.
#include "common.cuh"
#include "kernels.h"
#include "qtile.cuh"

namespace fp8 {


// ------------------------------------------------------------------ amax ---

__global__ void __launch_bounds__(256) amax_kernel(const uint16_t *__restrict__ x, int64_t n,
                                                   float *__restrict__ amax_out) {
    __shared__ uint32_t red[8];
    pdl_wait_prior();
    pdl_allow_next();
    uint32_t m = 0;
    const int64_t nvec = n >> 3;  // 8 bf16 per 16-byte vector
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        uint4 a = ldg_nc_v4(xv + i), b = ldg_nc_v4(xv + i + stride);
        uint4 c = ldg_nc_v4(xv + i + 2 * stride), d = ldg_nc_v4(xv + i + 3 * stride);
        m = max(m, max(max(absmax_bits8(a), absmax_bits8(b)), max(absmax_bits8(c), absmax_bits8(d))));
    }
    for (; i < nvec; i += stride) m = max(m, absmax_bits8(ldg_nc_v4(xv + i)));
    if (blockIdx.x == 0)
        for (int64_t j = (nvec << 3) + threadIdx.x; j < n; j += blockDim.x)
            m = max(m, (uint32_t)(x[j] & 0x7FFFu));
    m = block_max_u32(m, red);
    if (threadIdx.x == 0 && m != 0)
        atomicMax(reinterpret_cast<unsigned int *>(amax_out), bf16bits_to_f32bits(m));
}

// ------------------------------------------------------ tensorwise cast ---
// DELAYED: scale_inv is read from `scale_src`; the kernel also emits amax
//          (if amax_out != nullptr).
// DYNAMIC: `scale_src` holds this tensor's amax (from amax_kernel); each block
//          derives scale_inv from it, block 0 publishes scale and scale_inv.
template <bool kDynamic>
__global__ void __launch_bounds__(256)
    quantize_kernel(const uint16_t *__restrict__ x, int64_t n, const float *__restrict__ scale_src,
                    uint8_t *__restrict__ q, float *__restrict__ amax_out,
                    float *__restrict__ scale_out, float *__restrict__ scale_inv_out) {
    __shared__ uint32_t red[8];
    pdl_wait_prior();
    pdl_allow_next();
    float si;
    if (kDynamic) {
        float s;
        scales_from_amax(*scale_src, s, si);
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            *scale_out = s;
            *scale_inv_out = si;
        }
    } else {
        si = *scale_src;
    }
    // 16-byte vectors of 8 bf16 -> 8 e4m3 bytes; consecutive lanes take
    // consecutive vectors (full 512-byte loads per warp instruction), four
    // vectors in flight per thread
    uint32_t m = 0;
    const int64_t nvec = n >> 3;
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    uint2 *qv = reinterpret_cast<uint2 *>(q);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        const uint4 a = ldg_nc_v4(xv + i), b = ldg_nc_v4(xv + i + stride);
        const uint4 c = ldg_nc_v4(xv + i + 2 * stride), d = ldg_nc_v4(xv + i + 3 * stride);
        if (!kDynamic)
            m = max(m, max(max(absmax_bits8(a), absmax_bits8(b)),
                           max(absmax_bits8(c), absmax_bits8(d))));
        qv[i] = make_uint2(quant4(a.x, a.y, si), quant4(a.z, a.w, si));
        qv[i + stride] = make_uint2(quant4(b.x, b.y, si), quant4(b.z, b.w, si));
        qv[i + 2 * stride] = make_uint2(quant4(c.x, c.y, si), quant4(c.z, c.w, si));
        qv[i + 3 * stride] = make_uint2(quant4(d.x, d.y, si), quant4(d.z, d.w, si));
    }
    for (; i < nvec; i += stride) {
        const uint4 a = ldg_nc_v4(xv + i);
        if (!kDynamic) m = max(m, absmax_bits8(a));
        qv[i] = make_uint2(quant4(a.x, a.y, si), quant4(a.z, a.w, si));
    }
    if (blockIdx.x == 0) {  // ragged tail: fewer than 8 elements
        for (int64_t j = (nvec << 3) + threadIdx.x; j < n; j += blockDim.x) {
            uint32_t h = x[j];
            if (!kDynamic) m = max(m, h & 0x7FFFu);
            q[j] = (uint8_t)(cvt_e4m3x2(__fmul_rn(__uint_as_float(h << 16), si), 0.0f) & 0xFFu);
        }
    }
    if (!kDynamic && amax_out != nullptr) {
        m = block_max_u32(m, red);
        if (threadIdx.x == 0 && m != 0)
            atomicMax(reinterpret_cast<unsigned int *>(amax_out), bf16bits_to_f32bits(m));
    }
}

// ----------------------------------------------------- 1x128 row tiles ---
// One warp per group of 8 consecutive 128-element tiles (2 KB of bf16): for
// j < 4, lane l reads 16 bytes of tile 2j + l/16, so each load instruction
// covers 512 contiguous bytes.  Tile maxima are reduced within half-warps,
// then gathered so that lane t < 8 holds tile t's: the two IEEE divisions of
// the scale rule run once per 8 tiles instead of in all 16 lanes of every
// tile (they were a third of the kernel's instructions: 2^30 elements 5.14
// -> 6.65 TB/s with this layout and the u16x2 maxima), lanes 0..7 store 8
// consecutive scales with one 32-byte store each, and each half-warp takes
// its tile's scale_inv back by shuffle.  Scale layout [rows, cols/128]
// row-major = tile index order; emits the global amax if asked.
__global__ void __launch_bounds__(256)
    quantize_rowtiles_kernel(const uint16_t *__restrict__ x, int64_t ntiles,
                             uint8_t *__restrict__ q, float *__restrict__ scale,
                             float *__restrict__ scale_inv, float *__restrict__ amax_out) {
    __shared__ uint32_t red[8];
    pdl_wait_prior();
    pdl_allow_next();
    const int lane = threadIdx.x & 31, half = lane >> 4, lane16 = lane & 15;
    const int64_t wg = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t ngroups = (ntiles + 7) >> 3;
    uint32_t gm = 0;
    for (int64_t grp = wg; grp < ngroups; grp += nw) {  // uniform across the warp
        const int64_t t0 = grp << 3;
        uint4 v[4];
        uint32_t m[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t t = t0 + 2 * j + half;
            v[j] = t < ntiles ? ldg_nc_v4(reinterpret_cast<const uint4 *>(x + t * 128) + lane16)
                              : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) m[j] = absmax_bits8_u16x2(v[j]);
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
#pragma unroll
            for (int j = 0; j < 4; ++j) m[j] = max(m[j], __shfl_xor_sync(0xFFFFFFFFu, m[j], o));
        // lane t < 8 takes tile t = 2j + h (j = t/2, h = t%2) from half h
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t mj = __shfl_sync(0xFFFFFFFFu, m[j], 16 * (lane & 1));
            gm = max(gm, m[j]);
            if ((lane >> 1) == j) mine = mj;
        }
        float s, si;
        scales_from_amax(__uint_as_float(mine << 16), s, si);
        if (lane < 8 && t0 + lane < ntiles) {
            scale[t0 + lane] = s;
            scale_inv[t0 + lane] = si;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float sij = __shfl_sync(0xFFFFFFFFu, si, 2 * j + half);
            const int64_t t = t0 + 2 * j + half;
            if (t < ntiles)
                reinterpret_cast<uint2 *>(q + t * 128)[lane16] =
                    make_uint2(quant4(v[j].x, v[j].y, sij), quant4(v[j].z, v[j].w, sij));
        }
    }
    if (amax_out != nullptr) {
        gm = block_max_u32(gm, red);
        if (threadIdx.x == 0 && gm != 0)
            atomicMax(reinterpret_cast<unsigned int *>(amax_out), bf16bits_to_f32bits(gm));
    }
}
constexpr int kRowtilesPerBlock = 64;  // 8 warps x 8 tiles per pass

// ------------------------------------------------ fused cast + transpose ---
// One CTA of 256 threads per 128x128 tile of x [R, C] (R, C multiples of 16;
// edge tiles are masked).  Load: thread t holds rows (t>>4)+16*i, i < 8, and
// the 8 columns 8*(t&15)..+7 — 8 x 16-byte loads in flight.  The tile is
// quantised in registers, q is stored directly (8 bytes per row chunk), and
// the bytes quantised for the transpose go to a 16 KB shared tile whose
// 32-bit words are XOR-swizzled by 4*(row/16).  Read back: lane (a = l&7,
// b = l>>3) of warp wp takes word column w = 4*wp + b of rows 16a..16a+15 —
// conflict-free under the swizzle — transposes four 4x4 byte blocks with
// byte permutes and stores 16 bytes to each of qt's rows 4w..4w+3, so 8
// lanes write one contiguous 128-byte row segment.
//
// Scale modes:
//   kTensorDelayed: one scale_inv read from scale_src; amax emitted.
//   kTensorDynamic: scale_src holds amax; scales derived and published by
//                   block (0,0).
//   kTile2D:        one scale per 128x128 tile from the tile's amax
//                   (scale grid [R/128, C/128]), used for q and qt.
//   kRowCol:        q uses 1x128 row-tile scales (scale/scale_inv
//                   [R, C/128]); qt uses 128x1 column-tile scales
//                   (scale_t/scale_inv_t [R/128, C]: one row of scales per
//                   128-row block, contiguous over the columns, which is the
//                   order the block GEMM reads them in).
enum QtMode { kTensorDelayed = 0, kTensorDynamic = 1, kTile2D = 2, kRowCol = 3 };

// One launch may cover two tensors (a "job" each, same mode): the first
// job's tiles take blocks 0..tiles-1, the second's the rest.  A step issues
// its independent quantisations in one launch this way, halving the launch
// ramps of these short, HBM-bound kernels.
struct QtJob {
    const uint16_t *x;
    int R, C, tiles_x, tiles;
    const float *scale_src;
    uint8_t *q, *qt;
    float *amax_out, *scale, *scale_inv, *scale_t, *scale_inv_t;
    // tensor modes: per-tile column sums of x, [tiles_y, C] fp32 (nullable);
    // colsum_reduce_kernel turns them into the bias gradient
    float *colsum;
};
// A byte transpose riding in the same launch (delayed mode): qt [C, R] =
// q [R, C]ᵀ for e4m3 bytes that already exist, in 128 x 128 tiles after the
// two jobs' tiles.  The step uses it to give dgrad Wqᵀ from Wq in the
// backward launch, off the forward's critical path, with the same bytes a
// second cast of W would give.
struct QtBytes {
    const uint8_t *q;
    int R, C, tiles_x, tiles;
    uint8_t *qt;
};
struct QtJobs {
    QtJob job[2];
    QtBytes bytes;
    // optional scalar copy done by block 0 (snap_dst = *snap_src): lets a
    // step keep the scale its forward GEMM must use while a concurrent state
    // update replaces it
    const float *snap_src;
    float *snap_dst;
};

// Four CTAs per SM for the row+column, 2D-tile and dynamic modes (the
// row+column mode would otherwise take 120 registers and run two: 32768 x 8192,
// 4625 against 3839 GB/s), five for the delayed mode the training step runs:
// 48 registers without spills, so 760 slots take a 4096^2 step's 2048 tiles in
// 2.7 waves instead of 3.4 (in-step forward / backward launches 23.2-23.5 /
// 24.4-24.7 us against 23.6-23.9 / 24.9-25.2; six CTAs at 40 registers spill
// and took 27.2 / 28.8).
template <int kMode>
__global__ void __launch_bounds__(256, kMode == kTensorDelayed ? 5 : 4) quantize_transpose_kernel(const QtJobs jobs) {
    __shared__ __align__(16) uint32_t tile[128 * 32];
    __shared__ uint32_t red[8];
    __shared__ uint32_t colmax[8][128];
    __shared__ float col_si[128];
    __shared__ float tile_si;
    pdl_wait_prior();
    pdl_allow_next();
    if (blockIdx.x == 0 && threadIdx.x == 0 && jobs.snap_dst != nullptr)
        *jobs.snap_dst = *jobs.snap_src;
    if (kMode == kTensorDelayed) {
        const int cast_tiles = jobs.job[0].tiles + jobs.job[1].tiles;
        if ((int)blockIdx.x >= cast_tiles) {
            // byte transpose: thread t moves 16-byte chunk t%8 of rows t/8 + 32i
            // into the shared tile's layout (chunk c of row r at word
            // 4 * (c ^ (r / 16 % 8)), conflict-free), then the same
            // transposed store as the cast
            const QtBytes &B = jobs.bytes;
            const int id = (int)blockIdx.x - cast_tiles;
            const int r0 = (id / B.tiles_x) * 128, c0 = (id % B.tiles_x) * 128;
            const int ch = threadIdx.x & 7, rs = threadIdx.x >> 3;
            const int gc = c0 + 16 * ch;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = rs + 32 * i, gr = r0 + row;
                const uint4 v = (gr < B.R && gc < B.C) ? ldg_nc_v4(B.q + (int64_t)gr * B.C + gc)
                                                       : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(&tile[row * 32 + 4 * (ch ^ ((row >> 4) & 7))]) = v;
            }
            __syncthreads();
            tile_transpose_store(tile, B.qt, B.R, B.C, r0, c0);
            return;
        }
    }

    const bool second = (int)blockIdx.x >= jobs.job[0].tiles;
    const QtJob J = second ? jobs.job[1] : jobs.job[0];
    const int tile_id = (int)blockIdx.x - (second ? jobs.job[0].tiles : 0);
    const int bx = tile_id % J.tiles_x, by = tile_id / J.tiles_x;
    const uint16_t *__restrict__ x = J.x;
    const int R = J.R, C = J.C;
    const float *__restrict__ scale_src = J.scale_src;
    uint8_t *__restrict__ q = J.q;
    uint8_t *__restrict__ qt = J.qt;
    float *__restrict__ amax_out = J.amax_out;
    float *__restrict__ scale = J.scale;
    float *__restrict__ scale_inv = J.scale_inv;
    float *__restrict__ scale_t = J.scale_t;
    float *__restrict__ scale_inv_t = J.scale_inv_t;

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int r0 = by * 128, c0 = bx * 128;
    const int chunk = t & 15, rsub = t >> 4;
    const int gc = c0 + chunk * 8;

    uint4 v[8];
    tile_load(x, R, C, r0, c0, v);

    float si_all = 0.f;
    if (kMode == kTensorDelayed) si_all = *scale_src;
    if (kMode == kTensorDynamic) {
        float s;
        scales_from_amax(*scale_src, s, si_all);
        if (bx == 0 && by == 0 && t == 0) {
            *scale = s;
            *scale_inv = si_all;
        }
    }

    // column sums of the tile (bias gradient): per thread over its 8 rows in
    // row order, then lanes l and l^16, then the 8 warps in warp order
    if ((kMode == kTensorDelayed || kMode == kTensorDynamic) && J.colsum != nullptr) {
        float cs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) cs[e] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                cs[2 * e] = __fadd_rn(cs[2 * e], bf16_lo(w4[e]));
                cs[2 * e + 1] = __fadd_rn(cs[2 * e + 1], bf16_hi(w4[e]));
            }
        }
        float *colsum_sh = reinterpret_cast<float *>(&colmax[0][0]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, cs[e], 16);
            cs[e] = lane < 16 ? __fadd_rn(cs[e], o) : __fadd_rn(o, cs[e]);
        }
        if (lane < 16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) colsum_sh[warp * 128 + chunk * 8 + e] = cs[e];
        }
        __syncthreads();
        if (t < 128 && c0 + t < C) {
            float acc = colsum_sh[t];
#pragma unroll
            for (int w = 1; w < 8; ++w) acc = __fadd_rn(acc, colsum_sh[w * 128 + t]);
            J.colsum[(int64_t)by * C + c0 + t] = acc;
        }
    }

    // amax: whole tile (tensor / tile modes), or per row and per column.
    float row_si[8];
    uint32_t m_delayed = 0;  // this thread's |x| maximum (delayed mode)
    if (kMode == kRowCol) {
        // rows: the 16 threads sharing rsub hold one 128-element row per i
        // (a warp holds rows 2*warp + h + 16*i, h = lane/16)
        uint32_t mrow[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t m = absmax_bits8_u16x2(v[i]);
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            mrow[i] = m;
        }
        // each row's scales in the row's own 16 lanes.  Gathering the warp's
        // 16 row maxima so that one lane per row divides (as the 1x128
        // row-tile kernel does) measured faster inside the block step (X, W,
        // G quantisation 455 -> 420 us) but slower alone (5.20 -> 4.44 TB/s
        // at 32768 x 8192), so it is not used here.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float s, si;
            scales_from_amax(__uint_as_float(mrow[i] << 16), s, si);
            row_si[i] = si;
            const int gr = r0 + rsub + 16 * i;
            if (chunk == 0 && gr < R && scale != nullptr) {
                const int64_t idx = (int64_t)gr * (C >> 7) + bx;
                scale[idx] = s;
                scale_inv[idx] = si;
            }
        }
        // columns: per thread 8 columns over its 8 rows (as 16-bit pairs),
        // then across lanes l and l^16 (same chunk), then across the 8 warps
        // in shared memory.
        uint32_t cmp[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) cmp[e] = max_u16x2(cmp[e], w4[e] & 0x7FFF7FFFu);
        }
        uint32_t cm[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            cm[2 * e] = cmp[e] & 0xFFFFu;
            cm[2 * e + 1] = cmp[e] >> 16;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) cm[e] = max(cm[e], __shfl_xor_sync(0xFFFFFFFFu, cm[e], 16));
        if (lane < 16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) colmax[warp][chunk * 8 + e] = cm[e];
        }
        __syncthreads();
        if (t < 128) {
            uint32_t m = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) m = max(m, colmax[w][t]);
            float s, si;
            scales_from_amax(__uint_as_float(m << 16), s, si);
            col_si[t] = si;
            if (c0 + t < C) {
                const int64_t idx = (int64_t)by * C + (c0 + t);  // [R/128, C]
                scale_t[idx] = s;
                scale_inv_t[idx] = si;
            }
        }
        if (amax_out != nullptr && t < 128) {
            uint32_t m = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) m = max(m, colmax[w][t]);
            m = __reduce_max_sync(0xFFFFFFFFu, m);
            if (lane == 0 && m != 0)
                atomicMax(reinterpret_cast<unsigned int *>(amax_out), bf16bits_to_f32bits(m));
        }
        __syncthreads();
    } else {
        uint32_t m = 0;
        if (kMode != kTensorDynamic) {
#pragma unroll
            for (int i = 0; i < 8; ++i) m = max(m, absmax_bits8_u16x2(v[i]));
            // delayed scaling casts with a known scale: its block reduction
            // waits until after the stores (below), so no warp holds its
            // cast back for the other warps' loads
            if (kMode != kTensorDelayed) m = block_max_u32(m, red);
        }
        m_delayed = m;
        if (kMode == kTile2D) {
            if (t == 0) {
                float s, si;
                scales_from_amax(__uint_as_float(m << 16), s, si);
                const int64_t idx = (int64_t)by * J.tiles_x + bx;
                scale[idx] = s;
                scale_inv[idx] = si;
                tile_si = si;
            }
            __syncthreads();
            si_all = tile_si;
        }
        if (kMode != kTensorDynamic && kMode != kTensorDelayed && amax_out != nullptr && t == 0 &&
            m != 0)
            atomicMax(reinterpret_cast<unsigned int *>(amax_out), bf16bits_to_f32bits(m));
    }

    // quantise: q (row scales) straight to global, transpose bytes to smem
    float csi[8];
    if (kMode == kRowCol) {
#pragma unroll
        for (int e = 0; e < 8; ++e) csi[e] = col_si[chunk * 8 + e];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = rsub + 16 * i;
        const int gr = r0 + row;
        uint32_t t0, t1;
        if (kMode == kRowCol) {
            const float si = row_si[i];
            if (q != nullptr && gr < R && gc < C)
                *reinterpret_cast<uint2 *>(q + (int64_t)gr * C + gc) =
                    make_uint2(quant4(v[i].x, v[i].y, si), quant4(v[i].z, v[i].w, si));
            t0 = cvt_e4m3x2(__fmul_rn(bf16_lo(v[i].x), csi[0]), __fmul_rn(bf16_hi(v[i].x), csi[1])) |
                 (cvt_e4m3x2(__fmul_rn(bf16_lo(v[i].y), csi[2]), __fmul_rn(bf16_hi(v[i].y), csi[3]))
                  << 16);
            t1 = cvt_e4m3x2(__fmul_rn(bf16_lo(v[i].z), csi[4]), __fmul_rn(bf16_hi(v[i].z), csi[5])) |
                 (cvt_e4m3x2(__fmul_rn(bf16_lo(v[i].w), csi[6]), __fmul_rn(bf16_hi(v[i].w), csi[7]))
                  << 16);
        } else {
            t0 = quant4(v[i].x, v[i].y, si_all);
            t1 = quant4(v[i].z, v[i].w, si_all);
            if (q != nullptr && gr < R && gc < C)
                *reinterpret_cast<uint2 *>(q + (int64_t)gr * C + gc) = make_uint2(t0, t1);
        }
        if (qt != nullptr) {  // bytes for the transpose (the same for the whole CTA)
            const int wcol = (chunk * 2) ^ (4 * (row >> 4));
            *reinterpret_cast<uint2 *>(&tile[row * 32 + wcol]) = make_uint2(t0, t1);
        }
    }
    if (kMode == kTensorDelayed && amax_out != nullptr) {
        const uint32_t m = block_max_u32(m_delayed, red);
        if (t == 0 && m != 0)
            atomicMax(reinterpret_cast<unsigned int *>(amax_out), bf16bits_to_f32bits(m));
    }
    if (qt == nullptr) return;  // q only: no transpose
    __syncthreads();

    tile_transpose_store(tile, qt, R, C, r0, c0);
}

// ------------------------------------------------------- bias gradient ---
// dbias[n] = bf16( sum over the tiles' column sums of column n, in tile
// order ); one thread per column.
__global__ void __launch_bounds__(256) colsum_reduce_kernel(const float *__restrict__ part,
                                                            int tiles_y, int cols,
                                                            uint16_t *__restrict__ dbias) {
    pdl_wait_prior();
    pdl_allow_next();
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= cols) return;
    float acc = 0.f;
    for (int b = 0; b < tiles_y; ++b) acc = __fadd_rn(acc, part[(int64_t)b * cols + n]);
    const __nv_bfloat16 h = __float2bfloat16_rn(acc);
    dbias[n] = *reinterpret_cast<const uint16_t *>(&h);
}

// --------------------------------------------------------------- padding ---

__global__ void __launch_bounds__(256) pad_rows_kernel_v16(const uint4 *__restrict__ x,
                                                           int64_t n_in, int64_t n_out,
                                                           uint4 *__restrict__ out) {
    pdl_wait_prior();
    pdl_allow_next();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_out; i += stride)
        out[i] = i < n_in ? ldg_nc_v4(x + i) : make_uint4(0, 0, 0, 0);
}

__global__ void __launch_bounds__(256) pad_rows_kernel_scalar(const uint16_t *__restrict__ x,
                                                              int64_t n_in, int64_t n_out,
                                                              uint16_t *__restrict__ out) {
    pdl_wait_prior();
    pdl_allow_next();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_out; i += stride)
        out[i] = i < n_in ? x[i] : (uint16_t)0;
}

// ------------------------------------------------------------ launchers ---

static int grid_for(int64_t work_items, int per_block) {
    int64_t g = (work_items + per_block - 1) / per_block;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

cudaError_t launch_amax(const uint16_t *x, int64_t n, float *amax_out, cudaStream_t s) {
    cudaError_t e = launch_zero_f32(amax_out, 1, s);
    if (e != cudaSuccess || n == 0) return e;
    return launch_pdl(amax_kernel, grid_for((n >> 3) / 4 + 1, 256), 256, 0, s, x, n, amax_out);
}

cudaError_t launch_quantize_tensor(const uint16_t *x, int64_t n, bool dynamic, float *scale,
                                   float *scale_inv, uint8_t *q, float *amax_out,
                                   cudaStream_t s) {
    cudaError_t e;
    const int grid = grid_for((n >> 3) / 4 + 1, 256);
    if (dynamic) {
        if ((e = launch_amax(x, n, amax_out, s)) != cudaSuccess) return e;
        e = launch_pdl(quantize_kernel<true>, grid, 256, 0, s, x, n, (const float *)amax_out, q,
                       (float *)nullptr, scale, scale_inv);
        if (e != cudaSuccess) return e;
    } else {
        if (amax_out != nullptr && (e = launch_zero_f32(amax_out, 1, s)) != cudaSuccess)
            return e;
        if (n == 0) return cudaSuccess;
        e = launch_pdl(quantize_kernel<false>, grid, 256, 0, s, x, n, (const float *)scale_inv, q,
                       amax_out, (float *)nullptr, (float *)nullptr);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize_rowtiles(const uint16_t *x, int64_t rows, int64_t cols, float *scale,
                                     float *scale_inv, uint8_t *q, float *amax_out,
                                     cudaStream_t s) {
    cudaError_t e;
    if (amax_out != nullptr && (e = launch_zero_f32(amax_out, 1, s)) != cudaSuccess)
        return e;
    const int64_t ntiles = rows * (cols / 128);
    if (ntiles == 0) return cudaSuccess;
    return launch_pdl(quantize_rowtiles_kernel, grid_for(ntiles, kRowtilesPerBlock), 256, 0, s, x, ntiles, q,
                      scale, scale_inv, amax_out);
}

static QtJob make_job(const uint16_t *x, int64_t rows, int64_t cols, const float *src,
                      float *scale, float *scale_inv, uint8_t *q, uint8_t *qt, float *scale_t,
                      float *scale_inv_t, float *amax_k) {
    QtJob j;
    j.x = x;
    j.R = (int)rows;
    j.C = (int)cols;
    j.tiles_x = (int)((cols + 127) / 128);
    j.tiles = rows * cols == 0 ? 0 : j.tiles_x * (int)((rows + 127) / 128);
    j.scale_src = src;
    j.q = q;
    j.qt = qt;
    j.amax_out = amax_k;
    j.scale = scale;
    j.scale_inv = scale_inv;
    j.scale_t = scale_t;
    j.scale_inv_t = scale_inv_t;
    j.colsum = nullptr;
    return j;
}

static cudaError_t launch_jobs(int mode, const QtJobs &jobs, cudaStream_t s) {
    const int grid = jobs.job[0].tiles + jobs.job[1].tiles +
                     (mode == kTensorDelayed ? jobs.bytes.tiles : 0);
    if (grid == 0) return cudaSuccess;
    switch (mode) {
    case kTensorDelayed: return launch_pdl(quantize_transpose_kernel<kTensorDelayed>, grid, 256, 0, s, jobs);
    case kTensorDynamic: return launch_pdl(quantize_transpose_kernel<kTensorDynamic>, grid, 256, 0, s, jobs);
    case kTile2D: return launch_pdl(quantize_transpose_kernel<kTile2D>, grid, 256, 0, s, jobs);
    default: return launch_pdl(quantize_transpose_kernel<kRowCol>, grid, 256, 0, s, jobs);
    }
}

cudaError_t launch_quantize_transpose(const uint16_t *x, int64_t rows, int64_t cols, int mode,
                                      float *scale, float *scale_inv, uint8_t *q, uint8_t *qt,
                                      float *scale_t, float *scale_inv_t, float *amax_out,
                                      cudaStream_t s, float *colsum) {
    cudaError_t e;
    const float *src = nullptr;
    if (mode == kTensorDynamic) {
        if ((e = launch_amax(x, rows * cols, amax_out, s)) != cudaSuccess) return e;
        src = amax_out;
    } else {
        if (amax_out != nullptr && (e = launch_zero_f32(amax_out, 1, s)) != cudaSuccess)
            return e;
        if (mode == kTensorDelayed) src = scale_inv;
    }
    QtJobs jobs;
    jobs.job[0] = make_job(x, rows, cols, src, scale, scale_inv, q, qt, scale_t, scale_inv_t,
                           mode == kTensorDynamic ? nullptr : amax_out);
    jobs.job[0].colsum = colsum;
    jobs.job[1] = jobs.job[0];
    jobs.job[1].tiles = 0;
    jobs.bytes = QtBytes{};
    jobs.snap_src = nullptr;
    jobs.snap_dst = nullptr;
    return launch_jobs(mode, jobs, s);
}

cudaError_t launch_quantize_delayed_pair(const DelayedQuantJob &a, const DelayedQuantJob &b,
                                         cudaStream_t s, const float *snap_src,
                                         float *snap_dst, const ByteTransposeJob *bt) {
    QtJobs jobs;
    jobs.bytes = QtBytes{};
    if (bt != nullptr && bt->rows * bt->cols > 0) {
        jobs.bytes.q = bt->q;
        jobs.bytes.R = (int)bt->rows;
        jobs.bytes.C = (int)bt->cols;
        jobs.bytes.tiles_x = (int)((bt->cols + 127) / 128);
        jobs.bytes.tiles = jobs.bytes.tiles_x * (int)((bt->rows + 127) / 128);
        jobs.bytes.qt = bt->qt;
    }
    jobs.snap_src = snap_src;
    jobs.snap_dst = snap_dst;
    jobs.job[0] = make_job(a.x, a.rows, a.cols, a.scale_inv, nullptr, nullptr, a.q, a.qt, nullptr,
                           nullptr, a.amax_out);
    jobs.job[0].colsum = a.colsum;
    jobs.job[1] = make_job(b.x, b.rows, b.cols, b.scale_inv, nullptr, nullptr, b.q, b.qt, nullptr,
                           nullptr, b.amax_out);
    jobs.job[1].colsum = b.colsum;
    return launch_jobs(kTensorDelayed, jobs, s);
}

cudaError_t launch_colsum_reduce(const float *partials, int64_t rows, int64_t cols,
                                 uint16_t *dbias, cudaStream_t s) {
    if (cols == 0) return cudaSuccess;
    const int tiles_y = (int)((rows + 127) / 128);
    return launch_pdl(colsum_reduce_kernel, (int)((cols + 255) / 256), 256, 0, s, partials,
                      tiles_y, (int)cols, dbias);
}

cudaError_t launch_pad_rows(const uint16_t *x, int64_t rows, int64_t cols, int64_t padded,
                            uint16_t *out, cudaStream_t s) {
    const int64_t n_in = rows * cols, n_out = padded * cols;
    if (n_out == 0) return cudaSuccess;
    if (cols % 8 == 0) {
        return launch_pdl(pad_rows_kernel_v16, grid_for(n_out / 8, 256), 256, 0, s,
                          reinterpret_cast<const uint4 *>(x), n_in / 8, n_out / 8,
                          reinterpret_cast<uint4 *>(out));
    }
    return launch_pdl(pad_rows_kernel_scalar, grid_for(n_out, 256), 256, 0, s, x, n_in, n_out, out);
}

}  // namespace fp8
