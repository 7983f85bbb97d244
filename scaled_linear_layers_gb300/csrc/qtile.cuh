// Tile helpers of the HBM-bound cast kernels: one 128 x 128 tile of a bf16
// [R, C] matrix per CTA of 256 threads.  Thread t holds rows (t>>4)+16*i,
// i < 8, and the 8 columns 8*(t&15)..+7 (8 x 16-byte loads in flight).  The
// bytes quantised for the transpose go to a 16 KB shared tile whose 32-bit
// words are XOR-swizzled by 4*(row/16); the read-back gives lane (a = l&7,
// b = l>>3) of warp wp the word column w = 4*wp + b of rows 16a..16a+15
// (conflict-free under the swizzle), transposes four 4x4 byte blocks with
// byte permutes and stores 16 bytes to each of qt's rows 4w..4w+3, so 8
// lanes write one contiguous 128-byte row segment.
#pragma once

#include "common.cuh"

namespace fp8 {


__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t absmax_bits8(const uint4 &v) {
    return max(max(absmax_bits2(v.x), absmax_bits2(v.y)), max(absmax_bits2(v.z), absmax_bits2(v.w)));
}

// The same maximum with sign bits cleared, unsigned 16-bit lane maxima (one
// max.u16x2 per pair of words), then the larger half: fewer instructions.
// Faster in the tile kernels (1x128 row tiles, row+column cast+transpose:
// 4.70 -> 4.83 TB/s); slower in the tensorwise loop of quantize_kernel
// (6.04 -> 5.43 TB/s at 2^30 elements), which keeps absmax_bits8.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t absmax_bits8_u16x2(const uint4 &v) {
    const uint32_t m = max_u16x2(max_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                 max_u16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16);
}

// Block-wide max of a per-thread bf16-magnitude bit pattern; result valid in
// thread 0.  `red` holds one word per warp.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red) {
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, red[w]);
        v = m;
    }
    return v;
}

// amax bits (a bf16 magnitude pattern) -> fp32 bits of the same value.
__device__ __forceinline__ unsigned int bf16bits_to_f32bits(uint32_t b) { return b << 16; }


// Loads the tile at (r0, c0); out-of-range elements read as zero (R and C
// are multiples of 16, so a 16-byte chunk is either wholly in or out).
__device__ __forceinline__ void tile_load(const uint16_t *__restrict__ x, int R, int C, int r0,
                                          int c0, uint4 (&v)[8]) {
    const int t = threadIdx.x, chunk = t & 15, rsub = t >> 4;
    const int gc = c0 + chunk * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gr = r0 + rsub + 16 * i;
        v[i] = (gr < R && gc < C) ? ldg_nc_v4(x + (int64_t)gr * C + gc) : make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ uint32_t tile_absmax_bits(const uint4 (&v)[8]) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = max(m, absmax_bits8_u16x2(v[i]));
    return m;
}

// Casts the tile with one scale_inv: q (nullable) straight to global, the
// bytes for the transpose into the shared tile.
__device__ __forceinline__ void tile_quant_tensor(const uint4 (&v)[8], float si,
                                                  uint8_t *__restrict__ q, uint32_t *tile, int R,
                                                  int C, int r0, int c0) {
    const int t = threadIdx.x, chunk = t & 15, rsub = t >> 4;
    const int gc = c0 + chunk * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = rsub + 16 * i;
        const int gr = r0 + row;
        const uint32_t t0 = quant4(v[i].x, v[i].y, si);
        const uint32_t t1 = quant4(v[i].z, v[i].w, si);
        if (q != nullptr && gr < R && gc < C)
            *reinterpret_cast<uint2 *>(q + (int64_t)gr * C + gc) = make_uint2(t0, t1);
        const int wcol = (chunk * 2) ^ (4 * (row >> 4));
        *reinterpret_cast<uint2 *>(&tile[row * 32 + wcol]) = make_uint2(t0, t1);
    }
}

// Reads the shared tile back transposed and stores qt [C, R] (caller
// synchronises the block between filling the tile and calling this).
__device__ __forceinline__ void tile_transpose_store(const uint32_t *tile, uint8_t *__restrict__ qt,
                                                     int R, int C, int r0, int c0) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int a = lane & 7, b = lane >> 3;
    const int w = 4 * warp + b;
    uint32_t wv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) wv[i] = tile[(16 * a + i) * 32 + (w ^ (4 * a))];
    uint32_t col[4][4];  // col[j][k]: rows 16a+4k..+3 of column 4w+j
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t x0 = wv[4 * k], x1 = wv[4 * k + 1], x2 = wv[4 * k + 2], x3 = wv[4 * k + 3];
        const uint32_t p0 = __byte_perm(x0, x1, 0x5140), p1 = __byte_perm(x0, x1, 0x7362);
        const uint32_t p2 = __byte_perm(x2, x3, 0x5140), p3 = __byte_perm(x2, x3, 0x7362);
        col[0][k] = __byte_perm(p0, p2, 0x5410);
        col[1][k] = __byte_perm(p0, p2, 0x7632);
        col[2][k] = __byte_perm(p1, p3, 0x5410);
        col[3][k] = __byte_perm(p1, p3, 0x7632);
    }
    const int gr = r0 + 16 * a;
    if (gr < R) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gcc = c0 + 4 * w + j;
            if (gcc < C)
                *reinterpret_cast<uint4 *>(qt + (int64_t)gcc * R + gr) =
                    make_uint4(col[j][0], col[j][1], col[j][2], col[j][3]);
        }
    }
}


}  // namespace fp8
