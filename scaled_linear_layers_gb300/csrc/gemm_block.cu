// Block-scaled FP8 GEMM (the TE "recipe=block" layout: 1x128 tiles along the
// contraction dim for activations and gradients, 128x128 tiles for weights).
//
//   D[i,j] = bf16( sum_kb sA[i,kb] * sB[j,kb] * sum_{k in block kb} A[i,k] B[j,k] )
//
// Each 128-wide contraction block is one pipeline stage.  The MMA warp writes
// that block's partial product (128x128 fp32, fresh accumulation) into one of
// four TMEM slots; eight epilogue warps read it back (two per TMEM lane
// quarter, 64 columns each), multiply by the two block scales and accumulate
// in registers, so the tensor cores never wait for the promotion as long as
// the epilogue keeps up (four slots of slack).  B's scale is one value per
// 128-row tile (weights) or one per row (wgrad's Xᵀ operand, staged through
// shared memory per block).  Same TMA/mbarrier pipeline and bounded waits as
// the tensorwise kernel.
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8 {

extern uint64_t g_wait_limit_ns;

namespace {

constexpr int BM = 128, BN = 128, BK = 128, STAGES = 6, SLOTS = 4;
constexpr int A_STAGE = BM * BK, B_STAGE = BN * BK, STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = SLOTS * BN;  // 512
constexpr int GROUP_M = 8;
constexpr uint32_t IDESC = idesc_f8_f32(BM, BN);
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 2 * BN * sizeof(float) + 256;

struct BlockArgs {
    int M, N, K;
    const float *sa;
    int64_t sa_ld;
    const float *sb;
    int64_t sb_row_stride, sb_k_stride;
    uint16_t *d;
    int64_t ldd;
    uint64_t wait_limit_ns;
    unsigned int *status;
};

__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int &tm, int &tn) {
    grouped_tile(tile, m_tiles, n_tiles, GROUP_M, tm, tn);
}

__device__ __forceinline__ void epi_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(EPI_WARPS * 32) : "memory");
}


template <bool kPerRowB>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_f8_block_kernel(const __grid_constant__ CUtensorMap tma_a,
                         const __grid_constant__ CUtensorMap tma_b, const BlockArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_STAGE;
    float *sbuf = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);  // [2][BN]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbuf + 2 * BN);
    uint64_t *full = bars;                // [STAGES]
    uint64_t *empty = bars + STAGES;      // [STAGES]
    uint64_t *sfull = bars + 2 * STAGES;  // [SLOTS] MMA -> epilogue
    uint64_t *sempty = sfull + SLOTS;     // [SLOTS] epilogue -> MMA
    uint64_t *drain = sempty + SLOTS;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (p.M + BM - 1) / BM, n_tiles = (p.N + BN - 1) / BN;
    const int num_tiles = m_tiles * n_tiles;
    const int nk = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sempty[s], EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tma_a);
        tma_prefetch_desc(&tma_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                int tm, tn;
                tile_coords(tile, m_tiles, n_tiles, tm, tn);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.wait_limit_ns,
                                           kStatusTimeoutTma, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_2d(sA + stage * A_STAGE, &tma_a, &full[stage], kb * BK, tm * BM);
                    tma_load_2d(sB + stage * B_STAGE, &tma_b, &full[stage], kb * BK, tn * BN);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < STAGES; ++s) {
                    stage = stage == 0 ? STAGES - 1 : stage - 1;
                    if (stage == STAGES - 1) phase ^= 1u;
                    volatile int no_abort = 0;
                    mbar_wait_bounded(&full[stage], phase, &no_abort, 10000000ull,
                                      kStatusTimeoutTma, p.status);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t g = 0;  // contraction blocks issued so far (across tiles)
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const uint32_t slot = g % SLOTS, sphase = (g / SLOTS) & 1u;
                    if (!mbar_wait_bounded(&sempty[slot], sphase ^ 1u, abort_flag, p.wait_limit_ns,
                                           kStatusTimeoutMma, p.status) ||
                        !mbar_wait_bounded(&full[stage], phase, abort_flag, p.wait_limit_ns,
                                           kStatusTimeoutMma, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * A_STAGE);
                    const uint32_t b0 = smem_u32(sB + stage * B_STAGE);
                    const uint32_t d_tmem = tmem_base + slot * BN;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_f8(d_tmem, smem_desc_sw128(a0 + 32 * k), smem_desc_sw128(b0 + 32 * k),
                               IDESC, k != 0);
                    mma_commit(&empty[stage]);
                    mma_commit(&sfull[slot]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            mma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait_bounded(drain, 0, &no_abort, p.wait_limit_ns, kStatusTimeoutMma, p.status);
        }
    } else {
        // ------------------------------------------------- epilogue (8 warps)
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;  // 0..255
        bool ok = true;
        uint32_t g = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int tm, tn;
            tile_coords(tile, m_tiles, n_tiles, tm, tn);
            const int row = tm * BM + quarter * 32 + lane;
            const int n0 = tn * BN;
            const bool row_ok = row < p.M;
            const float *sa_row = p.sa + (int64_t)(row_ok ? row : 0) * p.sa_ld;
            const float *sb_base = kPerRowB ? p.sb + (int64_t)min(n0 + (et & (BN - 1)), p.N - 1) *
                                                        p.sb_row_stride
                                            : p.sb + (int64_t)tn * p.sb_row_stride;
            float acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0.f;
            float sa_next = sa_row[0];
            float sb_next = sb_base[0];
            for (int kb = 0; kb < nk; ++kb, ++g) {
                const uint32_t slot = g % SLOTS, sphase = (g / SLOTS) & 1u;
                const float sa_cur = sa_next, sb_cur = sb_next;
                if (kPerRowB && et < BN) sbuf[(kb & 1) * BN + et] = sb_cur;
                if (kb + 1 < nk) {
                    sa_next = sa_row[kb + 1];
                    sb_next = sb_base[(int64_t)(kb + 1) * p.sb_k_stride];
                }
                if (ok)
                    ok = mbar_wait_bounded(&sfull[slot], sphase, abort_flag, p.wait_limit_ns,
                                           kStatusTimeoutEpilogue, p.status);
                ok = __all_sync(0xFFFFFFFFu, ok);
                uint32_t r0[32], r1[32];
                if (ok) {
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                           slot * BN + (uint32_t)(half * 64);
                    tmem_ld_32x32b_x32(taddr, r0);
                    tmem_ld_32x32b_x32(taddr + 32, r1);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sempty[slot]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r0[j] = r1[j] = 0u;
                }
                if (kPerRowB) {
                    epi_barrier();
                    const float4 *sv = reinterpret_cast<const float4 *>(sbuf + (kb & 1) * BN + half * 64);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float4 s4 = sv[q];
                        const float c[4] = {s4.x * sa_cur, s4.y * sa_cur, s4.z * sa_cur, s4.w * sa_cur};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * q + e;
                            const float v = __uint_as_float(j < 32 ? r0[j] : r1[j - 32]);
                            acc[j] = __fmaf_rn(v, c[e], acc[j]);
                        }
                    }
                } else {
                    const float f = sa_cur * sb_cur;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        acc[j] = __fmaf_rn(__uint_as_float(r0[j]), f, acc[j]);
                        acc[j + 32] = __fmaf_rn(__uint_as_float(r1[j]), f, acc[j + 32]);
                    }
                }
            }
            if (ok && row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.d + (int64_t)row * p.ldd + n0 + half * 64);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_uint4(pack_bf16x2(acc[8 * c + 0], acc[8 * c + 1]),
                                        pack_bf16x2(acc[8 * c + 2], acc[8 * c + 3]),
                                        pack_bf16x2(acc[8 * c + 4], acc[8 * c + 5]),
                                        pack_bf16x2(acc[8 * c + 6], acc[8 * c + 7]));
            }
        }
    }

    __syncwarp();  // lanes that skipped a role wait here for their warp's lane 0
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <bool kPerRowB>
cudaError_t launch_block(const CUtensorMap &ta, const CUtensorMap &tb, const BlockArgs &args,
                         int grid, cudaStream_t s) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_f8_block_kernel<kPerRowB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    gemm_f8_block_kernel<kPerRowB><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(ta, tb, args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_block(const uint8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K,
                              const float *sa, int64_t sa_ld, const float *sb,
                              int64_t sb_row_stride, int64_t sb_k_stride, int b_rows_per_scale,
                              uint16_t *D, cudaStream_t s, const char **why) {
    CUtensorMap ta, tb;
    if (!make_tmap_k128(&ta, A, M, K, BM) || !make_tmap_k128(&tb, B, N, K, BN)) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    BlockArgs args;
    args.M = (int)M;
    args.N = (int)N;
    args.K = (int)K;
    args.sa = sa;
    args.sa_ld = sa_ld;
    args.sb = sb;
    args.sb_row_stride = sb_row_stride;
    args.sb_k_stride = sb_k_stride;
    args.d = D;
    args.ldd = N;
    args.wait_limit_ns = g_wait_limit_ns;
    args.status = device_status_word();
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = (int)(tiles < num_sms() ? tiles : num_sms());
    if (b_rows_per_scale == 1) return launch_block<true>(ta, tb, args, grid, s);
    if (b_rows_per_scale == BN) return launch_block<false>(ta, tb, args, grid, s);
    *why = "B scales must be per row or per 128-row tile";
    return cudaErrorInvalidValue;
}

}  // namespace fp8
