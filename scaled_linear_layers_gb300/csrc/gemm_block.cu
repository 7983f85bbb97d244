// Block-scaled FP8 GEMM (the TE "recipe=block" layout: 1x128 tiles along the
// contraction dim for activations and gradients, 128x128 tiles for weights).
//
//   D[i,j] = bf16( sum_kb sA(i,kb) * sB(j,kb) * sum_{k in block kb} A[i,k] B[j,k] )
//
// One persistent CTA per SM owns 128 x 128 output tiles.  The contraction is
// walked in groups of two 128-deep blocks: one TMA stage, one round of MMAs
// and one hand-off per group.  The MMA warp writes each block's partial
// product (fresh accumulation) into its own 128-column TMEM slot; the four
// slots form two group slots, so the MMAs of one group run while the
// promotion reads the other.  Eight epilogue warps (two per TMEM lane
// quarter, 64 columns each) read a group's partials back one block at a
// time, hand the group slot back after the last read and fold each partial
// into fp32 register accumulators with its two block scales (packed fp32x2
// FMAs for per-tile B, a multiply and an FMA per element for per-row B).  A hand-off costs a few hundred cycles of barrier traffic
// whatever it carries, so pairing the blocks halves that cost per block.
// B's scale is one value per 128-row tile (weights) or one per row (wgrad's
// Xᵀ operand: each warp stages its 64 scales of the next group into shared
// memory with cp.async, from a layout contiguous over rows).  Every handshake
// is local to the SM, and every wait is bounded, as in the other GEMM kernels.
//
// The same pipeline also runs on CTA pairs (tcgen05 cta_group::2,
// as in the tensorwise pair kernel): a pair owns a 256 x 128 tile, each CTA
// loads its 128 rows of A and 64 rows of B, the leader issues M=256 MMAs whose
// rows land in both CTAs' TMEM, commits multicast to both, and both CTAs'
// epilogue warps hand group slots back to the leader.  Each SM then streams
// 128 x (128 + 64) operand bytes per block instead of 128 x (128 + 128), with
// the same promotion work per SM.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8 {

extern uint64_t g_wait_limit_ns;

namespace {

constexpr int BM = 128, BN = 128, BK = 128;
constexpr int KG = 2;      // contraction blocks per group (stage, MMA round, hand-off)
constexpr int GSLOTS = 2;  // group slots of KG TMEM slots each
constexpr int A_BLK = BM * BK;
// B rows each CTA loads per block: the whole N tile, or half of it in a pair
template <bool kPair> struct Shape {
    static constexpr int B_ROWS = kPair ? BN / 2 : BN;
    static constexpr int B_BLK = B_ROWS * BK;
    static constexpr int A_STAGE = KG * A_BLK, B_STAGE = KG * B_BLK;
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
    static constexpr int STAGES = kPair ? 4 : 3;  // TMA ring depth, in groups
    static constexpr uint32_t IDESC = idesc_f8_f32(kPair ? 2 * BM : BM, BN);
};
#ifndef FP8_BLOCK_EPI_WARPS
#define FP8_BLOCK_EPI_WARPS 8
#endif
constexpr int EPI_WARPS = FP8_BLOCK_EPI_WARPS;  // 8 or 16
constexpr int NUM_THREADS = 64 + EPI_WARPS * 32;
constexpr int COLS = BN * 4 / EPI_WARPS;  // accumulator columns per epilogue thread
static_assert(COLS % 32 == 0 && COLS >= 32, "each epilogue warp reads whole 32-column loads");
constexpr uint32_t TMEM_COLS = GSLOTS * KG * BN;  // 512
static_assert(TMEM_COLS == 512, "the four block slots fill TMEM");
constexpr int GROUP_M = 8;
// Scales are fetched PD groups ahead of their use.  One group (about 0.7 us
// at the block workload's speed) measured best: deeper prefetch costs
// registers the promotion needs (32768 x 8192 x 8192, PD 1/2/3: fprop 1828 /
// 1772 / 1730, wgrad 1298 / 881 / 886 TFLOP/s).
#ifndef FP8_BLOCK_PREFETCH
#define FP8_BLOCK_PREFETCH 1
#endif
constexpr int PD = FP8_BLOCK_PREFETCH;
static_assert(PD >= 1 && PD <= 4, "prefetch distance");
// per-warp B-row scales: [PD + 1 groups in flight][KG blocks][COLS]
constexpr int SBUF_FLOATS = EPI_WARPS * (PD + 1) * KG * COLS;
template <bool kPair>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)Shape<kPair>::STAGES * Shape<kPair>::STAGE_BYTES +
           SBUF_FLOATS * sizeof(float) + 256;
}
static_assert(smem_bytes<false>() <= 227 * 1024 && smem_bytes<true>() <= 227 * 1024, "smem");

struct BlockArgs {
    int M, N, K;
    BlockScales sc;
    uint16_t *d;
    int64_t ldd;
    uint64_t wait_limit_ns;
    unsigned int *status;
};

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// d = a * b + c on two fp32 lanes (each lane one IEEE fma, round to nearest)
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

template <bool kPerRowB, bool kPair>
__device__ __forceinline__ void block_gemm_body(const CUtensorMap &tma_a, const CUtensorMap &tma_b,
                                                const BlockArgs &p) {
    using S = Shape<kPair>;
    constexpr int STAGES = S::STAGES, A_STAGE = S::A_STAGE, B_STAGE = S::B_STAGE;
    constexpr int B_BLK = S::B_BLK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_STAGE;
    float *sbuf = reinterpret_cast<float *>(smem + STAGES * S::STAGE_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbuf + SBUF_FLOATS);
    uint64_t *full = bars;                // [STAGES] TMA -> MMA
    uint64_t *empty = bars + STAGES;      // [STAGES] MMA -> TMA
    uint64_t *sfull = bars + 2 * STAGES;  // [GSLOTS] MMA -> epilogue
    uint64_t *sempty = sfull + GSLOTS;    // [GSLOTS] epilogue -> MMA (the leader's, in a pair)
    uint64_t *drain = sempty + GSLOTS;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a pair's CTAs share one tile index: rank 0 (leader) holds rows 0..127
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const int unit = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int units = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    constexpr int TM = kPair ? 2 * BM : BM;  // output rows per tile
    const int m_tiles = (p.M + TM - 1) / TM, n_tiles = (p.N + BN - 1) / BN;
    const int num_tiles = m_tiles * n_tiles;
    const int nk = (p.K + BK - 1) / BK;
    const int ngroups = (nk + KG - 1) / KG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < GSLOTS; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sempty[s], kPair ? 2 * EPI_WARPS : EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tma_a);
        tma_prefetch_desc(&tma_b);
    }
    if (warp == 1) {
        if constexpr (kPair) {
            tmem_alloc_pair(tmem_holder, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_holder, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if constexpr (kPair)
        cluster_sync_all();  // barriers of both CTAs initialised before any remote use
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_wait_prior();  // set-up done; the previous kernel's results are needed from here
    pdl_allow_next();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = unit; tile < num_tiles && ok; tile += units) {
                int tm, tn;
                grouped_tile(tile, m_tiles, n_tiles, GROUP_M, tm, tn);
                const int arow = tm * TM + (int)rank * BM;
                const int brow = tn * BN + (int)rank * S::B_ROWS;
                for (int q = 0; q < ngroups; ++q) {
                    const int nb = min(KG, nk - q * KG);
                    if (!mbar_wait_bounded<true>(&empty[stage], phase ^ 1u, abort_flag,
                                                 p.wait_limit_ns, kStatusTimeoutTma, p.status)) {
                        ok = false;
                        break;
                    }
                    if constexpr (kPair) {
                        // the leader's `full` counts the bytes of both CTAs
                        if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * nb * (A_BLK + B_BLK));
                        const uint32_t leader_full = mapa_shared(smem_u32(&full[stage]), 0);
                        for (int j = 0; j < nb; ++j) {
                            const int kb = q * KG + j;
                            tma_load_2d_pair(sA + stage * A_STAGE + j * A_BLK, &tma_a, leader_full,
                                             kb * BK, arow);
                            tma_load_2d_pair(sB + stage * B_STAGE + j * B_BLK, &tma_b, leader_full,
                                             kb * BK, brow);
                        }
                    } else {
                        mbar_arrive_expect_tx(&full[stage], nb * (A_BLK + B_BLK));
                        for (int j = 0; j < nb; ++j) {
                            const int kb = q * KG + j;
                            tma_load_2d(sA + stage * A_STAGE + j * A_BLK, &tma_a, &full[stage],
                                        kb * BK, arow);
                            tma_load_2d(sB + stage * B_STAGE + j * B_BLK, &tma_b, &full[stage],
                                        kb * BK, brow);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && rank == 0) {
                // wait (bounded) for the copies still in flight before teardown
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
        if (lane == 0 && rank == 0) {
            // ------------------------------------------- MMA issuer (leader)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t g = 0;  // groups issued so far (across tiles)
            bool ok = true;
            for (int tile = unit; tile < num_tiles && ok; tile += units) {
                for (int q = 0; q < ngroups; ++q, ++g) {
                    const int nb = min(KG, nk - q * KG);
                    const uint32_t gs = g % GSLOTS, gphase = (g / GSLOTS) & 1u;
                    if (!mbar_wait_bounded<true>(&sempty[gs], gphase ^ 1u, abort_flag,
                                                 p.wait_limit_ns, kStatusTimeoutMma, p.status) ||
                        !mbar_wait_bounded<true>(&full[stage], phase, abort_flag, p.wait_limit_ns,
                                                 kStatusTimeoutMma, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int j = 0; j < nb; ++j) {
                        const uint32_t a0 = smem_u32(sA + stage * A_STAGE + j * A_BLK);
                        const uint32_t b0 = smem_u32(sB + stage * B_STAGE + j * B_BLK);
                        const uint32_t d_tmem = tmem_base + (gs * KG + j) * BN;
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            if constexpr (kPair)
                                mma_f8_pair(d_tmem, smem_desc_sw128(a0 + 32 * k),
                                            smem_desc_sw128(b0 + 32 * k), S::IDESC, k != 0);
                            else
                                mma_f8(d_tmem, smem_desc_sw128(a0 + 32 * k),
                                       smem_desc_sw128(b0 + 32 * k), S::IDESC, k != 0);
                        }
                    }
                    if constexpr (kPair) {
                        mma_commit_pair(&empty[stage], 0x3);
                        mma_commit_pair(&sfull[gs], 0x3);
                    } else {
                        mma_commit(&empty[stage]);
                        mma_commit(&sfull[gs]);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if constexpr (kPair)
                mma_commit_pair(drain, 0x1);
            else
                mma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait_bounded(drain, 0, &no_abort, p.wait_limit_ns, kStatusTimeoutMma, p.status);
        }
    } else {
        // ------------------------------------------------- epilogue (8 warps)
        const int quarter = warp & 3;
        const int group = (warp - 2) >> 2;  // columns group*COLS .. +COLS-1 of the tile
        float *wbuf = sbuf + (warp - 2) * (PD + 1) * KG * COLS;  // [PD+1][KG][COLS] B-row scales
        constexpr int PER_LANE = COLS / 32;                // B-row scales each lane stages
        const BlockScales &sc = p.sc;
        bool ok = true;
        uint32_t g = 0;
        for (int tile = unit; tile < num_tiles; tile += units) {
            int tm, tn;
            grouped_tile(tile, m_tiles, n_tiles, GROUP_M, tm, tn);
            const int row = tm * TM + (int)rank * BM + quarter * 32 + lane;
            const int j0 = tn * BN + group * COLS;  // first output column of this thread
            const float *sa_row = sc.sa + (int64_t)min(row, p.M - 1) * sc.sa_row;
            // per-tile B: one scale per block for this thread's columns (all in
            // one 128-row weight tile); per-row B: lane l stages rows
            // j0 + PER_LANE*l .. of each block's scales
            const float *sb_ptr =
                kPerRowB ? sc.sb + (int64_t)min(j0 + PER_LANE * lane, p.N - PER_LANE) * sc.sb_row
                         : sc.sb + (int64_t)(min(j0, p.N - 1) / sc.b_rows) * sc.sb_row;
            // fp32 accumulators: in pairs for per-tile B (one packed FMA per
            // pair), single for per-row B (a multiply and an FMA per element
            // measured faster there than their packed forms: 1356 against
            // 1297 TFLOP/s for wgrad at 32768 x 8192 x 8192)
            uint64_t acc[COLS / 2];
            float accs[COLS];
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) acc[j] = 0ull;
#pragma unroll
            for (int j = 0; j < COLS; ++j) accs[j] = 0.f;
            // scalar scales of the next PD groups (contraction blocks past the
            // end read the last block's scales and go unused)
            float sa_pf[PD][KG], sb_pf[PD][KG];
            auto fetch = [&](int qn, float (&sa)[KG], float (&sb)[KG]) {
#pragma unroll
                for (int j = 0; j < KG; ++j) {
                    const int kb = min(qn * KG + j, nk - 1);
                    sa[j] = sa_row[(int64_t)kb * sc.sa_k];
                    sb[j] = kPerRowB ? 0.f : sb_ptr[(int64_t)kb * sc.sb_k];
                }
            };
#pragma unroll
            for (int d = 0; d < PD; ++d) fetch(d, sa_pf[d], sb_pf[d]);
            // per-row B: one cp.async group per contraction group (empty past
            // the end, so that wait_group counts stay uniform)
            auto stage_scales = [&](int qn) {
                const int nbn = qn < ngroups ? min(KG, nk - qn * KG) : 0;
                for (int j = 0; j < nbn; ++j) {
                    const float *src = sb_ptr + (int64_t)(qn * KG + j) * sc.sb_k;
                    float *dst = wbuf + ((qn % (PD + 1)) * KG + j) * COLS + PER_LANE * lane;
                    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)),
                                 "l"(src), "n"(PER_LANE * 4)
                                 : "memory");
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
            };
            if (kPerRowB)
                for (int d = 0; d < PD; ++d) stage_scales(d);
            for (int q = 0; q < ngroups; ++q, ++g) {
                const int nb = min(KG, nk - q * KG);
                const uint32_t gs = g % GSLOTS, gphase = (g / GSLOTS) & 1u;
                float sa_cur[KG], sb_cur[KG];
#pragma unroll
                for (int j = 0; j < KG; ++j) {
                    sa_cur[j] = sa_pf[0][j];
                    sb_cur[j] = sb_pf[0][j];
                }
#pragma unroll
                for (int d = 0; d + 1 < PD; ++d)
#pragma unroll
                    for (int j = 0; j < KG; ++j) {
                        sa_pf[d][j] = sa_pf[d + 1][j];
                        sb_pf[d][j] = sb_pf[d + 1][j];
                    }
                fetch(q + PD, sa_pf[PD - 1], sb_pf[PD - 1]);
                if (kPerRowB) {
                    // this group's copies were the oldest of PD in flight
                    asm volatile("cp.async.wait_group %0;" ::"n"(PD - 1) : "memory");
                    __syncwarp();  // every lane's part of this group's scales has landed
                    stage_scales(q + PD);
                }
                if (ok)
                    ok = mbar_wait_bounded<true>(&sfull[gs], gphase, abort_flag, p.wait_limit_ns,
                                                 kStatusTimeoutEpilogue, p.status);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) continue;  // outputs invalid; keep the loop shape
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < KG; ++j) {
                    if (j >= nb) break;
                    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                           (gs * KG + j) * BN + (uint32_t)(group * COLS);
                    uint32_t r[COLS / 32][32];
#pragma unroll
                    for (int c = 0; c < COLS / 32; ++c)
                        tmem_ld_32x32b_x32(taddr + 32 * c, r[c]);
                    tmem_ld_wait();
                    if (j == nb - 1) {  // the group's last partial is in registers
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (kPair)
                                mbar_arrive_cluster(mapa_shared(smem_u32(&sempty[gs]), 0));
                            else
                                mbar_arrive(&sempty[gs]);
                        }
                    }
                    const float *buf = wbuf + ((q % (PD + 1)) * KG + j) * COLS;
                    const float f1 = sa_cur[j] * sb_cur[j];
                    const uint64_t fts = pack2(f1, f1);
                    if constexpr (kPerRowB) {
#pragma unroll
                        for (int a = 0; a < COLS; ++a) {
                            const float f = __fmul_rn(buf[a], sa_cur[j]);
                            accs[a] = __fmaf_rn(__uint_as_float(r[a / 32][a % 32]), f, accs[a]);
                        }
                    } else {
#pragma unroll
                        for (int a = 0; a < COLS / 2; ++a) {
                            const uint64_t pv =
                                pack2(__uint_as_float(r[a / 16][(2 * a) % 32]),
                                      __uint_as_float(r[a / 16][(2 * a) % 32 + 1]));
                            acc[a] = fma2(pv, fts, acc[a]);
                        }
                    }
                }
            }
            if (ok && row < p.M && j0 < p.N) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.d + (int64_t)row * p.ldd + j0);
#pragma unroll
                for (int c = 0; c < COLS / 8; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if constexpr (kPerRowB) {
                            v[2 * e] = accs[8 * c + 2 * e];
                            v[2 * e + 1] = accs[8 * c + 2 * e + 1];
                        } else {
                            unpack2(acc[4 * c + e], v[2 * e], v[2 * e + 1]);
                        }
                    }
                    dst[c] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                        pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                }
            }
        }
    }

    __syncwarp();  // lanes that skipped a role wait here for their warp's lane 0
    tc_fence_before();
    if constexpr (kPair)
        cluster_sync_all();  // the peer's smem/TMEM stay alive until the leader's MMAs drained
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <bool kPerRowB>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_f8_block_kernel(const __grid_constant__ CUtensorMap tma_a,
                         const __grid_constant__ CUtensorMap tma_b, const BlockArgs p) {
    block_gemm_body<kPerRowB, false>(tma_a, tma_b, p);
}

template <bool kPerRowB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_f8_block_pair_kernel(const __grid_constant__ CUtensorMap tma_a,
                              const __grid_constant__ CUtensorMap tma_b, const BlockArgs p) {
    block_gemm_body<kPerRowB, true>(tma_a, tma_b, p);
}

template <bool kPerRowB, bool kPair>
cudaError_t launch_block(const CUtensorMap &ta, const CUtensorMap &tb, const BlockArgs &args,
                         int grid, cudaStream_t s) {
    auto kernel = kPair ? gemm_f8_block_pair_kernel<kPerRowB> : gemm_f8_block_kernel<kPerRowB>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_bytes<kPair>());
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    return launch_pdl(kernel, grid, NUM_THREADS, smem_bytes<kPair>(), s, ta, tb, args);
}

template <bool kPair>
cudaError_t launch_shape(const uint8_t *A, const uint8_t *B, const BlockArgs &args,
                         cudaStream_t s, const char **why) {
    CUtensorMap ta, tb;
    if (!make_tmap_k128(&ta, A, args.M, args.K, BM) ||
        !make_tmap_k128(&tb, B, args.N, args.K, Shape<kPair>::B_ROWS)) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    const int64_t tm = kPair ? 2 * BM : BM;
    const int64_t tiles = ((args.M + tm - 1) / tm) * ((args.N + BN - 1) / BN);
    const int64_t units = kPair ? num_sms() / 2 : num_sms();
    const int grid = (int)(tiles < units ? tiles : units) * (kPair ? 2 : 1);
    if (args.sc.b_rows == 1) return launch_block<true, kPair>(ta, tb, args, grid, s);
    if (args.sc.b_rows == 128) return launch_block<false, kPair>(ta, tb, args, grid, s);
    *why = "B scales must be per row or per 128-row tile";
    return cudaErrorInvalidValue;
}

}  // namespace

// One-CTA tiles by default.  The pair kernel streams half as many B bytes per
// SM but measured no faster (32768 x 8192 x 8192: fprop 1857 vs 1845 TFLOP/s,
// wgrad 1119 vs 1187): at this tile width both run into the promotion's cost
// per block, not the operand traffic.  FP8LINEAR_BLOCK_PAIR=1 selects it (the
// tests run both kernels).
cudaError_t launch_gemm_block(const uint8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K,
                              const BlockScales &sc, uint16_t *D, cudaStream_t s,
                              const char **why) {
    BlockArgs args;
    args.M = (int)M;
    args.N = (int)N;
    args.K = (int)K;
    args.sc = sc;
    args.d = D;
    args.ldd = N;
    args.wait_limit_ns = g_wait_limit_ns;
    args.status = device_status_word();
    const char *pe = getenv("FP8LINEAR_BLOCK_PAIR");
    const int pair_mode = pe ? atoi(pe) : -1;
    return pair_mode == 1 ? launch_shape<true>(A, B, args, s, why)
                          : launch_shape<false>(A, B, args, s, why);
}

}  // namespace fp8
