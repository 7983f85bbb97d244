// Block-scaled FP8 GEMM (the TE "recipe=block" layout: 1x128 tiles along the
// contraction dim for activations and gradients, 128x128 tiles for weights).
//
//   D[i,j] = bf16( sum_kb sA(i,kb) * sB(j,kb) * sum_{k in block kb} A[i,k] B[j,k] )
//
// One persistent CTA per SM owns 128 x 256 (or 128 x 128) output tiles.  The
// contraction is walked in groups (one 128-deep block for 256-wide tiles, two
// for 128-wide ones): one TMA stage, one round of MMAs and one hand-off per
// group.  The MMA warp writes each block's partial product (fresh
// accumulation) into its own TMEM slot; the slots form two group slots, so
// the MMAs of one group run while the promotion reads the other.  Eight
// epilogue warps (two per TMEM lane quarter, half the tile's columns each)
// read a group's partials back, hand the group slot back after the last read
// and fold each partial into fp32 register accumulators with its two block
// scales (a packed fp32x2 FMA per pair for per-tile B; a multiply and an FMA
// per element or pair for per-row B).  A hand-off costs a few hundred cycles
// of barrier traffic whatever it carries, so each carries 128 x 256 partial
// products.  B's scale is one value per 128-row tile (weights) or one per row
// (wgrad's Xᵀ operand: each warp stages its columns' scales of the next group
// into shared memory with cp.async, from a layout contiguous over rows; with
// wide tiles each thread reads four rows x 32 columns of the partial, so that
// it needs a quarter of those scales).  Every handshake is local to the SM
// (or the CTA pair), and every wait is bounded, as in the other GEMM kernels.
//
// The same pipeline also runs on CTA pairs (tcgen05 cta_group::2,
// as in the tensorwise pair kernel): a pair owns a 256 x BN tile, each CTA
// loads its 128 rows of A and BN/2 rows of B, the leader issues M=256 MMAs
// whose rows land in both CTAs' TMEM, commits multicast to both, and both
// CTAs' epilogue warps hand group slots back to the leader.  Each SM then
// streams half of B's bytes, with the same promotion work per SM.
#include <cuda.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8 {

extern std::atomic<uint64_t> g_wait_limit_ns;

namespace {

constexpr int BM = 128, BK = 128;
constexpr int GSLOTS = 2;  // group slots of KG TMEM slots each
constexpr int A_BLK = BM * BK;
constexpr int EPI_WARPS = 8;
// Scales are fetched PD groups ahead of their use.  One group (about 0.7 us
// at the block workload's speed) measured best: deeper prefetch costs
// registers the promotion needs (32768 x 8192 x 8192, PD 1/2/3: fprop 1828 /
// 1772 / 1730, wgrad 1298 / 881 / 886 TFLOP/s).
// Wide tiles: the TMEM load of the next 32-column chunk is in flight while
// the current chunk is folded in (wgrad 1476 against 1449 TFLOP/s without;
// fprop unchanged at 2552-2554).
#ifndef FP8_BLOCK_PIPE
#define FP8_BLOCK_PIPE 1
#endif
#ifndef FP8_BLOCK_PREFETCH
#define FP8_BLOCK_PREFETCH 1
#endif
constexpr int PD = FP8_BLOCK_PREFETCH;
static_assert(PD >= 1 && PD <= 4, "prefetch distance");

// Tile geometry.  kBN = 128: two contraction blocks per group in four
// 128-column TMEM slots, 64 accumulator columns per epilogue thread; warps 0
// (TMA) and 1 (MMA) then the epilogue warps, 10 in all, which caps a thread at
// 168 registers (three warps share some SM sub-partitions).  kBN = 256: one
// block per group in two 256-column slots and 128 accumulator columns per
// thread, which do not fit in 168 registers: the CTA has three warpgroups
// (TMA, MMA and two idle warps; then the eight epilogue warps) and moves
// registers from the first to the others with setmaxnreg, 40 + 2 x 232 per
// lane of a warp triple = 3 x 168, the launch's own allocation.  Either way a
// hand-off carries 128 x 256 partial products.
template <bool kPair, int kBN> struct Shape {
    static constexpr int BN = kBN;
    static constexpr int KG = kBN == 256 ? 1 : 2;  // contraction blocks per group
    // B rows each CTA loads per block: the whole N tile, or half of it in a pair
    static constexpr int B_ROWS = kPair ? BN / 2 : BN;
    static constexpr int B_BLK = B_ROWS * BK;
    static constexpr int A_STAGE = KG * A_BLK, B_STAGE = KG * B_BLK;
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
    static constexpr int STAGES = (192 * 1024) / STAGE_BYTES;  // TMA ring depth, in groups
    static constexpr uint32_t IDESC = idesc_f8_f32(kPair ? 2 * BM : BM, BN);
    static constexpr int COLS = BN * 4 / EPI_WARPS;  // accumulator columns per epilogue thread
    // 32-column TMEM loads per wait: with 128 accumulator columns a second
    // load in flight costs more in registers than it saves in latency
    // (32768 x 8192 x 8192, one CTA: fprop 2582 / 2565 / 2029 TFLOP/s for 1 /
    // 2 / 4 loads per wait)
    static constexpr int CH = COLS >= 128 ? 1 : 2;
    // per-row B, wide tiles: each epilogue thread reads four rows x 32
    // columns of the accumulator (16-lane TMEM loads) instead of one row x 128
    // columns, so that it needs 32 column scales per block instead of 128: the
    // broadcast shared-memory loads of those scales, not the arithmetic, bound
    // the one-row form (ncu: 639 M shared wavefronts per wgrad launch, L1 83 %
    // busy).  128-wide tiles keep one row per thread with scalar arithmetic
    // (1374 TFLOP/s against 1265 for packed pairs at 168 registers).
    static constexpr bool ROWS4 = kBN == 256;
    static constexpr uint32_t TMEM_COLS = GSLOTS * KG * BN;
    static constexpr bool SPLIT_REGS = kBN == 256;
    static constexpr int EPI0 = SPLIT_REGS ? 4 : 2;  // first epilogue warp
    static constexpr int THREADS = 32 * (EPI0 + EPI_WARPS);
    static constexpr int REGS_LOW = 40, REGS_HIGH = 232;
    static_assert(!SPLIT_REGS || 128 * REGS_LOW + 256 * REGS_HIGH <= 384 * 168,
                  "the register split fits the 384-thread launch's allocation");
    // per-warp B-row scales: [PD + 1 groups in flight][KG blocks][COLS]
    static constexpr int SBUF_FLOATS = EPI_WARPS * (PD + 1) * KG * COLS;
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES +
                                   SBUF_FLOATS * sizeof(float) + 256;
    static_assert(COLS % 32 == 0 && COLS >= 32, "each epilogue warp reads whole 32-column loads");
    static_assert((COLS / 32) % CH == 0, "loads per wait divide a thread's columns");
    static_assert(TMEM_COLS == 512, "the block slots fill TMEM");
    static_assert(STAGES >= 3, "TMA ring depth");
    static_assert(SMEM <= 227 * 1024, "smem");
};

struct BlockArgs {
    int M, N, K;
    BlockScales sc;
    uint16_t *d;
    int64_t ldd;
    int group_m;  // row tiles per raster group (block_raster_group)
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

// d = a * b on two fp32 lanes (round to nearest)
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// d = a * b + c on two fp32 lanes (each lane one IEEE fma, round to nearest)
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// A pair of fp32 accumulators, kept either packed in one 64-bit register
// (folded in with one fma.rn.f32x2, whose first operand, two TMEM values,
// must first be moved into an aligned register pair) or as two scalars
// (folded in with two fma.rn on the TMEM registers as they are).  Both do the
// same two IEEE fmas, so the results are identical.
struct F2 {
    float x, y;
};

__device__ __forceinline__ void acc_zero(uint64_t &a) { a = 0ull; }
__device__ __forceinline__ void acc_zero(F2 &a) { a.x = a.y = 0.f; }

// a += (p0, p1) * f2, lane by lane
__device__ __forceinline__ void acc_fma(uint64_t &a, uint32_t p0, uint32_t p1, uint64_t f2) {
    uint64_t pv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(pv) : "r"(p0), "r"(p1));
    a = fma2(pv, f2, a);
}
__device__ __forceinline__ void acc_fma(F2 &a, uint32_t p0, uint32_t p1, uint64_t f2) {
    float f0, f1;
    unpack2(f2, f0, f1);
    a.x = __fmaf_rn(__uint_as_float(p0), f0, a.x);
    a.y = __fmaf_rn(__uint_as_float(p1), f1, a.y);
}

__device__ __forceinline__ uint32_t acc_bf16x2(uint64_t a) {
    float lo, hi;
    unpack2(a, lo, hi);
    return pack_bf16x2(lo, hi);
}
__device__ __forceinline__ uint32_t acc_bf16x2(const F2 &a) { return pack_bf16x2(a.x, a.y); }

template <bool kPerRowB, bool kPair, int kBN, bool kScalar = false>
__device__ __forceinline__ void block_gemm_body(const CUtensorMap &tma_a, const CUtensorMap &tma_b,
                                                const BlockArgs &p) {
    using AccT = typename std::conditional<kScalar, F2, uint64_t>::type;
    using S = Shape<kPair, kBN>;
    constexpr int STAGES = S::STAGES, A_STAGE = S::A_STAGE, B_STAGE = S::B_STAGE;
    constexpr int B_BLK = S::B_BLK, BN = S::BN, KG = S::KG, COLS = S::COLS, CH = S::CH;
    constexpr int SBUF_FLOATS = S::SBUF_FLOATS;
    constexpr uint32_t TMEM_COLS = S::TMEM_COLS;
    constexpr int EPI0 = S::EPI0;
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
    // register split (wide tiles): each warp of the first warpgroup gives
    // registers back as it enters its role, each epilogue warp takes more;
    // inside the branches so that the compiler sizes each role to its limit
    auto regs_low = [] {
        if constexpr (S::SPLIT_REGS)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(S::REGS_LOW));
    };

    if (warp == 0) {
        regs_low();
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = unit; tile < num_tiles && ok; tile += units) {
                int tm, tn;
                grouped_tile(tile, m_tiles, n_tiles, p.group_m, tm, tn);
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
        regs_low();
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
    } else if (warp < EPI0) {
        regs_low();  // idle warps of the first warpgroup
    } else {
        // ------------------------------------------------- epilogue (8 warps)
        if constexpr (S::SPLIT_REGS)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(S::REGS_HIGH));
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int group = (warp - EPI0) >> 2;  // columns group*COLS .. +COLS-1 of the tile
        float *wbuf = sbuf + (warp - EPI0) * (PD + 1) * KG * COLS;  // [PD+1][KG][COLS] B-row scales
        constexpr int PER_LANE = COLS / 32;                // B-row scales each lane stages
        const BlockScales &sc = p.sc;
        bool ok = true;
        uint32_t g = 0;
        if constexpr (kPerRowB && S::ROWS4) {
            // Four-row fragments: thread t of a warp holds rows 8i + t/4
            // (i = 0..3) of its lane quarter and, in each 8-column group j of
            // its COLS columns, columns 8j + 2(t%4) and +1, as packed pairs.
            static_assert(KG == 1 && CH == 1, "wide tiles: one block per group");
            const int fr = lane >> 2, fc = lane & 3;
            for (int tile = unit; tile < num_tiles; tile += units) {
                int tm, tn;
                grouped_tile(tile, m_tiles, n_tiles, p.group_m, tm, tn);
                const int row0 = tm * TM + (int)rank * BM + quarter * 32 + fr;
                const int j0 = tn * BN + group * COLS;
                const float *sa_rows[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    sa_rows[i] = sc.sa + (int64_t)min(row0 + 8 * i, p.M - 1) * sc.sa_row;
                const float *sb_ptr =
                    sc.sb + (int64_t)min(j0 + PER_LANE * lane, p.N - PER_LANE) * sc.sb_row;
                AccT acc[4][COLS / 8];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < COLS / 8; ++j) acc_zero(acc[i][j]);
                float sa_pf[PD][4];
                auto fetch = [&](int qn, float (&sa)[4]) {
                    const int kb = min(qn, nk - 1);
#pragma unroll
                    for (int i = 0; i < 4; ++i) sa[i] = sa_rows[i][(int64_t)kb * sc.sa_k];
                };
#pragma unroll
                for (int d = 0; d < PD; ++d) fetch(d, sa_pf[d]);
                auto stage_scales = [&](int qn) {
                    if (qn < ngroups) {
                        const float *src = sb_ptr + (int64_t)qn * sc.sb_k;
                        float *dst = wbuf + (qn % (PD + 1)) * COLS + PER_LANE * lane;
                        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)),
                                     "l"(src), "n"(PER_LANE * 4)
                                     : "memory");
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                };
                for (int d = 0; d < PD; ++d) stage_scales(d);
                for (int q = 0; q < ngroups; ++q, ++g) {
                    const uint32_t gs = g % GSLOTS, gphase = (g / GSLOTS) & 1u;
                    uint64_t sa2[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) sa2[i] = pack2(sa_pf[0][i], sa_pf[0][i]);
#pragma unroll
                    for (int d = 0; d + 1 < PD; ++d)
#pragma unroll
                        for (int i = 0; i < 4; ++i) sa_pf[d][i] = sa_pf[d + 1][i];
                    fetch(q + PD, sa_pf[PD - 1]);
                    asm volatile("cp.async.wait_group %0;" ::"n"(PD - 1) : "memory");
                    __syncwarp();
                    stage_scales(q + PD);
                    if (ok)
                        ok = mbar_wait_bounded<true>(&sfull[gs], gphase, abort_flag,
                                                     p.wait_limit_ns, kStatusTimeoutEpilogue,
                                                     p.status);
                    ok = __all_sync(0xFFFFFFFFu, ok);
                    if (!ok) continue;
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                           gs * BN + (uint32_t)(group * COLS);
                    const float *buf = wbuf + (q % (PD + 1)) * COLS + 2 * fc;
                    auto hand_back = [&] {  // the block's partial is in registers
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (kPair)
                                mbar_arrive_cluster(mapa_shared(smem_u32(&sempty[gs]), 0));
                            else
                                mbar_arrive(&sempty[gs]);
                        }
                    };
                    // chunk c's lanes +0..15 / +16..31 of the quarter in
                    // ra / rb [c % 2]; with FP8_BLOCK_PIPE the load of chunk
                    // c + 1 is in flight while chunk c is folded in.  Scalar
                    // accumulators take 16-column chunks (8 registers per
                    // load instead of 16), which keeps the per-thread total
                    // of 128 accumulators plus the two chunks in flight
                    // within the 232 registers of the epilogue warps.
                    constexpr int CW = kScalar ? 16 : 32;  // columns per chunk
                    constexpr int NC = COLS / CW, JJ = CW / 8, R = CW / 2;
                    auto ld = [&](uint32_t addr, uint32_t(&r)[R]) {
                        if constexpr (R == 8)
                            tmem_ld_16x256b_x2(addr, r);
                        else
                            tmem_ld_16x256b_x4(addr, r);
                    };
                    uint32_t ra[2][R], rb[2][R];
                    if (FP8_BLOCK_PIPE) {
                        ld(taddr, ra[0]);
                        ld(taddr + (16u << 16), rb[0]);
                        tmem_ld_wait();
                        tmem_regs_ready(ra[0]);
                        tmem_regs_ready(rb[0]);
                        if (NC == 1) hand_back();
                    }
#pragma unroll
                    for (int c0 = 0; c0 < NC; ++c0) {
                        uint32_t(&r0)[R] = ra[c0 & 1];
                        uint32_t(&r1)[R] = rb[c0 & 1];
                        if (!FP8_BLOCK_PIPE) {
                            ld(taddr + CW * c0, r0);
                            ld(taddr + (16u << 16) + CW * c0, r1);
                            tmem_ld_wait();
                            tmem_regs_ready(r0);
                            tmem_regs_ready(r1);
                            if (c0 + 1 == NC) hand_back();
                        } else if (c0 + 1 < NC) {
                            ld(taddr + CW * (c0 + 1), ra[(c0 + 1) & 1]);
                            ld(taddr + (16u << 16) + CW * (c0 + 1), rb[(c0 + 1) & 1]);
                        }
#pragma unroll
                        for (int jj = 0; jj < JJ; ++jj) {
                            const int j = JJ * c0 + jj;
                            const float2 sbv = *reinterpret_cast<const float2 *>(buf + 8 * j);
                            const uint64_t sb2 = pack2(sbv.x, sbv.y);
                            acc_fma(acc[0][j], r0[4 * jj], r0[4 * jj + 1], mul2(sb2, sa2[0]));
                            acc_fma(acc[1][j], r0[4 * jj + 2], r0[4 * jj + 3], mul2(sb2, sa2[1]));
                            acc_fma(acc[2][j], r1[4 * jj], r1[4 * jj + 1], mul2(sb2, sa2[2]));
                            acc_fma(acc[3][j], r1[4 * jj + 2], r1[4 * jj + 3], mul2(sb2, sa2[3]));
                        }
                        if (FP8_BLOCK_PIPE && c0 + 1 < NC) {
                            tmem_ld_wait();
                            tmem_regs_ready(ra[(c0 + 1) & 1]);
                            tmem_regs_ready(rb[(c0 + 1) & 1]);
                            if (c0 + 2 == NC) hand_back();
                        }
                    }
                }
                if (ok && j0 < p.N) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = row0 + 8 * i;
                        if (row >= p.M) continue;
                        uint32_t *dst = reinterpret_cast<uint32_t *>(p.d + (int64_t)row * p.ldd + j0 + 2 * fc);
#pragma unroll
                        for (int j = 0; j < COLS / 8; ++j) dst[4 * j] = acc_bf16x2(acc[i][j]);
                    }
                }
            }
        } else {
        for (int tile = unit; tile < num_tiles; tile += units) {
            int tm, tn;
            grouped_tile(tile, m_tiles, n_tiles, p.group_m, tm, tn);
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
            AccT acc[COLS / 2];
            float accs[COLS];
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) acc_zero(acc[j]);
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
                    const float *buf = wbuf + ((q % (PD + 1)) * KG + j) * COLS;
                    const float f1 = sa_cur[j] * sb_cur[j];
                    const uint64_t fts = pack2(f1, f1);
                    auto hand_back = [&] {  // the group's last partial is in registers
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (kPair)
                                mbar_arrive_cluster(mapa_shared(smem_u32(&sempty[gs]), 0));
                            else
                                mbar_arrive(&sempty[gs]);
                        }
                    };
                    // one 32-column load per wait (wide tiles): with
                    // FP8_BLOCK_PIPE the next chunk's load is in flight while
                    // the current one is folded in
                    constexpr bool kPipe = FP8_BLOCK_PIPE && CH == 1;
                    constexpr int NC = COLS / 32;
                    uint32_t rp[2][32];
                    if constexpr (kPipe) {
                        tmem_ld_32x32b_x32(taddr, rp[0]);
                        tmem_ld_wait();
                        tmem_regs_ready(rp[0]);
                        if (NC == 1 && j == nb - 1) hand_back();
                    }
#pragma unroll
                    for (int c0 = 0; c0 < COLS / 32; c0 += CH) {
                        uint32_t rl[CH][32];
                        if constexpr (!kPipe) {
#pragma unroll
                            for (int c = 0; c < CH; ++c)
                                tmem_ld_32x32b_x32(taddr + 32 * (c0 + c), rl[c]);
                            tmem_ld_wait();
                            if (j == nb - 1 && c0 + CH == COLS / 32) hand_back();
                        } else if (c0 + 1 < NC) {
                            tmem_ld_32x32b_x32(taddr + 32 * (c0 + 1), rp[(c0 + 1) & 1]);
                        }
                        uint32_t(&r)[CH][32] = *reinterpret_cast<uint32_t(*)[CH][32]>(
                            kPipe ? &rp[c0 & 1][0] : &rl[0][0]);
                        if constexpr (kPerRowB) {
#pragma unroll
                            for (int a = 0; a < 32 * CH; ++a) {
                                const float f = __fmul_rn(buf[32 * c0 + a], sa_cur[j]);
                                accs[32 * c0 + a] =
                                    __fmaf_rn(__uint_as_float(r[a / 32][a % 32]), f, accs[32 * c0 + a]);
                            }
                        } else {
#pragma unroll
                            for (int a = 0; a < 16 * CH; ++a)
                                acc_fma(acc[16 * c0 + a], r[a / 16][(2 * a) % 32],
                                        r[a / 16][(2 * a) % 32 + 1], fts);
                        }
                        if constexpr (kPipe) {
                            if (c0 + 1 < NC) {
                                tmem_ld_wait();
                                tmem_regs_ready(rp[(c0 + 1) & 1]);
                                if (c0 + 2 == NC && j == nb - 1) hand_back();
                            }
                        }
                    }
                }
            }
            if (ok && row < p.M && j0 < p.N) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.d + (int64_t)row * p.ldd + j0);
#pragma unroll
                for (int c = 0; c < COLS / 8; ++c) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if constexpr (kPerRowB)
                            w[e] = pack_bf16x2(accs[8 * c + 2 * e], accs[8 * c + 2 * e + 1]);
                        else
                            w[e] = acc_bf16x2(acc[4 * c + e]);
                    }
                    dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        }  // one-row epilogue
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

template <bool kPerRowB, int kBN, bool kScalar>
__global__ void __launch_bounds__(Shape<false, kBN>::THREADS, 1)
    gemm_f8_block_kernel(const __grid_constant__ CUtensorMap tma_a,
                         const __grid_constant__ CUtensorMap tma_b, const BlockArgs p) {
    block_gemm_body<kPerRowB, false, kBN, kScalar>(tma_a, tma_b, p);
}

template <bool kPerRowB, int kBN, bool kScalar>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Shape<true, kBN>::THREADS, 1)
    gemm_f8_block_pair_kernel(const __grid_constant__ CUtensorMap tma_a,
                              const __grid_constant__ CUtensorMap tma_b, const BlockArgs p) {
    block_gemm_body<kPerRowB, true, kBN, kScalar>(tma_a, tma_b, p);
}

template <bool kPerRowB, bool kPair, int kBN, bool kScalar>
cudaError_t launch_block(const CUtensorMap &ta, const CUtensorMap &tb, const BlockArgs &args,
                         int grid, cudaStream_t s, const char **why) {
    using S = Shape<kPair, kBN>;
    auto kernel = kPair ? gemm_f8_block_pair_kernel<kPerRowB, kBN, kScalar>
                        : gemm_f8_block_kernel<kPerRowB, kBN, kScalar>;
    constexpr size_t smem = S::SMEM;
    static std::atomic<bool> attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (S::SPLIT_REGS) {
            // setmaxnreg.inc waits until the CTA's own register allocation
            // (threads x registers per thread at launch) can supply the
            // raised counts; a build that launched with fewer registers than
            // the split assumes would wait forever, so it is refused here
            cudaFuncAttributes fa;
            cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            if ((int64_t)fa.numRegs * S::THREADS <
                (int64_t)128 * S::REGS_LOW + (int64_t)(S::THREADS - 128) * S::REGS_HIGH) {
                *why = "block GEMM: the register split does not fit the kernel's launch allocation";
                return cudaErrorInvalidConfiguration;
            }
        }
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    return launch_pdl(kernel, grid, S::THREADS, smem, s, ta, tb, args);
}

// Row tiles per raster group.  The CTAs running at one time cover `group`
// row tiles by units/group column tiles, and each streams its row panel of A
// (tm rows) and column panel of B (bn rows) over the whole contraction; with
// the panels in L2 while that wave runs, the wave reads
// group * tm + ceil(units / group) * bn rows of contraction bytes from DRAM,
// which this minimises (for 32768 x 8192 x 8192 on 152 SMs: 17 row tiles of
// 128 by 9 column tiles of 256, against the 8 by 19 of a fixed group of 8).
int block_raster_group(int64_t m_tiles, int64_t units, int tm, int bn) {
    int best = 1;
    int64_t best_rows = INT64_MAX;
    for (int64_t g = 1; g <= m_tiles && g <= units; ++g) {
        const int64_t rows = g * tm + ((units + g - 1) / g) * bn;
        if (rows < best_rows) {
            best_rows = rows;
            best = (int)g;
        }
    }
    return best;
}

template <bool kPair, int kBN, bool kScalar>
cudaError_t launch_shape(const uint8_t *A, const uint8_t *B, const BlockArgs &args_in,
                         cudaStream_t s, const char **why) {
    BlockArgs args = args_in;
    CUtensorMap ta, tb;
    if (!make_tmap_k128(&ta, A, args.M, args.K, BM) ||
        !make_tmap_k128(&tb, B, args.N, args.K, Shape<kPair, kBN>::B_ROWS)) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    const int64_t tm = kPair ? 2 * BM : BM;
    const int64_t tiles = ((args.M + tm - 1) / tm) * ((args.N + kBN - 1) / kBN);
    const int64_t units = kPair ? num_sms() / 2 : num_sms();
    const int grid = (int)(tiles < units ? tiles : units) * (kPair ? 2 : 1);
    const char *ge = getenv("FP8LINEAR_BLOCK_GROUP");
    args.group_m = ge != nullptr && atoi(ge) > 0
                       ? atoi(ge)
                       : block_raster_group((args.M + tm - 1) / tm, units, (int)tm, kBN);
    if (args.sc.b_rows == 1) return launch_block<true, kPair, kBN, kScalar>(ta, tb, args, grid, s, why);
    if (args.sc.b_rows == 128) return launch_block<false, kPair, kBN, kScalar>(ta, tb, args, grid, s, why);
    *why = "B scales must be per row or per 128-row tile";
    return cudaErrorInvalidValue;
}

}  // namespace

// Kernel choice, measured at 32768 x 8192 x 8192 (TFLOP/s):
//                       one CTA 128   one CTA 256   pair 128   pair 256
//   per-tile B (fprop)      1829          2541-2561     1697       2570-2593
//   per-row B (wgrad)       1374          1627-1636     1311       1633-1650
// (256-wide tiles: packed accumulators for per-tile B, scalar ones for
// per-row B.)  CTA pairs with 256-wide tiles by default; problems with fewer
// 128 x 256 tiles than SMs take one CTA with 128-wide tiles.
// FP8LINEAR_BLOCK_PAIR=0/1, FP8LINEAR_BLOCK_BN=128/256, FP8LINEAR_BLOCK_ACC=0/1
// and FP8LINEAR_BLOCK_GROUP=<row tiles> override the choice (the tests run
// every kernel).
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
    args.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    args.status = device_status_word();
    const char *pe = getenv("FP8LINEAR_BLOCK_PAIR");
    const char *be = getenv("FP8LINEAR_BLOCK_BN");
    const bool wide = be != nullptr ? atoi(be) == 256
                                    : ((M + 127) / 128) * ((N + 255) / 256) >= num_sms();
    // CTA pairs for wide tiles (each SM streams half of B's bytes), one CTA for
    // narrow ones; FP8LINEAR_BLOCK_PAIR=0/1 overrides
    const bool pair = pe != nullptr ? atoi(pe) == 1 : wide;
    // wide tiles, per-row B: scalar accumulators (below); FP8LINEAR_BLOCK_ACC=0/1 overrides
    const char *ae = getenv("FP8LINEAR_BLOCK_ACC");
    const bool scalar = ae != nullptr ? atoi(ae) == 1 : sc.b_rows == 1;
    if (wide) {
        if (scalar)
            return pair ? launch_shape<true, 256, true>(A, B, args, s, why)
                        : launch_shape<false, 256, true>(A, B, args, s, why);
        return pair ? launch_shape<true, 256, false>(A, B, args, s, why)
                    : launch_shape<false, 256, false>(A, B, args, s, why);
    }
    return pair ? launch_shape<true, 128, false>(A, B, args, s, why)
                : launch_shape<false, 128, false>(A, B, args, s, why);
}

}  // namespace fp8
