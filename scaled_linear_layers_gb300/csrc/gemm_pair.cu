// Scaled FP8 GEMM with 2-SM MMAs (tcgen05 cta_group::2) for large problems.
//
//   D[M,N] = bf16( s_A * s_B * sum_k A[m,k] * B[n,k] (+ bias[n]) )
//
// A cluster of two CTAs on neighbouring SMs owns a 256 x BN output tile.  CTA
// r (0 = leader, 1 = peer) loads rows r*128..+127 of the tile's A panel and
// rows r*BN/2..+BN/2-1 of its B panel into its own shared memory; one thread
// of the leader issues M=256 x N=BN x K=32 MMAs that read both CTAs' shared
// memory and write rows 0..127 of the accumulator to the leader's TMEM and
// rows 128..255 to the peer's.  Each SM therefore streams 128 x (128 + BN/2)
// operand bytes per 128-deep contraction block instead of 128 x (128 + BN),
// which is what limits the one-CTA kernel.
//
// One launch may carry two independent problems (a backward pass's dgrad and
// wgrad): their tiles form one index space that the persistent pairs walk,
// so the two GEMMs share waves instead of each ending in a partial one.
//
// Synchronisation: both CTAs' TMA loads complete on the leader's `full`
// barrier (which expects the bytes of both); the leader's MMA commits arrive
// on `empty` and `tfull` in both CTAs at once (multicast); both CTAs'
// epilogue warps arrive on the leader's `tempty`.  Every wait is bounded; the
// CTAs of a pair meet at cluster barriers after set-up and before teardown.
#include <cuda.h>

#include <atomic>
#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace fp8 {

extern std::atomic<uint64_t> g_wait_limit_ns;

namespace {

constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int GROUP_M = 4;  // 4 pair-rows of 256 = 1024 rows per raster group
constexpr size_t SMEM_LIMIT = 227 * 1024;

// A stage holds KSUB 128-byte-wide boxes of each operand (contraction depth
// 128*KSUB): narrower N tiles take two boxes per stage so each barrier round
// trip covers 8 MMAs (measured: +7% at 4096^3 for N=224, a loss at N=256
// where only three 64 KB stages would fit).
// Stage shape and MMA rounds, measured on the 4096^3 step (CUDA events, µs):
// the single thread that issues the MMAs paces the tensor pipe, so how many
// MMAs it issues per barrier round matters as much as the ring depth.
//   N tile 224: two 128-byte boxes per stage (three 60 KB stages), one stage per
//     round: fprop 48.0-48.3; one box per stage (seven 30 KB stages) taken one /
//     two / three per round: 52.4 / 48.95-49.5 / 49.4-49.9.
//   N tile 256: one box per stage (seven 32 KB stages) taken two per round:
//     dgrad+wgrad 85.3-86.5; one / three / four per round: 88.1-90.1 /
//     87.2-87.5 / 89.3; two boxes per stage (three 64 KB stages): 88.5.
// (Those figures predate the staged output path below, whose 16 KB leave the
// 256-wide tile six stages.)
//
// Output path, measured back to back on one GPU (fprop / dgrad+wgrad / whole
// step, µs; the same code differs by about 2 µs between GPUs, so only figures
// taken on one GPU compare):
//   per-thread 16-byte stores, one row per thread:  49.0 / 87.3 / 172.3
//   staged in shared memory, coalesced stores:       47.6 / 85.3 / 168.4
//   staged, one 32 x 32 TMA box store per chunk:     47.6 / 85.5 / 166.3
//   no global stores at all (timing probe only):     43.3 / 79.0 / 157.4
// Writing the staging boxes costs nothing measurable (43.9 / 78.7 without
// the copies); the global writes themselves cost 2.5-4 µs per launch whatever
// their shape, also when every tile writes one L2-resident region.  64-column
// boxes (128-byte swizzle, 32 KB of staging) gain 0.5 µs per launch but no
// longer leave room for the step's backward quantiser to run beside fprop,
// which costs the step 5 µs.
template <int BN, int KS = (BN < 256 ? 2 : 1), int BATCH = (BN < 256 ? 1 : 2)>
struct PairCfg {
    static_assert(BN % 32 == 0 && BN >= 128 && BN <= 256, "N tile");
    static constexpr int KSUB = KS;
    static constexpr int MMA_BATCH = BATCH;  // stages the MMA issuer takes per round
    static constexpr int BK = 128 * KSUB;
    static constexpr int BNH = BN / 2;  // B rows held by each CTA
    static constexpr int A_SUB = 128 * 128, B_SUB = BNH * 128;  // one 128-byte box
    static constexpr int A_STAGE = A_SUB * KSUB, B_STAGE = B_SUB * KSUB;
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;  // per CTA
    // output staging: two 32 x 32 bf16 boxes (2 KB each) per epilogue warp
    static constexpr int STAGING = 4 * 2 * 2048;
    static constexpr int STAGES_FIT = (int)((SMEM_LIMIT - 1024 - 1024 - STAGING) / STAGE_BYTES);
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr uint32_t IDESC = idesc_f8_f32(256, BN);
    // alignment slack, the stage ring, barriers (in a 1 KB slot), staging
    static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 1024 + STAGING;
};

struct PairProblem {
    int M, N, K;
    const float *sa, *sb;
    const uint16_t *bias;
    int m_tiles, n_tiles, tiles;
};

struct PairArgs {
    PairProblem pr[2];  // pr[1].tiles == 0 for a single problem
    uint64_t wait_limit_ns;
    unsigned int *status;
};

// Tile index -> problem, pair-row and column tile.  The fields are picked
// with selects so the argument block is read in place.
struct TileRef {
    int pi, tm, tn;
};
__device__ __forceinline__ TileRef locate(const PairArgs &p, int tile) {
    TileRef r;
    r.pi = tile >= p.pr[0].tiles ? 1 : 0;
    const int t = r.pi ? tile - p.pr[0].tiles : tile;
    const int mt = r.pi ? p.pr[1].m_tiles : p.pr[0].m_tiles;
    const int nt = r.pi ? p.pr[1].n_tiles : p.pr[0].n_tiles;
    grouped_tile(t, mt, nt, GROUP_M, r.tm, r.tn);
    return r;
}

template <int BN, int KS, int BATCH>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_f8_pair_kernel(const __grid_constant__ CUtensorMap tma_a0,
                        const __grid_constant__ CUtensorMap tma_b0,
                        const __grid_constant__ CUtensorMap tma_a1,
                        const __grid_constant__ CUtensorMap tma_b1,
                        const __grid_constant__ CUtensorMap tma_d0,
                        const __grid_constant__ CUtensorMap tma_d1, const PairArgs p) {
    using C = PairCfg<BN, KS, BATCH>;
    constexpr int STAGES = C::STAGES, A_STAGE = C::A_STAGE, B_STAGE = C::B_STAGE;
    constexpr int BNH = C::BNH, BK = C::BK, KSUB = C::KSUB;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * C::STAGE_BYTES);
    uint64_t *full = bars;                // [STAGES] (leader's counts both CTAs' bytes)
    uint64_t *empty = bars + STAGES;      // [STAGES]
    uint64_t *tfull = bars + 2 * STAGES;  // [2]
    uint64_t *tempty = tfull + 2;         // [2] (leader's counts 8 epilogue warps)
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    uint8_t *staging = smem + STAGES * C::STAGE_BYTES + 1024;  // 1024-byte aligned

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int num_tiles = p.pr[0].tiles + p.pr[1].tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tma_a0);
        tma_prefetch_desc(&tma_b0);
        tma_prefetch_desc(&tma_d0);
        if (p.pr[1].tiles > 0) {
            tma_prefetch_desc(&tma_a1);
            tma_prefetch_desc(&tma_b1);
            tma_prefetch_desc(&tma_d1);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised before any remote use
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
            for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
                const TileRef r = locate(p, tile);
                const CUtensorMap *ta = r.pi ? &tma_a1 : &tma_a0;
                const CUtensorMap *tb = r.pi ? &tma_b1 : &tma_b0;
                const int nk = ((r.pi ? p.pr[1].K : p.pr[0].K) + BK - 1) / BK;
                const int arow = r.tm * 256 + (int)rank * 128;
                const int brow = r.tn * BN + (int)rank * BNH;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.wait_limit_ns,
                                           kStatusTimeoutTma, p.status)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                    const uint32_t leader_full = mapa_shared(smem_u32(&full[stage]), 0);
#pragma unroll
                    for (int ks = 0; ks < KSUB; ++ks) {
                        tma_load_2d_pair(sA + stage * A_STAGE + ks * C::A_SUB, ta, leader_full,
                                         kb * BK + 128 * ks, arow);
                        tma_load_2d_pair(sB + stage * B_STAGE + ks * C::B_SUB, tb, leader_full,
                                         kb * BK + 128 * ks, brow);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && rank == 0) {
                // the leader's `full` barriers count both CTAs' copies: wait
                // (bounded) for the last STAGES issues to land before teardown
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
            bool ok = true;
            int it = 0;
            // descriptors of stage 0's A and B boxes; a descriptor's address
            // field holds (address >> 4) in 14 bits and shared addresses stay
            // below 2^18, so adding an offset >> 4 never carries out of it
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA));
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB));
            for (int tile = pair; tile < num_tiles && ok; tile += npairs, ++it) {
                const int nk = ((tile >= p.pr[0].tiles ? p.pr[1].K : p.pr[0].K) + BK - 1) / BK;
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, p.wait_limit_ns,
                                       kStatusTimeoutMma, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                // One round: wait for NB stages, then issue their MMAs and a
                // commit per stage.  This single thread's instruction path
                // paces the tensor pipe, so the rounds are unrolled and the
                // shared-memory descriptors advance by adding the byte
                // offset >> 4 to the address field of a precomputed base.
                int kb = 0;
                auto round = [&](auto nb_const) -> bool {
                    constexpr int NB = decltype(nb_const)::value;
                    int st = stage;
                    uint32_t ph = phase;
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        if (!mbar_wait_bounded(&full[st], ph, abort_flag, p.wait_limit_ns,
                                               kStatusTimeoutMma, p.status))
                            return false;
                        if (++st == STAGES) {
                            st = 0;
                            ph ^= 1u;
                        }
                    }
                    tc_fence_after();
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const uint64_t ad = a_desc0 + (uint64_t)((stage * A_STAGE) >> 4);
                        const uint64_t bd = b_desc0 + (uint64_t)((stage * B_STAGE) >> 4);
#pragma unroll
                        for (int ks = 0; ks < KSUB; ++ks)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_f8_pair(d_tmem, ad + (uint64_t)((ks * C::A_SUB + 32 * k) >> 4),
                                            bd + (uint64_t)((ks * C::B_SUB + 32 * k) >> 4),
                                            C::IDESC, ((kb + b) | ks | k) != 0);
                        mma_commit_pair(&empty[stage], 0x3);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    kb += NB;
                    return true;
                };
                while (ok && kb + C::MMA_BATCH <= nk)
                    ok = round(std::integral_constant<int, C::MMA_BATCH>{});
                while (ok && kb < nk) ok = round(std::integral_constant<int, 1>{});
                if (ok) mma_commit_pair(&tfull[acc], 0x3);
            }
            mma_commit_pair(drain, 0x1);
            volatile int no_abort = 0;
            mbar_wait_bounded(drain, 0, &no_abort, p.wait_limit_ns, kStatusTimeoutMma, p.status);
        }
    } else {
        // ---------------------------------------------- epilogue (both CTAs)
        // Warp q owns accumulator lanes 32q..32q+31 (one output row per
        // thread).  Each 32-column chunk is scaled, rounded to bf16 and
        // written into one of the warp's two 2 KB staging boxes in the 64-byte
        // swizzled layout (conflict-free), and lane 0 stores the box with one
        // TMA copy.  Per-thread row stores (32 rows per warp instruction) cost
        // the MMA pipe 7-10 µs per launch at 4096^3 in measurement; the
        // staged box needs one issue per chunk.
        const int quarter = warp & 3;
        uint8_t *stg = staging + quarter * 4096;
        uint32_t chunk = 0;
        int it = 0;
        for (int tile = pair; tile < num_tiles; tile += npairs, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            const bool ok = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, p.wait_limit_ns,
                                              kStatusTimeoutEpilogue, p.status);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const TileRef tr = locate(p, tile);
            const int tm = tr.tm, tn = tr.tn;
            const int pN = tr.pi ? p.pr[1].N : p.pr[0].N;
            const uint16_t *bias = tr.pi ? p.pr[1].bias : p.pr[0].bias;
            const CUtensorMap *td = tr.pi ? &tma_d1 : &tma_d0;
            const float s = tr.pi ? __fmul_rn(*p.pr[1].sa, *p.pr[1].sb)
                                  : __fmul_rn(*p.pr[0].sa, *p.pr[0].sb);
            const int row0 = tm * 256 + (int)rank * 128 + quarter * 32;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                       (uint32_t)(acc * BN + c * 32),
                                   r);
                tmem_ld_wait();
                const int col = tn * BN + c * 32;
                if (col >= pN) continue;  // warp-uniform; rows past M are clipped by the copy
                uint32_t packed[16];
                if (bias != nullptr) {
                    // N is a multiple of 16: a last chunk may hold only 16
                    // columns, whose upper half is neither read nor stored
                    const int jn = col + 16 < pN ? 16 : 8;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float b0 =
                            j < jn ? __uint_as_float((uint32_t)bias[col + 2 * j] << 16) : 0.f;
                        const float b1 =
                            j < jn ? __uint_as_float((uint32_t)bias[col + 2 * j + 1] << 16) : 0.f;
                        packed[j] =
                            pack_bf16x2(__fadd_rn(__fmul_rn(__uint_as_float(r[2 * j]), s), b0),
                                        __fadd_rn(__fmul_rn(__uint_as_float(r[2 * j + 1]), s), b1));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        packed[j] = pack_bf16x2(__fmul_rn(__uint_as_float(r[2 * j]), s),
                                                __fmul_rn(__uint_as_float(r[2 * j + 1]), s));
                }
                uint8_t *box = stg + (chunk & 1u) * 2048;
                ++chunk;
                if (lane == 0) bulk_wait_group_read<1>();  // this box's previous copy has read it
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4 *>(box + lane * 64 + 16 * (q ^ ((lane >> 1) & 3))) =
                        make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                   packed[4 * q + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(td, smem_u32(box), col, row0);
                    bulk_commit_group();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
        }
        if (lane == 0) bulk_wait_group_all();  // outputs written before the CTA retires
    }

    __syncwarp();  // lanes that skipped a role wait here for their warp's lane 0
    tc_fence_before();
    cluster_sync_all();  // the peer's smem/TMEM stay alive until the leader's MMAs drained
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int BN, int KS = (BN < 256 ? 2 : 1), int BATCH = (BN < 256 ? 1 : 2)>
cudaError_t launch_pair_bn(const PairGemm *g, int n, cudaStream_t s, const char **why) {
    using C = PairCfg<BN, KS, BATCH>;
    static std::atomic<bool> attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_f8_pair_kernel<BN, KS, BATCH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    CUtensorMap ta[2], tb[2], td[2];
    PairArgs args;
    int64_t tiles = 0;
    for (int i = 0; i < 2; ++i) {
        const PairGemm &q = g[i < n ? i : 0];  // an absent second problem: copies, no tiles
        if (!make_tmap_k128(&ta[i], q.A, q.M, q.K, 128) ||
            !make_tmap_k128(&tb[i], q.B, q.N, q.K, C::BNH) ||
            !make_tmap_bf16_store32(&td[i], q.D, q.M, q.N, q.N)) {
            *why = "cuTensorMapEncodeTiled failed";
            return cudaErrorInvalidValue;
        }
        PairProblem &pr = args.pr[i];
        pr.M = (int)q.M;
        pr.N = (int)q.N;
        pr.K = (int)q.K;
        pr.sa = q.sa;
        pr.sb = q.sb;
        pr.bias = q.bias;
        pr.m_tiles = (int)((q.M + 255) / 256);
        pr.n_tiles = (int)((q.N + BN - 1) / BN);
        pr.tiles = i < n ? pr.m_tiles * pr.n_tiles : 0;
        tiles += pr.tiles;
    }
    args.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    args.status = device_status_word();
    const int64_t pairs = num_sms() / 2;
    const int grid = 2 * (int)(tiles < pairs ? tiles : pairs);
    return launch_pdl(gemm_f8_pair_kernel<BN, KS, BATCH>, grid, NUM_THREADS, C::SMEM_BYTES, s, ta[0], tb[0],
                      ta[1], tb[1], td[0], td[1], args);
}

}  // namespace

// Same cost model as the one-CTA chooser, per SM of a pair: waves of 256 x BN
// tiles (of all the launch's problems) over the pairs times the bytes each SM
// streams per block, 128 + BN/2.
int choose_pair_bn(const PairGemm *g, int n, int pairs) {
    static const int cand[] = {256, 224, 192, 160, 128};
    int best = 256;
    double best_cost = 1e30;
    for (int bn : cand) {
        int64_t tiles = 0;
        for (int i = 0; i < n; ++i) tiles += ((g[i].M + 255) / 256) * ((g[i].N + bn - 1) / bn);
        const int64_t waves = (tiles + pairs - 1) / pairs;
        const double cost = (double)waves * (128 + bn / 2);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

cudaError_t launch_gemm_pair(const PairGemm *g, int n, int bn, cudaStream_t s, const char **why) {
    if (n < 1 || n > 2) {
        *why = "a pair launch takes one or two problems";
        return cudaErrorInvalidValue;
    }
    const int b = bn ? bn : choose_pair_bn(g, n, num_sms() / 2);
    switch (b) {
    case 224: return launch_pair_bn<224>(g, n, s, why);
    case 192: return launch_pair_bn<192>(g, n, s, why);
    case 160: return launch_pair_bn<160>(g, n, s, why);
    case 128: return launch_pair_bn<128>(g, n, s, why);
    default: return launch_pair_bn<256>(g, n, s, why);
    }
}

}  // namespace fp8
