// Block-scaled FP8 GEMM (the TE "recipe=block" layout: 1x128 tiles along the
// contraction dim for activations and gradients, 128x128 tiles for weights).
//
//   D[i,j] = bf16( sum_kb sA(i,kb) * sB(j,kb) * sum_{k in block kb} A[i,k] B[j,k] )
//
// One persistent CTA per SM owns 128 x 128 output tiles; each 128-deep
// contraction block is one stage of a TMA ring.  The MMA warp writes that
// block's partial product (fresh accumulation) into one of four 128-column
// TMEM slots, so it can run three blocks ahead of the promotion; eight
// epilogue warps (two per TMEM lane quarter, 64 columns each) read a partial
// back in one round trip, hand the slot back and fold it into fp32 register
// accumulators with the two block scales using packed fp32x2 FMAs.  B's scale
// is one value per 128-row tile (weights) or one per row (wgrad's Xᵀ operand:
// each warp stages its 64 scales of the next block into shared memory with
// cp.async, from a layout contiguous over rows).  Every handshake is local to
// the SM: a CTA-pair version of this kernel measured at half the speed, the
// per-block slot hand-back across two SMs costing more than the slack.  Every
// wait is bounded, as in the other GEMM kernels.
#include <cuda.h>

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
constexpr int COLS = 64;  // accumulator columns per epilogue thread
constexpr uint32_t TMEM_COLS = SLOTS * BN;  // 512
constexpr int GROUP_M = 8;
constexpr uint32_t IDESC = idesc_f8_f32(BM, BN);
constexpr int SBUF_FLOATS = EPI_WARPS * 2 * COLS;  // per-warp double-buffered B-row scales
constexpr size_t SMEM_BYTES =
    1024 + (size_t)STAGES * STAGE_BYTES + SBUF_FLOATS * sizeof(float) + 256;

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

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
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
    float *sbuf = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbuf + SBUF_FLOATS);
    uint64_t *full = bars;                // [STAGES] TMA -> MMA
    uint64_t *empty = bars + STAGES;      // [STAGES] MMA -> TMA
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
    pdl_wait_prior();  // set-up done; the previous kernel's results are needed from here
    pdl_allow_next();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                int tm, tn;
                grouped_tile(tile, m_tiles, n_tiles, GROUP_M, tm, tn);
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
            // ------------------------------------------------ MMA issuer
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
        const int group = (warp - 2) >> 2;  // columns group*64 .. +63 of the tile
        float *wbuf = sbuf + (warp - 2) * 2 * COLS;  // this warp's [2][COLS] B-row scales
        constexpr int PER_LANE = COLS / 32;          // B-row scales each lane stages
        const BlockScales &sc = p.sc;
        bool ok = true;
        uint32_t g = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int tm, tn;
            grouped_tile(tile, m_tiles, n_tiles, GROUP_M, tm, tn);
            const int row = tm * BM + quarter * 32 + lane;
            const int j0 = tn * BN + group * COLS;  // first output column of this thread
            const float *sa_row = sc.sa + (int64_t)min(row, p.M - 1) * sc.sa_row;
            // per-tile B: one scale per block for this thread's columns (all in
            // one 128-row weight tile); per-row B: lane l stages rows
            // j0 + PER_LANE*l .. of the block's scales
            const float *sb_ptr =
                kPerRowB ? sc.sb + (int64_t)min(j0 + PER_LANE * lane, p.N - PER_LANE) * sc.sb_row
                         : sc.sb + (int64_t)(min(j0, p.N - 1) / sc.b_rows) * sc.sb_row;
            uint64_t acc[COLS / 2];  // fp32 accumulators in pairs
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) acc[j] = 0ull;
            float sa_next = sa_row[0];
            float sb_next = kPerRowB ? 0.f : sb_ptr[0];
            auto stage_scales = [&](int kbn) {
                const float *src = sb_ptr + (int64_t)kbn * sc.sb_k;
                float *dst = wbuf + (kbn & 1) * COLS + PER_LANE * lane;
                asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n\tcp.async.commit_group;" ::
                                 "r"(smem_u32(dst)),
                             "l"(src), "n"(PER_LANE * 4)
                             : "memory");
            };
            if (kPerRowB) stage_scales(0);
            for (int kb = 0; kb < nk; ++kb, ++g) {
                const uint32_t slot = g % SLOTS, sphase = (g / SLOTS) & 1u;
                const float sa_cur = sa_next;
                const float sb_cur = sb_next;
                const float *buf = wbuf + (kb & 1) * COLS;
                if (kPerRowB) {
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                    __syncwarp();  // every lane's part of this block's scales has landed
                    if (kb + 1 < nk) stage_scales(kb + 1);
                }
                if (kb + 1 < nk) {  // prefetch the next block's scalar scales
                    sa_next = sa_row[(int64_t)(kb + 1) * sc.sa_k];
                    if (!kPerRowB) sb_next = sb_ptr[(int64_t)(kb + 1) * sc.sb_k];
                }
                if (ok)
                    ok = mbar_wait_bounded(&sfull[slot], sphase, abort_flag, p.wait_limit_ns,
                                           kStatusTimeoutEpilogue, p.status);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) continue;  // outputs invalid; keep the loop shape
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + slot * BN +
                                       (uint32_t)(group * COLS);
                // all of this warp's columns in one round trip, then the slot
                // goes back before the math
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(taddr, r0);
                tmem_ld_32x32b_x32(taddr + 32, r1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sempty[slot]);
                const uint64_t fsa = pack2(sa_cur, sa_cur);
                const float f1 = sa_cur * sb_cur;
                const uint64_t fts = pack2(f1, f1);
#pragma unroll
                for (int a = 0; a < COLS / 2; ++a) {
                    const uint32_t lo = a < 16 ? r0[2 * a] : r1[2 * a - 32];
                    const uint32_t hi = a < 16 ? r0[2 * a + 1] : r1[2 * a - 31];
                    const uint64_t pv = pack2(__uint_as_float(lo), __uint_as_float(hi));
                    if (kPerRowB) {
                        const float2 sb2 = *reinterpret_cast<const float2 *>(buf + 2 * a);
                        const uint64_t f = mul2(pack2(sb2.x, sb2.y), fsa);
                        acc[a] = fma2(pv, f, acc[a]);
                    } else {
                        acc[a] = fma2(pv, fts, acc[a]);
                    }
                }
            }
            if (ok && row < p.M && j0 < p.N) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.d + (int64_t)row * p.ldd + j0);
#pragma unroll
                for (int c = 0; c < COLS / 8; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) unpack2(acc[4 * c + e], v[2 * e], v[2 * e + 1]);
                    dst[c] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                        pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                }
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
    return launch_pdl(gemm_f8_block_kernel<kPerRowB>, grid, NUM_THREADS, SMEM_BYTES, s, ta, tb,
                      args);
}

}  // namespace

cudaError_t launch_gemm_block(const uint8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K,
                              const BlockScales &sc, uint16_t *D, cudaStream_t s,
                              const char **why) {
    CUtensorMap ta, tb;
    if (!make_tmap_k128(&ta, A, M, K, BM) || !make_tmap_k128(&tb, B, N, K, BN)) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    BlockArgs args;
    args.M = (int)M;
    args.N = (int)N;
    args.K = (int)K;
    args.sc = sc;
    args.d = D;
    args.ldd = N;
    args.wait_limit_ns = g_wait_limit_ns;
    args.status = device_status_word();
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = (int)(tiles < num_sms() ? tiles : num_sms());
    if (sc.b_rows == 1) return launch_block<true>(ta, tb, args, grid, s);
    if (sc.b_rows == 128) return launch_block<false>(ta, tb, args, grid, s);
    *why = "B scales must be per row or per 128-row tile";
    return cudaErrorInvalidValue;
}

}  // namespace fp8
