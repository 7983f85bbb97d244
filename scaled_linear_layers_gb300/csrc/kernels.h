// Internal launchers shared by the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace fp8 {

int num_sms();  // SM count of the current device (cached per device)

// Host-side fault injection for the tests (fp8_inject_launch_failures): the
// calling thread's next n launches through launch_pdl return
// cudaErrorLaunchFailure without launching anything.
extern thread_local int tl_fail_launches;

// Launches `kernel` on `s` with programmatic stream serialisation allowed: it
// may begin while the previous kernel on the stream drains, and must wait
// (pdl_wait_prior) before reading or writing global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
    if (tl_fail_launches > 0) {
        --tl_fail_launches;
        return cudaErrorLaunchFailure;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device address of the status word of the current device (nullptr on error).
unsigned int *device_status_word();
// Reads the status word and clears it if it was set (synchronous copies).
cudaError_t read_and_clear_device_status(unsigned int *out);

cudaError_t launch_amax(const uint16_t *x, int64_t n, float *amax_out, cudaStream_t s);
cudaError_t launch_quantize_tensor(const uint16_t *x, int64_t n, bool dynamic, float *scale,
                                   float *scale_inv, uint8_t *q, float *amax_out, cudaStream_t s);
cudaError_t launch_quantize_rowtiles(const uint16_t *x, int64_t rows, int64_t cols, float *scale,
                                     float *scale_inv, uint8_t *q, float *amax_out,
                                     cudaStream_t s);
// mode: 0 tensor/delayed, 1 tensor/dynamic, 2 128x128 tiles, 3 row+column tiles
// colsum (tensor modes, nullable): per-tile column sums of x, [ceil(rows/128),
// cols] fp32, for launch_colsum_reduce.
cudaError_t launch_quantize_transpose(const uint16_t *x, int64_t rows, int64_t cols, int mode,
                                      float *scale, float *scale_inv, uint8_t *q, uint8_t *qt,
                                      float *scale_t, float *scale_inv_t, float *amax_out,
                                      cudaStream_t s, float *colsum = nullptr);
// dbias [cols] bf16 = the per-tile column sums added in tile order.
cudaError_t launch_colsum_reduce(const float *partials, int64_t rows, int64_t cols,
                                 uint16_t *dbias, cudaStream_t s);
// Two delayed-scaling quantisations in one launch (q and/or qt per tensor,
// rows and cols multiples of 16).  amax_out, when given, must already be
// zero: this launcher does not clear it.  If snap_dst is given, the launch
// also copies *snap_src to it (before any state update that follows).
struct DelayedQuantJob {
    const uint16_t *x;
    int64_t rows, cols;
    const float *scale_inv;
    uint8_t *q, *qt;
    float *amax_out;
    float *colsum = nullptr;  // per-tile column sums (bias gradient), nullable
};
// qt [cols, rows] = q [rows, cols]ᵀ for existing e4m3 bytes
struct ByteTransposeJob {
    const uint8_t *q;
    int64_t rows, cols;
    uint8_t *qt;
};
// The two delayed-mode casts in one launch, optionally with a byte transpose
// in the same launch (tiles after the casts').
cudaError_t launch_quantize_delayed_pair(const DelayedQuantJob &a, const DelayedQuantJob &b,
                                         cudaStream_t s, const float *snap_src = nullptr,
                                         float *snap_dst = nullptr,
                                         const ByteTransposeJob *bt = nullptr);
// Forward state update in one launch: history[idx] = *amax_w, then the lag
// update of the x scale from *amax_x.
cudaError_t launch_meta_fwd(float *dev, int idx, const float *amax_x, const float *amax_w,
                            cudaStream_t s);
// Current scaling in one cooperative launch (see quantize_fused.cu);
// workspace: kFusedWorkspaceBytes, zero before its first use.
cudaError_t launch_quantize_fused_dynamic(const uint16_t *x, int64_t rows, int64_t cols,
                                          float *scale, float *scale_inv, uint8_t *q, uint8_t *qt,
                                          float *amax_out, unsigned int *workspace, cudaStream_t s);
// The fused kernel indexes 128x128 tiles with 32-bit ints: false when a
// [rows, cols] tensor has more tiles than that.
bool fused_tiles_fit(int64_t rows, int64_t cols);
// The same with a static scratch array instead of a workspace (no allocation).
cudaError_t launch_quantize_fused_dynamic_noalloc(const uint16_t *x, int64_t rows, int64_t cols,
                                                  float *scale, float *scale_inv, uint8_t *q,
                                                  uint8_t *qt, float *amax_out, cudaStream_t s,
                                                  const char **why);
// Current-scaling fprop of one output tile in one launch (linear_small.cu):
// M <= 128, N <= 256, K <= 512 (linear_small_fits).
bool linear_small_fits(int64_t M, int64_t N, int64_t K);
cudaError_t launch_linear_small_dynamic(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N,
                                        int64_t K, const uint16_t *bias, float *scales,
                                        float *amax, uint8_t *xq, uint8_t *wq, uint16_t *y,
                                        cudaStream_t s);
// amax[i], scale[i], scale_inv[i] of the bf16 tensors w[i] (numel[i]
// elements, 16-byte aligned): current scaling, one amax launch per 64
// tensors and one scale launch.
cudaError_t launch_multi_amax_scales(const uint16_t *const *w, const int64_t *numel, int n,
                                     float *amax, float *scale, float *scale_inv, cudaStream_t s);
// out [B, Tp, H] = x [B, T, H] padded per sequence with zero rows (H % 8 == 0).
cudaError_t launch_pad_bshd(const uint16_t *x, int64_t B, int64_t T, int64_t H, int64_t Tp,
                            uint16_t *out, cudaStream_t s);
cudaError_t launch_pad_rows(const uint16_t *x, int64_t rows, int64_t cols, int64_t padded,
                            uint16_t *out, cudaStream_t s);

// D [M,N] (row-major, leading dim N) = s_a*s_b * A[M,K] · B[N,K]ᵀ (+ bias[N]),
// A and B e4m3 with K contiguous.  Tensorwise scales: sa, sb point to one
// float each.
cudaError_t launch_gemm_tensor(const uint8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K,
                               const float *sa, const float *sb, const uint16_t *bias,
                               uint16_t *D, cudaStream_t s, const char **why);

// One tensorwise GEMM as launch_gemm_tensor takes it.
struct PairGemm {
    const uint8_t *A, *B;
    int64_t M, N, K;
    const float *sa, *sb;
    const uint16_t *bias;
    uint16_t *D;
};
// The 2-SM (CTA pair) kernel behind launch_gemm_tensor for large problems:
// n = 1 or 2 independent problems in one launch; bn = 0 lets it choose the N
// tile (one for all problems).
cudaError_t launch_gemm_pair(const PairGemm *g, int n, int bn, cudaStream_t s, const char **why);
// Two tensorwise GEMMs: one pair launch when their tiles fill at least a wave
// of pairs and their contraction lengths are within 2x, else one launch each.
cudaError_t launch_gemm_tensor2(const PairGemm &a, const PairGemm &b, cudaStream_t s,
                                const char **why);

// Block-scaled variant: the contraction is split into 128-blocks; A's scale
// of (row i, block kb) is sa[i * sa_row + kb * sa_k]; B's scale of (row j,
// block kb) is sb[(j / b_rows) * sb_row + kb * sb_k], b_rows = 1 (per-row
// scales) or 128 (128x128 weight tiles).
struct BlockScales {
    const float *sa;
    int64_t sa_row, sa_k;
    const float *sb;
    int64_t sb_row, sb_k;
    int b_rows;
};
cudaError_t launch_gemm_block(const uint8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K,
                              const BlockScales &sc, uint16_t *D, cudaStream_t s, const char **why);

cudaError_t launch_meta_init(float *dev, int interval, cudaStream_t s);
cudaError_t launch_meta_copy(float *dst, const float *src, cudaStream_t s);
cudaError_t launch_meta_lag(float *scale, float *scale_inv, const float *amax, cudaStream_t s);
cudaError_t launch_meta_refresh(float *dev, int interval, cudaStream_t s);
// p[0..n) = 0 as a kernel launched with programmatic dependent launch, so
// that it keeps the launch chain of a stream unbroken (a memset node would
// not).
cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t s);
cudaError_t launch_selftest_wait(uint32_t timeout_us, cudaStream_t s);

}  // namespace fp8
