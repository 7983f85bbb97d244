/*
 * fp8linear.h — C ABI of the GB300 (sm_103a) FP8 scaled linear layer.
 *
 * The layer computes, for X [M,K] (tokens x in-features), W [N,K]
 * (out-features x in-features) and the upstream gradient G [M,N], all bf16
 * row-major:
 *     Y  = X  · Wᵀ   (fprop)   [M,N]
 *     dX = G  · W    (dgrad)   [M,K]
 *     dW = Gᵀ · X    (wgrad)   [N,K]
 * with every operand quantised to E4M3 and every GEMM computed as
 * D = s_A · s_B · (A · B) with fp32 accumulation and a bf16 result.  Sources:
 * AstrAI "astrai/extension/fp8_state.py" (the comment above FP8TensorMeta:
 * the GEMM scales its product by both operands' scales, per-tensor scales are
 * amax/448, quantisation multiplies by 1/scale; fp8_linear_forward /
 * fp8_linear_backward), the
 * SpecForge "Add training.fp8_linear" page (dynamic tensorwise scaling; token
 * counts must be a multiple of 16) and the NeMo "Add FP8 support for
 * SALMAutomodel" page (TE recipe=block, padding appended at the end).
 *
 * Conventions for every call:
 *   - All tensor pointers are caller-owned DEVICE memory, 16-byte aligned.
 *     bf16 tensors are passed as uint16_t bit patterns, e4m3 as uint8_t.
 *   - Scales are fp32 DEVICE pointers: `scale` = amax/448 multiplies the GEMM
 *     result (dequantisation), `scale_inv` = 448/amax multiplies the input
 *     before the cast (quantisation).  The host never reads them, so nothing
 *     synchronises.
 *   - Work is enqueued on the caller's stream `s` (NULL = legacy default
 *     stream).  No call synchronises except fp8_check_device_status.  No call
 *     allocates device memory.  Calls are re-entrant; the only global state is
 *     a thread-local error string and one device status word.
 *   - Every call returns an fp8_status; FP8_OK means the work was enqueued.
 *     Host-side validation happens before anything is enqueued, so a call that
 *     fails validation has no effect.  fp8_last_error() describes the last
 *     failure on the calling thread.
 */
#ifndef FP8LINEAR_H
#define FP8LINEAR_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8_OK = 0,
    FP8_ERR_NULL = 1,        /* a required pointer is NULL                          */
    FP8_ERR_SHAPE = 2,       /* a size is negative or the shapes disagree           */
    FP8_ERR_ALIGNMENT = 3,   /* a dim is not a multiple of 16 (128 for block tiles),
                                or a pointer is not 16-byte aligned.  Callers keep
                                such a linear in bf16.                             */
    FP8_ERR_UNSUPPORTED = 4, /* the current device is not sm_103 (GB300)            */
    FP8_ERR_CUDA = 5,        /* a CUDA runtime call failed                          */
    FP8_ERR_TIMEOUT = 6      /* a kernel's bounded wait ran out (see
                                fp8_check_device_status); its outputs are invalid  */
} fp8_status;

typedef enum {
    FP8_RECIPE_DELAYED = 0,  /* TE-style delayed scaling: scale_inv is an INPUT
                                (from the previous call or the amax history); the
                                quantiser emits this call's amax for the next one  */
    FP8_RECIPE_DYNAMIC = 1,  /* current tensorwise scaling: amax of this tensor,
                                then scale/scale_inv are OUTPUTS                    */
    FP8_RECIPE_BLOCK = 2,    /* 1x128 tiles along the contraction dim (activations,
                                gradients); fp32 scale per tile, OUTPUTS            */
    FP8_RECIPE_BLOCK_2D = 3  /* 128x128 tiles (weights); fp32 scale per tile,
                                OUTPUTS; one scale grid serves W and Wᵀ            */
} fp8_recipe;

/* ------------------------------------------------------------------------ */
/* Quantisation                                                              */
/* ------------------------------------------------------------------------ */

/* amax_out = max |x| over n bf16 elements, as fp32 (a NaN input makes it NaN).
 * amax_out is overwritten (the call zeroes it first).  Any n >= 0.
 * Source: AstrAI fp8_state.py module docstring (amax of each quantised tensor);
 * SpecForge page (dynamic tensorwise scaling takes the current amax). */
fp8_status fp8_amax(const uint16_t *x, int64_t n, float *amax_out, cudaStream_t s);

/* q = e4m3(fl32(x * scale_inv)), round-to-nearest-even, saturating to ±448,
 * for x [rows, cols] row-major; q [rows, cols] row-major.
 *   DELAYED: scale_inv [1] is read; scale is unused (may be NULL); amax_out
 *            (nullable) receives amax(x) — the quantiser's own amax, which the
 *            caller turns into the next call's scale (fp8_meta_record).
 *   DYNAMIC: amax_out [1] is REQUIRED and receives amax(x); scale [1] and
 *            scale_inv [1] receive max(amax,1e-12)/448 and 448/max(amax,1e-12).
 *   BLOCK:   cols % 128 == 0; scale and scale_inv [rows, cols/128] receive the
 *            per-1x128-tile scales; amax_out (nullable) receives amax(x).
 *   BLOCK_2D: rows % 128 == 0 and cols % 128 == 0; scale and scale_inv
 *            [rows/128, cols/128]; amax_out nullable.
 * Any rows, cols >= 0 for DELAYED/DYNAMIC (n = rows*cols need not be a
 * multiple of anything).  Source: AstrAI fp8_state.py, fp8_linear_forward
 * (its quantise kernel also yields the tensor's current amax),
 * _update_delayed_scale. */
fp8_status fp8_quantize(const uint16_t *x, int64_t rows, int64_t cols, fp8_recipe r,
                        float *scale, float *scale_inv, uint8_t *q, float *amax_out,
                        cudaStream_t s);

/* One read of x [rows, cols] producing q [rows, cols] (nullable) and its
 * transpose qt [cols, rows], both e4m3 with the same rounding as fp8_quantize.
 * qt gives wgrad and dgrad their operands with the contraction dim contiguous.
 * rows % 16 == 0 and cols % 16 == 0 (BLOCK/BLOCK_2D: % 128).
 *   DELAYED / DYNAMIC: scale, scale_inv, amax_out as for fp8_quantize;
 *            scale_t / scale_inv_t unused (may be NULL).
 *   BLOCK:   q uses 1x128 row tiles (scale/scale_inv [rows, cols/128]); qt uses
 *            128x1 column tiles, i.e. 1x128 tiles of its own rows; their scales
 *            scale_t/scale_inv_t are [rows/128, cols]: entry [b, c] is the
 *            scale of column c over rows 128b..128b+127 (qt row c, contraction
 *            block b), contiguous over c.  q and its scales may be NULL
 *            together when only qt is wanted (wgrad operands).
 *   BLOCK_2D: 128x128 tiles; scale/scale_inv [rows/128, cols/128] serve both q
 *            and qt; scale_t/scale_inv_t unused.
 * Source: AstrAI fp8_state.py fp8_linear_backward (x and w quantised again for
 * the backward GEMMs); NeMo SALMAutomodel page (TE recipe=block). */
fp8_status fp8_quantize_transpose(const uint16_t *x, int64_t rows, int64_t cols, fp8_recipe r,
                                  float *scale, float *scale_inv, uint8_t *q, uint8_t *qt,
                                  float *scale_t, float *scale_inv_t, float *amax_out,
                                  cudaStream_t s);

/* Bias gradient fused into the quantisation of the upstream gradient g
 * [rows, cols] (the linear backward's third output, which the AstrAI page's
 * fp8_linear_backward asks for through its output mask): the results of
 * fp8_quantize_transpose(g, ..., r, scale, scale_inv, q, qt, NULL, NULL,
 * amax_out), plus dbias [cols] bf16 = the column sums of g, summed in fp32
 * (per 128-row tile in a fixed order, then over the tiles in order) and
 * rounded once to bf16.  The cast pass reads g once for both.  `workspace`:
 * fp8_dbias_workspace_bytes(rows, cols) bytes of device memory (per-tile
 * partial sums), overwritten.  r: DELAYED or DYNAMIC (others
 * FP8_ERR_UNSUPPORTED).  rows = 0 gives dbias = 0. */
size_t fp8_dbias_workspace_bytes(int64_t rows, int64_t cols);
fp8_status fp8_quantize_transpose_dbias(const uint16_t *g, int64_t rows, int64_t cols,
                                        fp8_recipe r, float *scale, float *scale_inv, uint8_t *q,
                                        uint8_t *qt, float *amax_out, uint16_t *dbias,
                                        float *workspace, cudaStream_t s);

/* Bytes of workspace fp8_quantize_fused_dynamic needs (16 KiB). */
size_t fp8_quantize_fused_workspace_bytes(void);

/* Current (dynamic) tensorwise scaling of x [rows, cols] in ONE launch, with
 * the results of fp8_quantize_transpose(..., FP8_RECIPE_DYNAMIC, ...): amax_out
 * = amax(x), scale/scale_inv from it, q [rows, cols] (nullable) and qt
 * [cols, rows] (nullable; not both NULL).  A persistent grid computes the amax,
 * meets at a grid-wide barrier and then casts, re-reading x from L2 when it
 * fits there (3 instead of 5 HBM bytes per element when only q is written).
 * rows % 16 == 0 and cols % 16 == 0.
 * workspace: caller-owned device memory of fp8_quantize_fused_workspace_bytes()
 * bytes, 16-byte aligned, set to zero once before its first use; each call
 * leaves it ready for the next.  Calls that may overlap on the GPU (other
 * streams) need separate workspaces.  After FP8_ERR_TIMEOUT from
 * fp8_check_device_status, zero the workspace again.
 * Source: SpecForge "Add training.fp8_linear" page (dynamic tensorwise
 * scaling); AstrAI fp8_state.py _update_delayed_scale (the scale rule). */
fp8_status fp8_quantize_fused_dynamic(const uint16_t *x, int64_t rows, int64_t cols, float *scale,
                                      float *scale_inv, uint8_t *q, uint8_t *qt, float *amax_out,
                                      void *workspace, cudaStream_t s);

/* fp8_quantize_fused_dynamic without a workspace argument, for callers that
 * cannot allocate device memory: a host framework that owns every byte of the
 * device in a pre-planned pool and forbids libraries from allocating, or a
 * plain C caller with no allocator of its own that must not pull in
 * cudaMalloc and the synchronisation it implies.  The source pages have no
 * counterpart to this call; it exists only for such callers.
 * Same arguments (minus the workspace) and results as
 * fp8_quantize_fused_dynamic.  Its scratch is a 4 KiB array in the library's
 * own static device memory (barrier words plus one partial amax for each of
 * at most 1008 CTAs), which every GPU that loads the library keeps until the
 * process exits.  The persistent grid is clamped to those 1008 CTAs (fewer
 * CTAs walk more tiles each and give the same bytes), so every tensor size
 * the call accepts fits the array; shapes with more than 2^31 - 1 tiles of
 * 128 x 128 are rejected with FP8_ERR_SHAPE.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress), so make that
 * first call before any stream capture.  Every call clears the barrier words
 * on `s` first (so a call after an FP8_ERR_TIMEOUT starts clean), and all
 * calls share the one array, so calls that may overlap on the GPU (other
 * streams, other host threads) race: issue them in one stream order.
 * Nothing here calls cudaMalloc, cudaFree or any allocating routine. */
fp8_status fp8_quantize_fused_dynamic_noalloc(const uint16_t *x, int64_t rows, int64_t cols,
                                              float *scale, float *scale_inv, uint8_t *q,
                                              uint8_t *qt, float *amax_out, cudaStream_t s);

/* ------------------------------------------------------------------------ */
/* Scaled FP8 GEMMs (tcgen05, fp32 accumulation in tensor memory, bf16 out)  */
/* ------------------------------------------------------------------------ */
/* M, N, K > 0 and each a multiple of 16 (SpecForge page: float8 GEMMs need the
 * token count to be a multiple of 16; the same holds for the feature dims).
 * BLOCK recipe: M, N, K multiples of 128.  Results overwrite the output.
 * Tensorwise recipes (DELAYED, DYNAMIC): x_scale, w_scale, g_scale are [1].
 * BLOCK recipe: activation/gradient scales are per 1x128 tile of the operand
 * as passed (row-major [rows, contraction/128]) and w_scale is the 128x128
 * grid [N/128, K/128] of W.  Under BLOCK the scale pointers must also be
 * 16-byte aligned (else FP8_ERR_ALIGNMENT).
 * Kernel choice is automatic.  For tests and tuning, environment variables
 * read at each call override it: FP8LINEAR_GEMM_PAIR=0/1 (tensorwise: one-CTA
 * or 2-SM pair kernel), FP8LINEAR_GEMM_BN=256/224/192/160/128 (tensorwise N
 * tile), FP8LINEAR_BLOCK_PAIR=0/1, FP8LINEAR_BLOCK_BN=128/256,
 * FP8LINEAR_BLOCK_ACC=0/1 (block recipe: one CTA or a CTA pair, tile width,
 * packed or scalar fp32 accumulators) and FP8LINEAR_BLOCK_GROUP=<row tiles>
 * (block recipe raster).  Every setting computes the same products in the
 * same order; the tests run each against the oracle.
 * Source: AstrAI fp8_state.py, the comment above FP8TensorMeta (the product
 * is scaled by A's and B's scales) and fp8_linear_forward /
 * fp8_linear_backward. */

/* y [M,N] = bf16( x_scale·w_scale · xq[M,K] · wq[N,K]ᵀ + bias[N] ).
 * bias (bf16 [N]) is nullable; it is added in fp32 before the bf16 rounding.
 * BLOCK: x_scale [M, K/128]; bias is not supported (must be NULL). */
fp8_status fp8_linear_fprop(const uint8_t *xq, const float *x_scale,
                            const uint8_t *wq, const float *w_scale,
                            int64_t M, int64_t N, int64_t K, fp8_recipe r,
                            const uint16_t *bias, uint16_t *y, cudaStream_t s);

/* dx [M,K] = bf16( g_scale·w_scale · gq[M,N] · wqt[K,N]ᵀ ), wqt = Wqᵀ.
 * BLOCK: g_scale [M, N/128]; w_scale is W's [N/128, K/128] grid. */
fp8_status fp8_linear_dgrad(const uint8_t *gq, const float *g_scale,
                            const uint8_t *wqt, const float *w_scale,
                            int64_t M, int64_t N, int64_t K, fp8_recipe r,
                            uint16_t *dx, cudaStream_t s);

/* dw [N,K] = bf16( g_scale·x_scale · gqt[N,M] · xqt[K,M]ᵀ ), gqt = Gqᵀ,
 * xqt = Xqᵀ.  The result overwrites dw (no accumulation into a main grad).
 * BLOCK: g_scale [M/128, N] and x_scale [M/128, K] are the column-tile scales
 * that fp8_quantize_transpose writes to scale_t. */
fp8_status fp8_linear_wgrad(const uint8_t *gqt, const float *g_scale,
                            const uint8_t *xqt, const float *x_scale,
                            int64_t M, int64_t N, int64_t K, fp8_recipe r,
                            uint16_t *dw, cudaStream_t s);

/* dgrad and wgrad of one backward pass in one launch (tensorwise recipes):
 * dx = fp8_linear_dgrad(gq, g_scale, wqt, w_scale) and
 * dw = fp8_linear_wgrad(gqt, g_scale, xqt, x_scale), same arguments, layouts
 * and results as those two calls (AstrAI page, fp8_linear_backward: the two
 * products of the backward of one linear).  The GEMMs are independent; on
 * large shapes whose contraction lengths (N for dgrad, M for wgrad) are
 * within 2x of each other their output tiles share one persistent launch of
 * the 2-SM kernel, so neither ends in a partly filled wave; otherwise they
 * run one after the other.  BLOCK returns FP8_ERR_UNSUPPORTED (its two GEMMs read
 * different scale layouts of G: use the single calls). */
fp8_status fp8_linear_dgrad_wgrad(const uint8_t *gq, const uint8_t *gqt, const float *g_scale,
                                  const uint8_t *wqt, const float *w_scale, const uint8_t *xqt,
                                  const float *x_scale, int64_t M, int64_t N, int64_t K,
                                  fp8_recipe r, uint16_t *dx, uint16_t *dw, cudaStream_t s);

/* ------------------------------------------------------------------------ */
/* Delayed-scaling state (one per weight)                                    */
/* ------------------------------------------------------------------------ */
/* Device block layout (fp32), FP8_META_FLOATS(interval) floats, 16-B aligned:
 *   [0] scale   [1] scale_inv      weight, from the amax-history window
 *   [2] x_scale [3] x_scale_inv    activation, lagged one call
 *   [4] g_scale [5] g_scale_inv    gradient, lagged one call
 *   [6]     x scale used by the forward GEMM of the step in progress
 *   [7]     g scale used by the backward GEMMs of the step in progress
 *           ([6] and [7] are written by fp8_linear_step_delayed; otherwise
 *           unused)
 *   [8 .. 8+interval) amax_history ring
 * Source: AstrAI fp8_state.py FP8TensorMeta (all fields start at 1). */
enum { FP8_META_SCALE = 0, FP8_META_SCALE_INV = 1, FP8_META_X_SCALE = 2,
       FP8_META_X_SCALE_INV = 3, FP8_META_G_SCALE = 4, FP8_META_G_SCALE_INV = 5,
       FP8_META_X_SCALE_FWD = 6, FP8_META_G_SCALE_BWD = 7, FP8_META_HISTORY = 8 };
#define FP8_META_FLOATS(interval) (8 + (interval))

typedef struct {
    float *dev;      /* caller-owned device block, FP8_META_FLOATS(interval) floats */
    int32_t interval;/* history length = refresh period (16 by default)            */
    int32_t idx;     /* next history slot (host side, like FP8TensorMeta.idx)       */
} fp8_meta;

typedef enum { FP8_SLOT_W = 0, FP8_SLOT_X = 1, FP8_SLOT_G = 2 } fp8_slot;

/* Sets every scale and every history slot to 1 and idx to 0.
 * 1 <= interval <= 1024. */
fp8_status fp8_meta_init(fp8_meta *m, float *dev_block, int32_t interval, cudaStream_t s);

/* W: history[idx] = *amax_dev and idx = (idx+1) % interval (FP8TensorMeta.record).
 * X, G: a = max(*amax_dev, 1e-12); x_scale (g_scale) = a/448 and
 *       x_scale_inv (g_scale_inv) = 448/a, for the next call
 *       (_update_delayed_scale).  Device-side; no synchronisation. */
fp8_status fp8_meta_record(fp8_meta *m, fp8_slot which, const float *amax_dev, cudaStream_t s);

/* m = max(history); if m > 0: scale = m/448, scale_inv = 448/m; else unchanged
 * (FP8TensorMeta.refresh). */
fp8_status fp8_meta_refresh(fp8_meta *m, cudaStream_t s);

/* Checkpoint of one meta: the scaling state a restore must keep (the NeMo
 * Speech page "feat(speechlm2): add padding-free packed speech training"
 * lists a fix that keeps checkpoint metadata through a restore; the state is
 * FP8TensorMeta's on the AstrAI page plus the step counter): a host byte blob = header (magic "F8MS", version 1, interval, idx,
 * step_count; host byte order) + the FP8_META_FLOATS(interval) floats of the
 * device block.  fp8_meta_state_bytes gives the blob size (0 for a bad
 * interval).  Save copies the device block out and synchronises `s` before
 * returning; load checks the header, copies the floats into dev_block
 * (caller-owned, FP8_META_FLOATS(interval) floats, 16-byte aligned),
 * synchronises `s`, then sets m (dev, interval, idx) and *step_count
 * (nullable).  A run restored from a blob continues bit for bit as the run
 * that saved it. */
size_t fp8_meta_state_bytes(int32_t interval);
fp8_status fp8_meta_save(const fp8_meta *m, int64_t step_count, void *host_buf, size_t bytes,
                         cudaStream_t s);
fp8_status fp8_meta_load(fp8_meta *m, float *dev_block, int64_t *step_count, const void *host_buf,
                         size_t bytes, cudaStream_t s);

/* FP8State.step: *step_count += 1 and, when it becomes a multiple of
 * interval, refresh every meta in metas[0..n).  Call once per training step
 * (at autocast entry), never again for the backward of the same step. */
fp8_status fp8_state_step(int64_t *step_count, int32_t interval, fp8_meta *metas, int32_t n,
                          cudaStream_t s);

/* ------------------------------------------------------------------------ */
/* One training step of one linear, delayed scaling (composite)              */
/* ------------------------------------------------------------------------ */
/* Caller-owned device buffers of one step.  x, w, y, xq, wq, wqt, amax are
 * required; g, gq, gqt, xqt, dx, dw may all be NULL for a forward-only step;
 * bias is optional. */
typedef struct {
    const uint16_t *x;    /* [M,K] bf16 activations (input)                   */
    const uint16_t *w;    /* [N,K] bf16 weight (input)                        */
    const uint16_t *g;    /* [M,N] bf16 upstream gradient (input, nullable)   */
    const uint16_t *bias; /* [N] bf16 (input, nullable)                       */
    uint8_t *xq;          /* [M,K] e4m3, X with the lagged x scale            */
    uint8_t *xqt;         /* [K,M] e4m3, Xᵀ with the x scale of this step     */
    uint8_t *wq;          /* [N,K] e4m3                                       */
    uint8_t *wqt;         /* [K,N] e4m3                                       */
    uint8_t *gq;          /* [M,N] e4m3                                       */
    uint8_t *gqt;         /* [N,M] e4m3                                       */
    float *amax;          /* [3] amax of x, w, g of this step (output)        */
    uint16_t *y;          /* [M,N] bf16 output                                */
    uint16_t *dx;         /* [M,K] bf16 input gradient (nullable)             */
    uint16_t *dw;         /* [N,K] bf16 weight gradient, overwritten (nullable) */
    uint16_t *dbias;      /* [N] bf16 bias gradient (nullable; needs g)        */
    float *dbias_workspace; /* fp8_dbias_workspace_bytes(M, N) (with dbias)    */
    int32_t flags;        /* FP8_STEP_* bits, 0 for the default step           */
} fp8_linear_step_io;

/* Step option: keep the forward's quantised activation for the backward
 * instead of quantising x again there.  The forward launch writes xqt
 * (Xq transposed, with the x scale fprop uses) beside xq, the backward reads
 * no x, and wgrad takes that forward x scale (slot FP8_META_X_SCALE_FWD).
 * This is the torchao float8 behaviour the SpecForge page credits for its
 * memory saving (float8 activations saved for backward); the default follows
 * the AstrAI page (x re-quantised in backward with the just-updated scale).
 * The two agree bit for bit whenever that update leaves the x scale as it
 * was (amax of this step's x equal to the previous one's). */
#define FP8_STEP_SAVE_XQ_FWD 1

/* Number of events fp8_linear_step_delayed records when given an array. */
#define FP8_STEP_NEVENTS 8

/* The AstrAI page's training step for one linear (fp8_autocast entry, then
 * fp8_linear_forward, then fp8_linear_backward), as one call that enqueues
 * every kernel:
 *   fp8_state_step (refresh every m->interval steps); amax[0..2] cleared;
 *   X -> xq with x_scale_inv (amax[0]) and W -> wq with scale_inv
 *   (amax[1]; also wqt when g is NULL), one launch, which also copies
 *   x_scale to slot FP8_META_X_SCALE_FWD;
 *   y = fprop(xq, x scale of that slot, wq, scale, bias);
 *   history[idx] = amax[1] and the lag update of the x scale from amax[0],
 *   one launch;
 *   if g: G -> gq, gqt with g_scale_inv (amax[2]), X -> xqt with the
 *   updated x_scale_inv and wqt = wq's bytes transposed, one launch, which
 *   also copies g_scale to slot
 *   FP8_META_G_SCALE_BWD (and, with dbias, sums G's columns as
 *   fp8_quantize_transpose_dbias does); the lag update of the g scale from
 *   amax[2];
 *   dx = dgrad(gq, g scale of that slot, wqt, scale) and
 *   dw = wgrad(gqt, g scale of that slot, xqt, x_scale) (both through
 *   fp8_linear_dgrad_wgrad when dx and dw are given).
 * Results are those of the single calls of the page's order (the GEMMs read
 * the scales the page's GEMMs read).  The forward state update, the backward
 * quantisation and the g-scale update do not depend on fprop, so they run on
 * a second stream owned by the library (one per host thread and device),
 * forked from and joined back into `s` with events: the memory-bound
 * quantisation overlaps the compute-bound GEMM.  To the caller everything is
 * ordered on `s` (work enqueued on `s` after this call sees all results).
 * The backward's Wqᵀ is the forward's Wq transposed byte for byte: the page
 * quantises w again with the same scale_inv, which gives the same bytes.  M, N, K multiples of 16.
 * `events` (nullable) receives FP8_STEP_NEVENTS cudaEventRecord calls on the
 * stream of each segment (before: the forward quantisation, fprop, the
 * forward state update, the backward quantisation, the backward state
 * update, dgrad, wgrad; and at the end; with both dx and dw the combined
 * launch lies between events 5 and 6 and event 7 follows event 6 directly);
 * events between kernels stop their overlap, so the step runs slower while
 * they are recorded.  Argument checks happen before anything is enqueued. */
fp8_status fp8_linear_step_delayed(fp8_meta *m, int64_t *step_count, const fp8_linear_step_io *io,
                                   int64_t M, int64_t N, int64_t K, cudaEvent_t *events,
                                   cudaStream_t s);

/* One training step of one linear under current (dynamic tensorwise) scaling,
 * the torchao Float8Linear recipe of the SpecForge page ("Add
 * training.fp8_linear", Modifications): X -> xq (and xqt with g), W -> wq (and
 * wqt with g), each through the single-launch dynamic quantiser (amax[0],
 * amax[1]); y = fprop(xq, wq) (+ bias); with g: G -> gq, gqt (amax[2]), then
 * dx and dw as fp8_linear_dgrad_wgrad computes them (either may be NULL).
 * Every scale comes from its tensor's own amax of this call (the lag rule
 * applied to the current amax).  `scales`: 6 device floats, receives
 * scale, scale_inv of x, w and g in that order.  `workspace`:
 * 3 * fp8_quantize_fused_workspace_bytes() of device memory, all zero before
 * the first call and reused as each call leaves it; concurrent calls need
 * their own.  io->dbias must be NULL and io->flags 0.  No state: the step is the
 * same at every call.  Argument checks happen before anything is enqueued. */
fp8_status fp8_linear_step_dynamic(const fp8_linear_step_io *io, float *scales, void *workspace,
                                   int64_t M, int64_t N, int64_t K, cudaStream_t s);

/* Current-scaling (dynamic tensorwise) fprop of a linear that fits one output
 * tile, in one launch: amax of x [M,K] and of w [N,K], scale = amax/448 and
 * scale_inv = 448/amax for each (amax clamped to 1e-12), the saturating e4m3
 * casts, and y [M,N] = bf16(x_scale*w_scale * xq*wqᵀ (+ bias[N], fp32 add
 * before the rounding)).  The same bytes, scales and outputs as
 * fp8_quantize_fused_dynamic on x and on w followed by fp8_linear_fprop, in one
 * launch instead of three: for the small, latency-bound shapes on which the
 * NeMo SALMAutomodel page reports FP8 slower than bf16 (the configuration
 * X [64,256], W [256,256]).  M <= 128, N <= 256, K <= 512, each a multiple of
 * 16 (else FP8_ERR_ALIGNMENT or, for larger shapes, FP8_ERR_UNSUPPORTED).
 * `scales`: 4 device floats, receives x scale, x scale_inv, w scale,
 * w scale_inv.  `amax` (2 device floats: x, w), `xq` [M,K], `wq` [N,K] and
 * `bias` are nullable.  x, w, xq, wq, y 16-byte aligned.  No workspace.
 * Source: SpecForge "Add training.fp8_linear" (dynamic tensorwise scaling);
 * AstrAI fp8_state.py (scale rule, D = A_SCALE * B_SCALE * A * B). */
fp8_status fp8_linear_fprop_dynamic_small(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N,
                                          int64_t K, const uint16_t *bias, float *scales,
                                          float *amax, uint8_t *xq, uint8_t *wq, uint16_t *y,
                                          cudaStream_t s);

/* One training step of one linear under the block recipe (TE recipe=block,
 * the NeMo "Add FP8 support for SALMAutomodel" page; 1x128 activation and
 * gradient tiles, 128x128 weight tiles): X -> xq with 1x128 row-tile scales
 * and xqt with 128x1 column-tile scales (one launch), W -> wq and wqt with
 * 128x128 tile scales, y = fprop(xq, wq); with g: G -> gq and gqt with row
 * and column tiles (one launch), dx = dgrad(gq, wqt), dw = wgrad(gqt, xqt)
 * (either may be NULL).  Same results as fp8_quantize_transpose and the
 * three GEMM calls with the BLOCK / BLOCK_2D recipes.  M, N, K multiples of
 * 128.  io->amax (nullable) receives the tensor amaxes of x, w, g; bias,
 * dbias and flags are not supported (NULL / 0).  Every scale array is
 * required and 16-byte aligned (the forward-only step leaves the column-tile
 * arrays of X written but unused). */
typedef struct {
    float *x_scale, *x_scale_inv;     /* [M, K/128]     row tiles of X (fprop)        */
    float *x_scale_t, *x_scale_inv_t; /* [M/128, K]     column tiles of X (wgrad)     */
    float *w_scale, *w_scale_inv;     /* [N/128, K/128] 128x128 tiles of W            */
    float *g_scale, *g_scale_inv;     /* [M, N/128]     row tiles of G (dgrad)        */
    float *g_scale_t, *g_scale_inv_t; /* [M/128, N]     column tiles of G (wgrad)     */
} fp8_block_step_scales;
fp8_status fp8_linear_step_block(const fp8_linear_step_io *io, const fp8_block_step_scales *sc,
                                 int64_t M, int64_t N, int64_t K, cudaStream_t s);

/* ------------------------------------------------------------------------ */
/* Token padding                                                             */
/* ------------------------------------------------------------------------ */

/* Rows rounded up to a multiple: ((rows + multiple - 1) / multiple) * multiple.
 * Host only; returns -1 for rows < 0 or multiple < 1. */
int64_t fp8_padded_rows(int64_t rows, int64_t multiple);

/* out [padded_rows, cols] = x [rows, cols] followed by zero rows, padded_rows =
 * fp8_padded_rows(rows, multiple) (written to *padded_rows, host pointer,
 * nullable).  x and out must not overlap.  Zero rows change no amax and no
 * real output row.  Source: SpecForge page (multiple of 16), NeMo SALMAutomodel
 * review (pad tokens appended at the end). */
fp8_status fp8_pad_tokens(const uint16_t *x, int64_t rows, int64_t cols, int64_t multiple,
                          uint16_t *out, int64_t *padded_rows, cudaStream_t s);

/* Token multiples under context / tensor parallelism (NeMo page "Add FP8
 * support for SALMAutomodel", review of its BSHD and THD padding helpers:
 * a rank's linear sees M = B*T/(cp*tp) tokens).  The FP8 GEMMs need every
 * rank's token count to be a multiple of 16, so:
 *   fp8_pad_multiple(cp, tp) = 16*cp*tp, the multiple to pass to
 *     fp8_pad_tokens for a packed (THD) batch;
 *   fp8_padded_seq_len(B, T, cp, tp) = the smallest T' >= T with T' a
 *     multiple of cp*tp (the sequence dim splits evenly) and B*T' a multiple
 *     of 16*cp*tp;
 *   fp8_pad_tokens_bshd: out [B, T', H] = x [B, T, H] with T' - T zero rows
 *     at the end of every sequence (H a multiple of 8, else
 *     FP8_ERR_ALIGNMENT); *padded_seq (nullable) receives T'.
 * -1 / FP8_ERR_SHAPE for batch < 1, seq < 0, cp or tp < 1. */
int64_t fp8_pad_multiple(int32_t cp_size, int32_t tp_size);
int64_t fp8_padded_seq_len(int64_t batch, int64_t seq, int32_t cp_size, int32_t tp_size);
fp8_status fp8_pad_tokens_bshd(const uint16_t *x, int64_t batch, int64_t seq, int64_t hidden,
                               int32_t cp_size, int32_t tp_size, uint16_t *out,
                               int64_t *padded_seq, cudaStream_t s);

/* ------------------------------------------------------------------------ */
/* Many weights at once                                                      */
/* ------------------------------------------------------------------------ */
/* Current-scaling amax and scales of n bf16 tensors in one pass (the
 * SpecForge page runs torchao's precompute_float8_dynamic_scale_for_fsdp
 * after every optimizer step: every float8 weight's scale computed together
 * before its cast): for each i, amax[i] = max |w[i]| over numel[i] elements
 * and scale[i], scale_inv[i] from it by the rule of fp8_meta_record's lag
 * update (clamp 1e-12, a/448, 448/a).  w is a host array of n device
 * pointers (16-byte aligned); amax, scale, scale_inv are device arrays of n
 * floats.  One amax launch per 64 tensors plus one scale launch; the scales
 * can then drive fp8_quantize / fp8_quantize_transpose with the DELAYED
 * recipe (scale_inv as input). */
fp8_status fp8_multi_amax_scales(const uint16_t *const *w, const int64_t *numel, int32_t n,
                                 float *amax, float *scale, float *scale_inv, cudaStream_t s);

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */

/* Synchronises `s`, then reads and clears the device status word that kernels
 * set when a bounded wait runs out.  Returns FP8_ERR_TIMEOUT if it was set,
 * FP8_ERR_CUDA on a CUDA error, else FP8_OK. */
fp8_status fp8_check_device_status(cudaStream_t s);

/* Test hook (host-side fault injection, no GPU involvement): the calling
 * thread's next n kernel launches made by the library fail with
 * cudaErrorLaunchFailure without launching, so callers can test how they
 * handle FP8_ERR_CUDA; n = 0 clears it.  Entry points that launch several
 * kernels may have enqueued the earlier ones before the failing launch. */
fp8_status fp8_inject_launch_failures(int32_t n);

/* Limit of every bounded wait in the library's kernels (mbarrier waits of the
 * GEMMs, the grid barrier of the single-launch dynamic quantiser), in
 * nanoseconds of the GPU's global timer; default 2 s, and 0 restores the
 * default.  Returns the previous limit.  A process-wide setting, read when a
 * kernel is launched (launches already enqueued keep theirs).  A wait that
 * runs out sets the device status word (FP8_ERR_TIMEOUT from
 * fp8_check_device_status) and its kernel returns without finishing its
 * outputs.  For callers that want faster failure detection, and for tests
 * that drive a wait into its timeout path without faulting or hanging the
 * GPU.  Host only, no GPU work. */
uint64_t fp8_set_wait_limit_ns(uint64_t limit_ns);

/* Diagnostic: launches one block that waits on a barrier nothing will ever
 * complete, with a wait limit of timeout_us microseconds (1..1000000); the
 * wait gives up, sets the device status word and the kernel returns.  Used to
 * test the timeout path without faulting or hanging the GPU. */
fp8_status fp8_selftest_wait_timeout(uint32_t timeout_us, cudaStream_t s);

/* Text of the last failure on this thread ("" if none). */
const char *fp8_last_error(void);

/* Library version, e.g. "fp8linear 0.1 sm_103a". */
const char *fp8_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP8LINEAR_H */
