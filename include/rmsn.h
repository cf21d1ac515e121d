/*
 * rmsn.h -- C ABI of the GB300 (sm_103a) RMSNorm library.
 *
 * Three operations, each enqueued on a caller-provided CUDA stream:
 *
 *   rmsnorm_fwd                        y = x * rstd * w,  rstd = 1/sqrt(mean(x^2) + eps)
 *   rmsnorm_bwd                        dx = rstd * (g - xhat * mean(g * xhat)),
 *                                      dw = sum over rows of dy * xhat
 *                                      (g = dy * w, xhat = x * rstd), one fused pass
 *   fused_add_rmsnorm_fp8_block_quant  h = bf16(x + residual) -> residual (in place),
 *                                      normed = bf16(h * rstd * w),
 *                                      per 1x128 block: scale = amax/448,
 *                                      q = e4m3(normed / scale)
 *
 * Sources (page title and section):
 *   FlashInfer PR #5741 "cake_rmsnorm_train" (BF16 RMSNorm training forward and
 *     one-launch backward): Design (Forward, Backward), API, Memory, Determinism,
 *     Precision.
 *   Liger-Kernel PR #1336 "perf(cutedsl): fused dX+dW backward + host-enqueue caching
 *     for RMSNorm": Summary (fused single-pass dX+dW strip-reduction backward), review
 *     (persistent CTAs, 16-byte copies, warps per token).
 *   miles-ext-kernels PR #15 (re-vendoring the Cake RMSNorm packages): Changes
 *     (deterministic package, TwoSum per-thread weight-gradient sums), Accuracy
 *     (weight-gradient budget).
 *   FlashInfer PR #4480 "Add FusedAddRMSNormFP8BlockQuant": Summary, Kernel, API.
 *
 * Conventions shared by every entry point
 *   - Device pointers only (except where stated); the caller allocates every buffer,
 *     the library allocates nothing, never synchronizes the stream and keeps no
 *     pointer after it returns.  All work is enqueued on `stream` (NULL = the legacy
 *     default stream); completion is the caller's to observe.
 *   - [T, H] tensors are row-major and contiguous (row stride H elements).  Every
 *     [T, H] / [H] base pointer must be 16-byte aligned.  H must be a multiple of 8 for
 *     bf16 and of 4 for fp32 tensors (16-byte vectors) and at most RMSN_MAX_H.
 *   - Arguments are checked before anything is enqueued; a failed check returns a
 *     status and enqueues nothing.  A launch failure returns RMSN_ERR_CUDA.  Errors that
 *     the stream reports later (asynchronously) are the caller's to observe.
 *   - T == 0 is valid and enqueues no kernel (rmsnorm_bwd still zeroes dw).
 *   - Arithmetic: FP32 statistics and reductions, IEEE division and square root, no
 *     fast-math; bf16 outputs are rounded once, to nearest even.
 */
#ifndef RMSN_H_
#define RMSN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Stream handle; the same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* rmsn_stream_t;

/* Element types of x / dy / y / dx and of w. */
typedef enum {
    RMSN_F32 = 0,  /* IEEE binary32 */
    RMSN_BF16 = 1  /* bfloat16 */
} rmsn_dtype;

typedef enum {
    RMSN_OK = 0,
    RMSN_ERR_INVALID_ARG = 1,         /* NULL pointer, bad dtype code, T < 0, bad eps */
    RMSN_ERR_UNSUPPORTED_SHAPE = 2,   /* H out of range or not a multiple of the vector */
    RMSN_ERR_MISALIGNED = 3,          /* a pointer violates its alignment */
    RMSN_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace smaller than rmsnorm_bwd_workspace_bytes */
    RMSN_ERR_CUDA = 5,                /* a CUDA runtime call or a launch failed */
    RMSN_ERR_DEVICE_TIMEOUT = 6,      /* rmsn_device_status: a kernel's bounded wait ran out */
    RMSN_ERR_SCRATCH_LIMIT = 7        /* rmsnorm_bwd_noalloc: the call needs more scratch than
                                         the library's fixed RMSN_NOALLOC_SCRATCH_BYTES */
} rmsn_status;

#define RMSN_MAX_H 16384

/* Human-readable text of a status code (static storage; never NULL). */
const char* rmsn_status_string(int status);

/* ------------------------------------------------------------------------------------
 * rmsnorm_fwd -- RMSNorm forward; saves the FP32 reciprocal RMS for the backward.
 *
 * Source: FlashInfer PR #5741 "cake_rmsnorm_train", Design/Forward: FP32 sum of squares,
 * IEEE rsqrt in FP32, one pass that writes y = bf16(x * rstd * w) and the FP32 rstd;
 * API: cake_rmsnorm_train_forward(x, w, eps) -> (y, rstd).
 *
 *   x     [T, H] in x_dtype (device, read)
 *   w     [H] in w_dtype (device, read)
 *   y     [T, H] in x_dtype (device, written); y_ij = round(x_ij * rstd_i * w_j),
 *         the product formed in FP32 left to right and rounded once
 *   rstd  [T] fp32 (device, written); rstd_i = 1 / sqrt(sum_j x_ij^2 / H + eps)
 *   eps   finite, >= 0 (with eps == 0 an all-zero row gives rstd = inf)
 * The sum of squares is FP32, as the source states: a row whose sum of squares leaves the
 * FP32 range (finite elements of magnitude above about 1.8e19 / sqrt(H)) gets rstd = 0 and
 * y = 0, and its backward gives dx = 0 and no dW term.
 * Returns RMSN_OK or an error status (see conventions).
 * ---------------------------------------------------------------------------------- */
int rmsnorm_fwd(const void* x, int x_dtype, const void* w, int w_dtype, void* y, float* rstd,
                int64_t T, int64_t H, float eps, rmsn_stream_t stream);

/* ------------------------------------------------------------------------------------
 * rmsnorm_bwd_workspace_bytes -- size of the scratch buffer rmsnorm_bwd needs.
 *
 * Source: FlashInfer PR #5741, API (backward workspace query; caller-owned, reusable
 * across T) and Memory (per-chunk FP32 partials of dw).
 *
 * The workspace holds, per row chunk, the chunk's dw partial as two FP32 rows (the
 * high and low parts of a compensated sum): 8 * H bytes per chunk, at most
 * (SM count x CTAs per SM) chunks and never more than T.  The value returned for (T, H)
 * is an upper bound for every T' <= T with the same H and device, so one buffer can be
 * reused across calls.  `device` is a CUDA device ordinal (its SM count decides the
 * number of chunks); `compensated` does not change the size.  The same bound serves
 * rmsnorm_bwd_residual.  Returns 0 for T <= 0, for an unsupported H, or when the device
 * cannot be queried.
 * ---------------------------------------------------------------------------------- */
size_t rmsnorm_bwd_workspace_bytes(int64_t T, int64_t H, int compensated, int device);

/* ------------------------------------------------------------------------------------
 * rmsnorm_bwd -- fused single-pass RMSNorm backward: dx and dw together.
 *
 * Sources: FlashInfer PR #5741, Design/Backward: persistent CTAs, each owning a fixed
 * chunk of rows, compute dx = rstd * (dy*w - xhat * mean(dy*w*xhat)) for their rows in
 * FP32 and hold one FP32 dw partial per chunk; the partials are then reduced per
 * column in chunk order, without atomics.  Liger-Kernel PR #1336, Summary: the fused
 * dX+dW strip-reduction backward.  miles-ext-kernels PR #15, Changes: the
 * deterministic ("det") and non-deterministic ("fast") backward, and TwoSum per-thread
 * weight-gradient sums.
 *
 *   dy    [T, H] in x_dtype (device, read)
 *   x     [T, H] in x_dtype (device, read): the forward's input
 *   w     [H] in w_dtype (device, read)
 *   rstd  [T] fp32 (device, read): the forward's saved rstd
 *   dx    [T, H] in x_dtype (device, written)
 *   dw    [H] fp32 (device, written, overwritten -- not accumulated into)
 *   deterministic  != 0: each row chunk's partial goes to the workspace and a second
 *         kernel sums the partials per column in a fixed order; dw is bitwise
 *         reproducible and a function of (T, H, dtypes, compensated, the device, the
 *         library build and the launch policy) only.  For T <= rmsn_small_t_max() (256
 *         by default) one kernel does the whole backward instead, with dw summed over
 *         all rows per column slab in a fixed order (see rmsn_set_small_t_max).
 *         == 0: allows the library any order of the cross-chunk sum.  On GB300 the
 *         fixed-order reduction above is faster than the atomic sums measured (and plain
 *         FP32 atomics leave the weight-gradient budget at large T), so this setting runs
 *         the same kernels and its bits are reproducible too.
 *   compensated  != 0: each thread adds every product dy*xhat to an FP32 (high, low)
 *         pair with the error-free TwoSum transformation.
 *         == 0: each thread sums the products of the two rows of each row pair it
 *         processes with one FMA and adds that block sum to the (high, low) pair with
 *         TwoSum (blocked FP32 sums, blocks of two rows).  Where the kernel takes rows
 *         one at a time (bf16 rows of about three 16-byte vectors per consumer lane,
 *         e.g. H = 6144 with 8 consumer warps) the blocks are single rows, so both
 *         settings give the same bits.
 *         In both cases the chunk partials are (high, low) pairs and the column
 *         reduction merges them with TwoSum; dw = high + low rounded once.
 *   workspace, workspace_bytes  device scratch of at least
 *         rmsnorm_bwd_workspace_bytes(T, H, compensated, device) bytes, 16-byte
 *         aligned; its contents on entry do not matter and on exit are unspecified.
 *         Needed with either setting of deterministic.
 *   x_dtype fp32 supports H <= 8192 (bf16: H <= RMSN_MAX_H).
 * Returns RMSN_OK or an error status (see conventions).
 * ---------------------------------------------------------------------------------- */
int rmsnorm_bwd(const void* dy, const void* x, int x_dtype, const void* w, int w_dtype,
                const float* rstd, void* dx, float* dw, int64_t T, int64_t H,
                int deterministic, int compensated, void* workspace, size_t workspace_bytes,
                rmsn_stream_t stream);

/* ------------------------------------------------------------------------------------
 * fused_add_rmsnorm_fp8_block_quant -- residual add + RMSNorm + E4M3 1x128 block
 * quantization in one pass.
 *
 * Source: FlashInfer PR #4480 "Add FusedAddRMSNormFP8BlockQuant", Summary and Kernel:
 * emits the fp8 activation, one fp32 scale per 1x128 block in the column-major
 * (H/128, round_up(T, 4)) layout consumed by block-scaled fp8 GEMMs, the pre-norm
 * residual in place and the bf16 normed output; the fp8 is quantized from the
 * bf16-rounded normed value, so re-quantizing `normed` reproduces `q` exactly; a
 * block's amax is a register-only shuffle among the lanes that hold it.  API: the
 * caller allocates every output, residual is updated in place.
 *
 *   x         [T, H] bf16 (device, read)
 *   residual  [T, H] bf16 (device, read and written): residual_ij <- h_ij = bf16(x_ij + residual_ij)
 *   w         [H] bf16 (device, read)
 *   q         [T, H] E4M3 codes, one byte each (device, written):
 *             q_ij = e4m3_rn_satfinite(n_ij / scale_ib) with n = normed; if a block's
 *             amax is 0 its scale is 0 and q holds the signed zero of each element
 *   block_scale  fp32 (device, written): scale of (row m, block b = column/128) at
 *             block_scale[b * scale_ld + m], i.e. an (H/128, scale_ld) row-major buffer,
 *             unit stride along the rows; scale = amax_b(|n|) / 448 in IEEE FP32.
 *             Entries with m >= T are not written.
 *   scale_ld  >= round_up(T, 4)
 *   normed    [T, H] bf16 (device, written): n_ij = bf16(h_ij * rstd_i * w_j),
 *             rstd_i = 1/sqrt(mean_j h_ij^2 + eps)
 *   H         multiple of 128, at most RMSN_MAX_H
 * Alignment: x, residual, w, normed, q 16 bytes; block_scale 4 bytes.
 * Returns RMSN_OK or an error status (see conventions).
 * ---------------------------------------------------------------------------------- */
int fused_add_rmsnorm_fp8_block_quant(const void* x, void* residual, const void* w,
                                      uint8_t* q, float* block_scale, int64_t scale_ld,
                                      void* normed, int64_t T, int64_t H, float eps,
                                      rmsn_stream_t stream);

/* ------------------------------------------------------------------------------------
 * rmsnorm_fwd_residual -- the forward fused with the residual add of a transformer block.
 *
 * Source: FlashInfer PR #5741 "cake_rmsnorm_train", Design/Forward ("optionally fused with
 * a residual add: h_new = bf16(x + residual) is normalized") and API (the forward with
 * `residual=` returns y, rstd and h_new).
 *
 *   h_new[i, j] = round(x[i, j] + residual[i, j])      (one rounding to x's dtype)
 *   rstd[i]     = 1 / sqrt(mean_j(h_new[i, j]^2) + eps) (FP32)
 *   y[i, j]     = round((h_new[i, j] * rstd[i]) * w[j])
 *
 * Arguments: as rmsnorm_fwd, plus
 *   residual  device [T, H], x's dtype, row-major contiguous (read only)
 *   h_new     device [T, H], x's dtype (written); it is the input of rmsnorm_bwd_residual
 * Outputs may alias inputs of the same shape exactly (h_new == residual or h_new == x, the
 * usual in-place residual update): every row is read before it is written.  Partial
 * overlaps are not supported.  Alignment: x, residual, w, y, h_new 16 bytes; rstd 4 bytes.
 * T == 0 writes nothing.  Returns RMSN_OK or an error status (see conventions).
 * ---------------------------------------------------------------------------------- */
int rmsnorm_fwd_residual(const void* x, const void* residual, int x_dtype, const void* w,
                         int w_dtype, void* y, void* h_new, float* rstd, int64_t T, int64_t H,
                         float eps, rmsn_stream_t stream);

/* ------------------------------------------------------------------------------------
 * rmsnorm_bwd_residual -- the backward of rmsnorm_fwd_residual.
 *
 * Source: FlashInfer PR #5741 "cake_rmsnorm_train", Design/Backward (the residual backward
 * returns dx + g_residual as dx_total, the one gradient that x and residual, the two
 * addends of h_new, both receive) and API (the backward takes h_new, w, rstd and
 * g_residual).
 *
 *   dx_total[i, j] = round(rstd[i] * (dy*w - xhat * c_i)[j] + g_residual[i, j])  (FP32, one
 *                    rounding to h's dtype), xhat = h * rstd, c_i = mean_j(dy*w*xhat)
 *   dw[j]          = sum_i dy[i, j] * xhat[i, j]   (exactly as rmsnorm_bwd)
 *
 * Arguments: as rmsnorm_bwd with x = h (the forward's h_new), plus
 *   g_residual  device [T, H], h's dtype: the gradient reaching h_new through the residual
 *               stream (read only)
 *   dx_total    device [T, H], h's dtype (written); it may alias dy or g_residual exactly
 * The workspace and its size rule are those of rmsnorm_bwd (rmsnorm_bwd_workspace_bytes
 * covers both calls); the deterministic, compensated and error behaviour is the same.
 * Shapes: as rmsnorm_bwd.
 * ---------------------------------------------------------------------------------- */
int rmsnorm_bwd_residual(const void* dy, const void* h, int x_dtype, const void* w, int w_dtype,
                         const float* rstd, const void* g_residual, void* dx_total, float* dw,
                         int64_t T, int64_t H, int deterministic, int compensated,
                         void* workspace, size_t workspace_bytes, rmsn_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Launch policy (introspection).  The geometry the library uses for a call, computed
 * on the host without a GPU; `sm_count` is the device's multiprocessor count.
 *
 * Source: Liger-Kernel PR #1336, Summary and review (fast-path eligibility as a pure
 * host function of the shape: vector width and warp count; persistent CTAs; several
 * warps per token row).
 * ---------------------------------------------------------------------------------- */
typedef enum {
    RMSN_OP_FWD = 0,
    RMSN_OP_BWD = 1,
    RMSN_OP_FUSED_QUANT = 2,
    RMSN_OP_FWD_RESIDUAL = 3,
    RMSN_OP_BWD_RESIDUAL = 4
} rmsn_op;

/* Every kernel runs a persistent grid: a CTA is `consumer_warps` warps that share one
 * row at a time; the CTA's rows are streamed into a `stages`-deep shared-memory ring with
 * bulk copies (cp.async.bulk, mbarrier-tracked) by the first lane of one extra producer
 * warp (forward, fused quant) or by the first consumer thread (backward);
 * the weight vector is copied to shared memory once per CTA.  CTA b of a grid of G takes
 * the rows b, b + G, b + 2G, ...; the backward's CTAs are its row chunks.  At launch the
 * grid is clamped to the CTAs that are resident at once (the kernel's occupancy), so
 * `grid` below is an upper bound. */
typedef struct {
    int vec_elems;        /* elements per 16-byte vector */
    int consumer_warps;   /* warps that share one row */
    int chunks_per_lane;  /* 16-byte vectors each consumer lane holds per row */
    int threads;          /* threads per CTA: the consumer warps, plus one producer warp
                             in the forward and fused kernels */
    int stages;           /* depth of the shared-memory row ring */
    int ctas_per_sm;      /* CTAs per SM the grid is sized for */
    int64_t grid;         /* CTAs launched (for the backward: the number of row chunks) */
    int64_t smem_bytes;   /* dynamic shared memory per CTA */
    int64_t workspace_bytes; /* backward scratch (0 for the other ops) */
} rmsn_plan_t;

/* Fills *out for (op, T, H, dtypes) on a device with `sm_count` SMs and 228 KiB of
 * shared memory per SM (sm_100 / sm_103).  `compensated` does not change the plan.
 * Returns RMSN_OK, or the status the corresponding entry point would return for an
 * unsupported shape or dtype. */
int rmsn_plan(int op, int64_t T, int64_t H, int x_dtype, int w_dtype, int compensated,
              int sm_count, rmsn_plan_t* out);

/* Tuning hook for benchmarks: overrides the consumer warps per CTA (a power of two
 * <= 8, or 16 for the fused quant; any count <= 16 for the two backward ops), the CTAs per
 * SM and the maximum ring depth of
 * one op for the whole process (0 keeps a default).  The backward's chunk count, and so its dw bits, follow the CTAs
 * per SM; rmsnorm_bwd_workspace_bytes reflects the current setting.  Changing it while
 * calls are in flight on other host threads is a race.  Returns RMSN_ERR_INVALID_ARG for
 * values out of range (then nothing changes). */
int rmsn_set_policy(int op, int consumer_warps, int ctas_per_sm, int max_stages);

/* Small-T route of the deterministic backward (rmsnorm_bwd, rmsnorm_bwd_residual,
 * rmsnorm_bwd_noalloc).  Source: miles-ext-kernels PR #15, Changes (#8813: a column-task
 * weight-gradient kernel for the smallest T, one task per column slab summing the rows in
 * a fixed order with FP32 compensation).  Calls with deterministic = 1 and T <= t_max run
 * one kernel instead of the strip kernel and the column reduce: one CTA per row writes dx,
 * one CTA per 64 columns sums dy*xhat over all rows in a fixed order (8 interleaved row
 * sequences merged in order, compensated as `compensated` selects), and the workspace is
 * not touched (it is still required, so a call's arguments do not depend on the route).
 * dw bits depend on the route, so on (T, t_max) as well as on the other inputs.
 * rmsn_set_small_t_max sets t_max for the process (0 disables the route; default 256;
 * RMSN_ERR_INVALID_ARG above 2^20); changing it while calls are in flight on other host
 * threads is a race.  rmsn_small_t_max returns the current value. */
int rmsn_set_small_t_max(int64_t t_max);
int64_t rmsn_small_t_max(void);

/* ------------------------------------------------------------------------------------
 * rmsn_device_status -- every wait inside the kernels (a consumer waiting for a row to
 * land in shared memory, the producer waiting for a stage to be released) gives up after
 * 1 s, sets a bit in a per-device error word and ends the kernel early instead of
 * hanging; the outputs of that call are then incomplete.  This call synchronizes
 * `stream`, reads and clears the current device's error word into *flags (bit 0: a row
 * never landed; bit 1: a stage was never released; bit 2: copies were still in flight
 * when a CTA gave up) and returns RMSN_OK if it was 0, RMSN_ERR_DEVICE_TIMEOUT otherwise.
 * ---------------------------------------------------------------------------------- */
int rmsn_device_status(rmsn_stream_t stream, unsigned* flags);

/* Self-test of the bounded waits (no counterpart on the pages; it checks this library's
 * own failure path): enqueues on `stream` one CTA that waits on an mbarrier nobody will
 * complete, with a limit of `limit_ns` (1 .. 10^9), so the wait runs out and sets bit 0 of
 * the current device's error word, as a pipeline wait that never sees its row would.  No
 * copy is in flight and nothing else waits on it.  A following rmsn_device_status returns
 * RMSN_ERR_DEVICE_TIMEOUT with bit 0 set, and clears the word.  Returns RMSN_OK once the
 * kernel is enqueued, RMSN_ERR_INVALID_ARG for a limit out of range. */
int rmsn_selftest_wait_timeout(uint64_t limit_ns, rmsn_stream_t stream);

/* ------------------------------------------------------------------------------------
 * rmsnorm_bwd_noalloc -- the deterministic rmsnorm_bwd for callers that cannot allocate.
 *
 * The pages have no counterpart of this entry point.  rmsnorm_bwd needs a caller-owned
 * scratch workspace; some callers cannot provide one at the point of the call: a
 * framework whose allocator hands out all device memory up front from its own pool, a
 * latency-critical loop in which cudaMalloc's implicit device synchronization would stall
 * the pipeline, or a plain C caller with no allocator to size and own a workspace.  This
 * entry point keeps the workspace in a fixed array of RMSN_NOALLOC_SCRATCH_BYTES that the
 * library places in device memory when it is loaded (every GPU the library is used on
 * holds that array until the process exits); it calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Arguments, layouts and results are those of rmsnorm_bwd with deterministic = 1 (the
 * same kernels, so the same dx and, for the same device, dw).  The caller still provides
 * dy, x, w, rstd, dx and dw.
 *   - Calls with T <= rmsn_small_t_max() take the one-launch small-T route, which uses no
 *     scratch, so every supported H is accepted there.  Longer calls take the strip route,
 *     whose scratch is the workspace_bytes that rmsn_plan reports for RMSN_OP_BWD
 *     (8 * H * row chunks, the chunks being min(T, SMs * CTAs per SM)); when that exceeds
 *     RMSN_NOALLOC_SCRATCH_BYTES the call returns RMSN_ERR_SCRATCH_LIMIT and enqueues
 *     nothing.  On a 152-SM GB300 at the default policy the strip route fits for fp32 x
 *     at every supported H and for bf16 x at H <= 6896 and 8192 <= H <= 13792; the other
 *     bf16 widths (e.g. 16384) are accepted up to the small-T threshold only.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current, whichever route the call takes); make that first call
 *     before any stream capture.  The address is kept for the life of the process, so
 *     the library must not be used across cudaDeviceReset (the same holds for the
 *     device error word of rmsn_device_status).
 *   - All calls in the process share the one array.  Every call writes all the scratch it
 *     reads, so nothing has to start at zero, but calls that overlap on the GPU (on
 *     different streams, or from several host threads without ordering) race on the
 *     array and produce wrong dw: order them on one stream.
 * ---------------------------------------------------------------------------------- */
#define RMSN_NOALLOC_SCRATCH_BYTES (16u << 20)

int rmsnorm_bwd_noalloc(const void* dy, const void* x, int x_dtype, const void* w, int w_dtype,
                        const float* rstd, void* dx, float* dw, int64_t T, int64_t H,
                        int compensated, rmsn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RMSN_H_ */
