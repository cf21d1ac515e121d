// rmsn_internal.h -- interface between the host entry points and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

// Geometry of one launch (chosen by the planner in rmsn_api.cu).
//   Each CTA = `nw` consumer warps that share one row at a time + 1 producer warp whose
//   lane 0 streams the CTA's rows into a `stages`-deep shared-memory ring.
struct Launch {
    int nw;              // consumer warps per CTA
    int nch;             // 16-byte vectors per consumer lane per row (compile-time variant)
    bool single;         // backward: rows one at a time (bf16 rows of three vectors per lane)
    int stages;          // ring depth
    int ctas_per_sm;     // CTAs per SM the grid is sized for
    int sms;             // multiprocessors of the device
    uint32_t row_bytes;  // bytes of one input row
    uint32_t stage_bytes;// bytes of one stage (one or two padded rows)
    uint32_t w_bytes;    // bytes of the weight vector (copied to shared memory)
    uint32_t data_off;   // shared-memory offset of the first stage
    int64_t grid;        // CTAs planned (clamped to the kernel's occupancy at launch)
    int64_t smem;        // dynamic shared memory bytes per CTA
    unsigned* err;       // device error word (bounded waits that ran out)
    uint64_t limit_ns;   // time limit of every wait
};

// Chunk counts with a compiled kernel variant, per op (ascending).
constexpr int kFwdNch[] = {1, 2, 3, 4, 6, 8, 16};
constexpr int kBwdNch[] = {1, 2, 3, 4, 6, 8};
constexpr int kFusedNch[] = {1, 2, 3, 4, 6, 8};

// dtype codes match rmsn_dtype: 0 = fp32, 1 = bf16
// residual / h_new (forward) and g_residual (backward) select the residual variants
// (null: the plain ops); they have x's dtype.
cudaError_t launch_fwd(const Launch& L, const void* x, int x_dt, const void* w, int w_dt,
                       void* y, float* rstd, int64_t T, int64_t H, float eps, cudaStream_t s,
                       const void* residual = nullptr, void* h_new = nullptr);

cudaError_t launch_bwd(const Launch& L, const void* dy, const void* x, int x_dt, const void* w,
                       int w_dt, const float* rstd, void* dx, float* dw, int64_t T, int64_t H,
                       int deterministic, int compensated, float* ws, cudaStream_t s,
                       const void* g_residual = nullptr);

// One CTA that waits on an mbarrier nobody arrives at, with the given limit (self-test of
// the bounded wait; sets ERR_WAIT_FULL in *err).
cudaError_t launch_wait_selftest(unsigned* err, uint64_t limit_ns, cudaStream_t s);

// Deterministic backward for small T in one launch (row tasks for dx, column tasks for dw;
// no workspace).  g_residual selects the residual variant.
cudaError_t launch_bwd_small(const void* dy, const void* x, int x_dt, const void* w, int w_dt,
                             const float* rstd, void* dx, float* dw, int64_t T, int64_t H,
                             int compensated, cudaStream_t s, const void* g_residual = nullptr);

cudaError_t launch_fused(const Launch& L, const void* x, void* residual, const void* w,
                         uint8_t* q, float* block_scale, int64_t scale_ld, void* normed,
                         int64_t T, int64_t H, float eps, cudaStream_t s);

// Opts `kernel` into `smem` bytes of dynamic shared memory if that is above 48 KiB and
// returns in *grid the planned grid clamped to what stays resident at once (SMs x the
// kernel's occupancy at `threads` and `smem`), so a persistent grid never runs in two
// waves.  Cached per device and kernel.
cudaError_t fit_grid(const void* kernel, const Launch& L, int threads, int64_t* grid);

}  // namespace rmsn
