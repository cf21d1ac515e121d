// rmsn_internal.h -- interface between the host entry points and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

// Geometry of one launch (chosen by the planner in rmsn_api.cu).
struct Launch {
    int wpr;        // warps per row group
    int nch;        // 16-byte vectors per lane per row (compile-time variant)
    int threads;    // threads per CTA
    int groups;     // row groups per CTA = threads / (32 * wpr)
    int64_t grid;   // CTAs (backward: row chunks)
    int64_t smem;   // dynamic shared memory bytes
};

// Chunk counts with a compiled kernel variant, per op (ascending).
constexpr int kFwdNch[] = {1, 2, 3, 4, 5, 6, 8, 12};
constexpr int kBwdNch[] = {1, 2, 3, 4, 6, 8};
constexpr int kFusedNch[] = {1, 2, 3, 4, 6, 8};

// dtype codes match rmsn_dtype: 0 = fp32, 1 = bf16
cudaError_t launch_fwd(const Launch& L, const void* x, int x_dt, const void* w, int w_dt,
                       void* y, float* rstd, int64_t T, int64_t H, float eps, cudaStream_t s);

cudaError_t launch_bwd(const Launch& L, const void* dy, const void* x, int x_dt, const void* w,
                       int w_dt, const float* rstd, void* dx, float* dw, int64_t T, int64_t H,
                       int deterministic, int compensated, float* ws, cudaStream_t s);

cudaError_t launch_fused(const Launch& L, const void* x, void* residual, const void* w,
                         uint8_t* q, float* block_scale, int64_t scale_ld, void* normed,
                         int64_t T, int64_t H, float eps, cudaStream_t s);

}  // namespace rmsn
