// rmsn_fwd.cu -- persistent RMSNorm forward (FlashInfer PR #5741 "cake_rmsnorm_train",
// Design/Forward: FP32 sum of squares, two-level shuffle/shared reduce, IEEE rsqrt in
// FP32, one pass that writes y and the FP32 rstd).
//
// A persistent grid walks the rows with a grid stride; each row group (one or more
// warps, Liger-Kernel PR #1336 review: "each warp handles separate tokens") keeps its
// row in registers between the reduction and the write, so x is read from HBM once.
#include "rmsn_device.cuh"
#include "rmsn_internal.h"

namespace rmsn {

struct FwdArgs {
    const void* x;
    const void* w;
    void* y;
    float* rstd;
    int64_t T;
    int H;
    int wpr;
    float eps;
};

template <typename TX, typename TW, int NCH>
__global__ void __launch_bounds__(512) rmsnorm_fwd_kernel(FwdArgs a) {
    constexpr int VEC = Elem<TX>::VEC;
    __shared__ float red[2 * 32];
    const int G = 32 * a.wpr;
    const int groups = blockDim.x / G;
    const int group = threadIdx.x / G;
    const int gl = threadIdx.x - group * G;
    const int nvec = a.H / VEC;
    const float Hf = (float)a.H;
    const TX* __restrict__ X = static_cast<const TX*>(a.x);
    const TW* __restrict__ W = static_cast<const TW*>(a.w);
    TX* __restrict__ Y = static_cast<TX*>(a.y);

    int parity = 0;
    for (int64_t row = (int64_t)blockIdx.x * groups + group; row < a.T;
         row += (int64_t)gridDim.x * groups) {
        const TX* xr = X + row * a.H;
        uint4 xv[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * G + gl;
            xv[c] = (v < nvec) ? ld_stream(xr + (int64_t)v * VEC) : make_uint4(0, 0, 0, 0);
        }
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float f[VEC];
            Elem<TX>::unpack(xv[c], f);
#pragma unroll
            for (int k = 0; k < VEC; ++k) ss = fmaf(f[k], f[k], ss);
        }
        ss = group_sum(ss, a.wpr, red, group, parity);
        parity ^= 1;
        const float ms = __fdiv_rn(ss, Hf);
        const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, a.eps)));
        if (gl == 0) a.rstd[row] = rs;

        TX* yr = Y + row * a.H;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * G + gl;
            if (v < nvec) {
                float f[VEC], wf[VEC];
                Elem<TX>::unpack(xv[c], f);
                load_w<TW, VEC>(W, (int64_t)v * VEC, wf);
#pragma unroll
                for (int k = 0; k < VEC; ++k) f[k] = __fmul_rn(__fmul_rn(f[k], rs), wf[k]);
                st_stream(yr + (int64_t)v * VEC, Elem<TX>::pack(f));
            }
        }
    }
}

template <typename TX, typename TW>
static cudaError_t dispatch(const Launch& L, const FwdArgs& a, cudaStream_t s) {
#define RMSN_FWD_CASE(N)                                                                  \
    case N:                                                                               \
        rmsnorm_fwd_kernel<TX, TW, N><<<(unsigned)L.grid, L.threads, 0, s>>>(a);          \
        return cudaGetLastError();
    switch (L.nch) {
        RMSN_FWD_CASE(1)
        RMSN_FWD_CASE(2)
        RMSN_FWD_CASE(3)
        RMSN_FWD_CASE(4)
        RMSN_FWD_CASE(5)
        RMSN_FWD_CASE(6)
        RMSN_FWD_CASE(8)
        RMSN_FWD_CASE(12)
        default:
            return cudaErrorInvalidConfiguration;
    }
#undef RMSN_FWD_CASE
}

cudaError_t launch_fwd(const Launch& L, const void* x, int x_dt, const void* w, int w_dt,
                       void* y, float* rstd, int64_t T, int64_t H, float eps, cudaStream_t s) {
    FwdArgs a{x, w, y, rstd, T, (int)H, L.wpr, eps};
    if (x_dt == 1 && w_dt == 1) return dispatch<__nv_bfloat16, __nv_bfloat16>(L, a, s);
    if (x_dt == 1 && w_dt == 0) return dispatch<__nv_bfloat16, float>(L, a, s);
    if (x_dt == 0 && w_dt == 0) return dispatch<float, float>(L, a, s);
    if (x_dt == 0 && w_dt == 1) return dispatch<float, __nv_bfloat16>(L, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
