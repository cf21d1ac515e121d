// rmsn_bwd_small.cu -- deterministic RMSNorm backward for small T in one launch.
//
// miles-ext-kernels PR #15, Changes: a column-task weight-gradient kernel for the
// smallest T (#8813): one task per column slab sums the rows in a fixed order with FP32
// compensation, so the backward needs neither the chunk workspace nor the second-stage
// column reduce.
//
// The grid has two kinds of CTA that run side by side:
//   row CTAs    (blockIdx.x < T): CTA i computes row i's d = sum_j w_j * dy_j * x_j, the
//               scaled dot c' = rstd^2 * d / H and writes dx (the residual variant adds
//               g_residual), with the same per-element arithmetic as the strip kernel;
//   column CTAs (the rest): CTA s owns the columns [64 s, 64 s + 64); warp g sums the
//               rows g, g + 8, g + 16, ... in increasing order into a compensated (high,
//               low) pair per column, and the 8 warp partials are merged in warp order,
//               so dw[j] = the fixed-order compensated sum of dy_ij * x_ij * rstd_i,
//               rounded once.
// dw does not depend on the row dots, so no CTA waits for another.
#include <type_traits>

#include "rmsn_device.cuh"
#include "rmsn_internal.h"

namespace rmsn {

constexpr int kSmallThreads = 256;  // 8 warps
constexpr int kSlabCols = 64;       // columns per column CTA: one pair per lane

struct SmallArgs {
    const void* dy;
    const void* x;
    const void* w;
    const float* rstd;
    const void* gres;  // residual variant: g_residual rows (x's dtype), or null
    void* dx;
    float* dw;
    int64_t T;
    int H;
};

// Two consecutive elements (columns 2p, 2p+1) of a row as an FP32 pair.
template <typename T>
__device__ __forceinline__ f2 load_pair(const T* row, int p);
template <>
__device__ __forceinline__ f2 load_pair<float>(const float* row, int p) {
    const float2 v = __ldg(reinterpret_cast<const float2*>(row) + p);
    return f2_make(v.x, v.y);
}
template <>
__device__ __forceinline__ f2 load_pair<__nv_bfloat16>(const __nv_bfloat16* row, int p) {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(row) + p);
    return f2_make(bf16_lo(u), bf16_hi(u));
}

// The weights of 16-byte vector v of x (VEC = 2 NP elements) as FP32 pairs, from global
// memory (w is small and stays in L1/L2).
template <typename TW, int NP>
__device__ __forceinline__ void load_w_pairs(const void* w, int v, f2 (&wp)[NP]) {
    const TW* W = static_cast<const TW*>(w);
#pragma unroll
    for (int i = 0; i < NP; ++i) wp[i] = load_pair(W, v * NP + i);
}

template <typename TX, typename TW, bool COMP, bool RES>
__global__ void __launch_bounds__(kSmallThreads) rmsnorm_bwd_small_kernel(SmallArgs a) {
    constexpr int VEC = Elem<TX>::VEC;
    constexpr int NP = Pairs<TX>::NP;
    __shared__ float red[kSmallThreads / 32];
    __shared__ f2 part_hi[kSmallThreads / 32][32], part_lo[kSmallThreads / 32][32];
    const int t = threadIdx.x;
    const int H = a.H;
    const TX* __restrict__ X = static_cast<const TX*>(a.x);
    const TX* __restrict__ DY = static_cast<const TX*>(a.dy);

    if ((int64_t)blockIdx.x < a.T) {
        // ------------------------------------------------------------- row task: dx
        const int64_t row = blockIdx.x;
        const int nvec = H / VEC;
        const uint4* xr = reinterpret_cast<const uint4*>(X + row * H);
        const uint4* dr = reinterpret_cast<const uint4*>(DY + row * H);
        const float rs = __ldg(a.rstd + row);
        f2 acc = f2_splat(0.f);
        for (int v = t; v < nvec; v += kSmallThreads) {
            f2 p[NP], wp[NP];
            Pairs<TX>::prod(__ldg(dr + v), __ldg(xr + v), p);
            load_w_pairs<TW, NP>(a.w, v, wp);
#pragma unroll
            for (int i = 0; i < NP; ++i) acc = fma2(wp[i], p[i], acc);
        }
        const float d = __fadd_rn(f2_lo(acc), f2_hi(acc));
        // c' = rstd^2 * d / H: each warp's part of d is scaled by rstd^2 / H before the parts
        // are added (as in the strip kernel)
        const float m = __fmul_rn(rs, __fmul_rn(rs, __frcp_rn((float)H)));
        float dsum = d;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
        if ((t & 31) == 0) red[t >> 5] = __fmul_rn(dsum, m);
        __syncthreads();
        float c = red[0];
#pragma unroll
        for (int k = 1; k < kSmallThreads / 32; ++k) c += red[k];
        const f2 rs2 = f2_splat(rs), nc2 = f2_splat(-c);
        TX* dxr = static_cast<TX*>(a.dx) + row * H;
        const TX* gr = RES ? static_cast<const TX*>(a.gres) + row * H : nullptr;
        for (int v = t; v < nvec; v += kSmallThreads) {
            f2 xp[NP], dp[NP], wp[NP], o[NP];
            Pairs<TX>::get(__ldg(xr + v), xp);
            Pairs<TX>::get(__ldg(dr + v), dp);
            load_w_pairs<TW, NP>(a.w, v, wp);
#pragma unroll
            for (int i = 0; i < NP; ++i) o[i] = mul2(rs2, fma2(xp[i], nc2, mul2(dp[i], wp[i])));
            if constexpr (RES) {  // dx_total = dx + g_residual, rounded once
                Pairs<TX>::get(__ldg(reinterpret_cast<const uint4*>(gr) + v), xp);
#pragma unroll
                for (int i = 0; i < NP; ++i) o[i] = add2(o[i], xp[i]);
            }
            st_stream(dxr + (int64_t)v * VEC, Pairs<TX>::put(o));
        }
        return;
    }

    // ---------------------------------------------------------------- column task: dw
    const int s = (int)((int64_t)blockIdx.x - a.T);
    const int lane = t & 31, warp = t >> 5;
    const int p = s * (kSlabCols / 2) + lane;  // column pair 2p, 2p + 1
    const bool in = 2 * p < H;
    f2 hi = f2_splat(0.f), lo = f2_splat(0.f);
    if (in) {
        int64_t i = warp;
        constexpr int64_t kStride = kSmallThreads / 32;
        if constexpr (COMP) {
            for (; i < a.T; i += kStride) {
                const f2 pr = mul2(load_pair(DY + i * H, p), load_pair(X + i * H, p));
                comp_add2(hi, lo, mul2(f2_splat(__ldg(a.rstd + i)), pr));
            }
        } else {
            // blocked FP32: the terms of two consecutive rows of the warp's sequence are
            // summed with one FMA, the block sum is added with TwoSum
            for (; i + kStride < a.T; i += 2 * kStride) {
                const f2 p0 = mul2(load_pair(DY + i * H, p), load_pair(X + i * H, p));
                const f2 p1 = mul2(load_pair(DY + (i + kStride) * H, p),
                                   load_pair(X + (i + kStride) * H, p));
                const f2 q0 = mul2(f2_splat(__ldg(a.rstd + i)), p0);
                comp_add2(hi, lo, fma2(f2_splat(__ldg(a.rstd + i + kStride)), p1, q0));
            }
            if (i < a.T) {
                const f2 p0 = mul2(load_pair(DY + i * H, p), load_pair(X + i * H, p));
                comp_add2(hi, lo, mul2(f2_splat(__ldg(a.rstd + i)), p0));
            }
        }
    }
    part_hi[warp][lane] = hi;
    part_lo[warp][lane] = lo;
    __syncthreads();
    if (warp == 0 && in) {
        float h0 = f2_lo(part_hi[0][lane]), l0 = f2_lo(part_lo[0][lane]);
        float h1 = f2_hi(part_hi[0][lane]), l1 = f2_hi(part_lo[0][lane]);
#pragma unroll
        for (int k = 1; k < kSmallThreads / 32; ++k) {
            comp_merge(h0, l0, f2_lo(part_hi[k][lane]), f2_lo(part_lo[k][lane]));
            comp_merge(h1, l1, f2_hi(part_hi[k][lane]), f2_hi(part_lo[k][lane]));
        }
        *reinterpret_cast<float2*>(a.dw + 2 * p) = make_float2(__fadd_rn(h0, l0), __fadd_rn(h1, l1));
    }
}

template <typename TX, typename TW>
static cudaError_t dispatch(const SmallArgs& a, int compensated, cudaStream_t s) {
    const int64_t grid = a.T + (a.H + kSlabCols - 1) / kSlabCols;
    const bool res = a.gres != nullptr;
    auto k = compensated ? (res ? rmsnorm_bwd_small_kernel<TX, TW, true, true>
                                : rmsnorm_bwd_small_kernel<TX, TW, true, false>)
                         : (res ? rmsnorm_bwd_small_kernel<TX, TW, false, true>
                                : rmsnorm_bwd_small_kernel<TX, TW, false, false>);
    k<<<(unsigned)grid, kSmallThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_small(const void* dy, const void* x, int x_dt, const void* w, int w_dt,
                             const float* rstd, void* dx, float* dw, int64_t T, int64_t H,
                             int compensated, cudaStream_t s, const void* g_residual) {
    SmallArgs a{dy, x, w, rstd, g_residual, dx, dw, T, (int)H};
    if (x_dt == 1 && w_dt == 1) return dispatch<__nv_bfloat16, __nv_bfloat16>(a, compensated, s);
    if (x_dt == 1 && w_dt == 0) return dispatch<__nv_bfloat16, float>(a, compensated, s);
    if (x_dt == 0 && w_dt == 0) return dispatch<float, float>(a, compensated, s);
    if (x_dt == 0 && w_dt == 1) return dispatch<float, __nv_bfloat16>(a, compensated, s);
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
