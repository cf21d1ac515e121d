// rmsn_bwd.cu -- fused single-pass RMSNorm backward with a strip-reduced weight gradient.
//
// FlashInfer PR #5741 "cake_rmsnorm_train", Design/Backward: a persistent grid over
// static row chunks; each CTA writes dx for its rows and keeps an FP32 dw partial for
// its chunk; the partials are reduced per column in chunk order, with no atomics, so dw
// depends only on (T, device).  Liger-Kernel PR #1336, Summary: the fused dX+dW
// strip-reduction backward.  miles-ext-kernels PR #15, Changes: TwoSum per-thread
// weight-gradient sums.
//
// This build reduces the partials with a second kernel on the same stream (no grid-wide
// barrier, so no CTA ever waits on another).
//
// Main kernel, per CTA (chunk c owns rows [c*T/n, (c+1)*T/n)):
//   each row group takes every `groups`-th row of the chunk; per row it loads x and dy
//   into registers (16-byte vectors), forms xhat = x*rstd and g = dy*w, reduces
//   sum(g*xhat) across the group, writes dx = rstd*(g - xhat*mean) and adds dy*xhat into
//   per-lane column accumulators that live in registers for the whole strip.
//   At the end the groups' accumulators are folded in group order through shared memory
//   and the CTA writes one partial row (deterministic mode) or adds it to dw with FP32
//   atomics (non-deterministic mode).
// Column-reduce kernel: dw[j] = sum over chunks of partial[chunk][j], in a fixed order.
#include "rmsn_device.cuh"
#include "rmsn_internal.h"

namespace rmsn {

struct BwdArgs {
    const void* dy;
    const void* x;
    const void* w;
    const float* rstd;
    void* dx;
    float* dw;   // non-deterministic mode: zeroed dw, atomically accumulated
    float* ws;   // deterministic mode: [n_chunks, H] high parts, then [n_chunks, H] low parts
    int64_t T;
    int H;
    int wpr;
    int atomic;
};

template <typename TX, typename TW, int NCH, bool COMP>
__global__ void __launch_bounds__(512) rmsnorm_bwd_kernel(BwdArgs a) {
    constexpr int VEC = Elem<TX>::VEC;
    constexpr int NL = COMP ? NCH : 1;  // low-part accumulators (unused when !COMP)
    extern __shared__ float fold[];     // [H] running high parts (+ [H] low parts)
    __shared__ float red[2 * 32];
    const int G = 32 * a.wpr;
    const int groups = blockDim.x / G;
    const int group = threadIdx.x / G;
    const int gl = threadIdx.x - group * G;
    const int H = a.H;
    const int nvec = H / VEC;
    const float Hf = (float)H;
    const int64_t nch = gridDim.x;
    const int64_t r0 = (int64_t)blockIdx.x * a.T / nch;
    const int64_t r1 = ((int64_t)blockIdx.x + 1) * a.T / nch;

    const TX* __restrict__ DY = static_cast<const TX*>(a.dy);
    const TX* __restrict__ X = static_cast<const TX*>(a.x);
    const TW* __restrict__ W = static_cast<const TW*>(a.w);
    TX* __restrict__ DX = static_cast<TX*>(a.dx);

    float acc[NCH][VEC];
    float accl[NL][VEC];
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[c][k] = 0.f;
#pragma unroll
    for (int c = 0; c < NL; ++c)
#pragma unroll
        for (int k = 0; k < VEC; ++k) accl[c][k] = 0.f;

    int parity = 0;
    for (int64_t row = r0 + group; row < r1; row += groups) {
        const int64_t base = row * H;
        uint4 xv[NCH], dv[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * G + gl;
            const bool ok = v < nvec;
            xv[c] = ok ? ld_stream(X + base + (int64_t)v * VEC) : make_uint4(0, 0, 0, 0);
            dv[c] = ok ? ld_stream(DY + base + (int64_t)v * VEC) : make_uint4(0, 0, 0, 0);
        }
        const float rs = __ldg(a.rstd + row);

        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * G + gl;
            if (v < nvec) {
                float xf[VEC], df[VEC], wf[VEC];
                Elem<TX>::unpack(xv[c], xf);
                Elem<TX>::unpack(dv[c], df);
                load_w<TW, VEC>(W, (int64_t)v * VEC, wf);
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    const float xh = __fmul_rn(xf[k], rs);
                    const float g = __fmul_rn(df[k], wf[k]);
                    dot = fmaf(g, xh, dot);
                }
            }
        }
        dot = group_sum(dot, a.wpr, red, group, parity);
        parity ^= 1;
        const float cm = __fdiv_rn(dot, Hf);

#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * G + gl;
            if (v < nvec) {
                float xf[VEC], df[VEC], wf[VEC], o[VEC];
                Elem<TX>::unpack(xv[c], xf);
                Elem<TX>::unpack(dv[c], df);
                load_w<TW, VEC>(W, (int64_t)v * VEC, wf);
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    const float xh = __fmul_rn(xf[k], rs);
                    const float g = __fmul_rn(df[k], wf[k]);
                    o[k] = __fmul_rn(rs, fmaf(-xh, cm, g));
                    const float p = __fmul_rn(df[k], xh);
                    if constexpr (COMP) {
                        comp_add(acc[c][k], accl[c][k], p);
                    } else {
                        acc[c][k] = __fadd_rn(acc[c][k], p);
                    }
                }
                st_stream(DX + base + (int64_t)v * VEC, Elem<TX>::pack(o));
            }
        }
    }

    // ---- fold the row groups' partials in group order, then emit the chunk's partial
    for (int gi = 0; gi < groups; ++gi) {
        if (group == gi) {
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const int v = c * G + gl;
                if (v < nvec) {
                    const int col0 = v * VEC;
                    float hv[VEC], lv[VEC];
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        float h = acc[c][k];
                        float l = COMP ? accl[COMP ? c : 0][k] : 0.f;
                        if (gi > 0) {
                            if constexpr (COMP) {
                                float fh = fold[col0 + k], fl = fold[H + col0 + k];
                                comp_merge(fh, fl, h, l);
                                h = fh;
                                l = fl;
                            } else {
                                h = __fadd_rn(fold[col0 + k], h);
                            }
                        }
                        hv[k] = h;
                        lv[k] = l;
                    }
                    if (gi + 1 < groups) {
#pragma unroll
                        for (int k = 0; k < VEC; ++k) {
                            fold[col0 + k] = hv[k];
                            if constexpr (COMP) fold[H + col0 + k] = lv[k];
                        }
                    } else if (a.atomic) {
#pragma unroll
                        for (int k = 0; k < VEC; ++k)
                            atomicAdd(a.dw + col0 + k, COMP ? __fadd_rn(hv[k], lv[k]) : hv[k]);
                    } else {
                        float* dst = a.ws + (int64_t)blockIdx.x * H + col0;
#pragma unroll
                        for (int k = 0; k < VEC; k += 4)
                            *reinterpret_cast<float4*>(dst + k) =
                                make_float4(hv[k], hv[k + 1], hv[k + 2], hv[k + 3]);
                        if constexpr (COMP) {
                            float* dl = dst + nch * H;
#pragma unroll
                            for (int k = 0; k < VEC; k += 4)
                                *reinterpret_cast<float4*>(dl + k) =
                                    make_float4(lv[k], lv[k + 1], lv[k + 2], lv[k + 3]);
                        }
                    }
                }
            }
        }
        if (groups > 1) __syncthreads();
    }
}

// dw[j] = sum_{chunk} ws[chunk][j] in a fixed order: the 8 warps of a CTA each add a
// contiguous range of chunks in chunk order, and warp 0 adds the 8 range sums in range
// order.  One CTA covers 128 columns (a float4 per lane).
template <bool COMP>
__global__ void __launch_bounds__(256) rmsnorm_dw_reduce_kernel(const float* __restrict__ ws,
                                                                float* __restrict__ dw, int H,
                                                                int n_chunks) {
    __shared__ float4 part[8][32];
    __shared__ float4 partl[8][32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int col = (blockIdx.x * 32 + lane) * 4;
    const bool ok = col < H;
    const int k0 = warp * n_chunks / 8;
    const int k1 = (warp + 1) * n_chunks / 8;
    const int64_t lo_off = (int64_t)n_chunks * H;
    float s[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
        int k = k0;
        for (; k + 4 <= k1; k += 4) {
            float4 v[4], vl[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                v[u] = __ldcg(reinterpret_cast<const float4*>(ws + (int64_t)(k + u) * H + col));
                if constexpr (COMP)
                    vl[u] = __ldcg(reinterpret_cast<const float4*>(ws + lo_off +
                                                                   (int64_t)(k + u) * H + col));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float hv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                if constexpr (COMP) {
                    const float lv[4] = {vl[u].x, vl[u].y, vl[u].z, vl[u].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) comp_merge(s[q], e[q], hv[q], lv[q]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) s[q] = __fadd_rn(s[q], hv[q]);
                }
            }
        }
        for (; k < k1; ++k) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(ws + (int64_t)k * H + col));
            const float hv[4] = {v.x, v.y, v.z, v.w};
            if constexpr (COMP) {
                const float4 vl =
                    __ldcg(reinterpret_cast<const float4*>(ws + lo_off + (int64_t)k * H + col));
                const float lv[4] = {vl.x, vl.y, vl.z, vl.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) comp_merge(s[q], e[q], hv[q], lv[q]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) s[q] = __fadd_rn(s[q], hv[q]);
            }
        }
    }
    part[warp][lane] = make_float4(s[0], s[1], s[2], s[3]);
    if constexpr (COMP) partl[warp][lane] = make_float4(e[0], e[1], e[2], e[3]);
    __syncthreads();
    if (warp == 0 && ok) {
        float t[4] = {s[0], s[1], s[2], s[3]}, te[4] = {e[0], e[1], e[2], e[3]};
        for (int w = 1; w < 8; ++w) {
            const float4 p = part[w][lane];
            const float ph[4] = {p.x, p.y, p.z, p.w};
            if constexpr (COMP) {
                const float4 pl = partl[w][lane];
                const float pv[4] = {pl.x, pl.y, pl.z, pl.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) comp_merge(t[q], te[q], ph[q], pv[q]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) t[q] = __fadd_rn(t[q], ph[q]);
            }
        }
        float4 out;
        if constexpr (COMP)
            out = make_float4(__fadd_rn(t[0], te[0]), __fadd_rn(t[1], te[1]),
                              __fadd_rn(t[2], te[2]), __fadd_rn(t[3], te[3]));
        else
            out = make_float4(t[0], t[1], t[2], t[3]);
        *reinterpret_cast<float4*>(dw + col) = out;
    }
}

template <typename TX, typename TW, int NCH, bool COMP>
static cudaError_t run_main(const Launch& L, const BwdArgs& a, cudaStream_t s) {
    auto k = rmsnorm_bwd_kernel<TX, TW, NCH, COMP>;
    if (L.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)L.smem);
        if (e != cudaSuccess) return e;
    }
    k<<<(unsigned)L.grid, L.threads, (size_t)L.smem, s>>>(a);
    return cudaGetLastError();
}

template <typename TX, typename TW, bool COMP>
static cudaError_t dispatch_nch(const Launch& L, const BwdArgs& a, cudaStream_t s) {
    switch (L.nch) {
        case 1: return run_main<TX, TW, 1, COMP>(L, a, s);
        case 2: return run_main<TX, TW, 2, COMP>(L, a, s);
        case 3: return run_main<TX, TW, 3, COMP>(L, a, s);
        case 4: return run_main<TX, TW, 4, COMP>(L, a, s);
        case 6: return run_main<TX, TW, 6, COMP>(L, a, s);
        case 8: return run_main<TX, TW, 8, COMP>(L, a, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

template <typename TX, typename TW>
static cudaError_t dispatch_comp(const Launch& L, const BwdArgs& a, int comp, cudaStream_t s) {
    return comp ? dispatch_nch<TX, TW, true>(L, a, s) : dispatch_nch<TX, TW, false>(L, a, s);
}

cudaError_t launch_bwd(const Launch& L, const void* dy, const void* x, int x_dt, const void* w,
                       int w_dt, const float* rstd, void* dx, float* dw, int64_t T, int64_t H,
                       int deterministic, int compensated, float* ws, cudaStream_t s) {
    BwdArgs a{dy, x, w, rstd, dx, dw, ws, T, (int)H, L.wpr, deterministic ? 0 : 1};
    if (!deterministic) {
        cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)H * sizeof(float), s);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e;
    if (x_dt == 1 && w_dt == 1) e = dispatch_comp<__nv_bfloat16, __nv_bfloat16>(L, a, compensated, s);
    else if (x_dt == 1 && w_dt == 0) e = dispatch_comp<__nv_bfloat16, float>(L, a, compensated, s);
    else if (x_dt == 0 && w_dt == 0) e = dispatch_comp<float, float>(L, a, compensated, s);
    else if (x_dt == 0 && w_dt == 1) e = dispatch_comp<float, __nv_bfloat16>(L, a, compensated, s);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess || !deterministic) return e;
    const unsigned rgrid = (unsigned)((H + 127) / 128);
    if (compensated)
        rmsnorm_dw_reduce_kernel<true><<<rgrid, 256, 0, s>>>(ws, dw, (int)H, (int)L.grid);
    else
        rmsnorm_dw_reduce_kernel<false><<<rgrid, 256, 0, s>>>(ws, dw, (int)H, (int)L.grid);
    return cudaGetLastError();
}

}  // namespace rmsn
