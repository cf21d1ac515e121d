// rmsn_fused_quant.cu -- residual add + RMSNorm + E4M3 1x128 block quantization in one
// pass (FlashInfer PR #4480 "Add FusedAddRMSNormFP8BlockQuant", Summary and Kernel).
//
// Per row (bf16 only):
//   h = bf16(x + residual)          -> written back to residual (pre-norm, in place)
//   rstd = 1/sqrt(mean(h^2) + eps)  (FP32, IEEE)
//   n = bf16((h * rstd) * w)        -> written to normed
//   per block b of 128 columns: amax = max|n|, scale = amax / 448 (IEEE FP32)
//                                   -> block_scale[b * ld + row]
//   q = e4m3_rn_satfinite(n / scale) (IEEE FP32 division; a block with amax 0 keeps the
//                                   signed zero of each element)
// The quantization reads the bf16-rounded n, so re-quantizing the normed output gives
// back q exactly.  With 16-byte vectors of 8 bf16, a 128-column block is held by 16
// consecutive lanes of one warp (the vectors v = c*G + l, G a multiple of 16), so its
// amax is a register-only shuffle among those 16 lanes.
//
// Unlike the page's single-wave one-CTA-per-row launch, the grid here is persistent and
// each row group is one or more warps; the quantization arithmetic is the same.
#include "rmsn_device.cuh"
#include "rmsn_internal.h"

namespace rmsn {

struct FusedArgs {
    const __nv_bfloat16* x;
    __nv_bfloat16* res;
    const __nv_bfloat16* w;
    uint8_t* q;
    float* scale;
    __nv_bfloat16* normed;
    int64_t T;
    int64_t ld;
    int H;
    int wpr;
    float eps;
};

// Round-to-nearest-even, saturating conversion of two floats to E4M3 (a in the low byte).
__device__ __forceinline__ uint16_t to_e4m3x2(float a, float b) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

template <int NCH>
__global__ void __launch_bounds__(512) fused_add_rmsnorm_fp8_kernel(FusedArgs a) {
    constexpr int VEC = 8;
    __shared__ float red[2 * 32];
    const int G = 32 * a.wpr;
    const int groups = blockDim.x / G;
    const int group = threadIdx.x / G;
    const int gl = threadIdx.x - group * G;
    const int H = a.H;
    const int nvec = H / VEC;
    const float Hf = (float)H;

    int parity = 0;
    for (int64_t row = (int64_t)blockIdx.x * groups + group; row < a.T;
         row += (int64_t)gridDim.x * groups) {
        const int64_t base = row * H;
        uint4 hv[NCH];
        {
            uint4 xv[NCH];
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const int v = c * G + gl;
                const bool ok = v < nvec;
                xv[c] = ok ? ld_stream(a.x + base + (int64_t)v * VEC) : make_uint4(0, 0, 0, 0);
                hv[c] = ok ? ld_stream(a.res + base + (int64_t)v * VEC) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                float xf[VEC], rf[VEC];
                Elem<__nv_bfloat16>::unpack(xv[c], xf);
                Elem<__nv_bfloat16>::unpack(hv[c], rf);
#pragma unroll
                for (int k = 0; k < VEC; ++k) rf[k] = __fadd_rn(xf[k], rf[k]);
                hv[c] = Elem<__nv_bfloat16>::pack(rf);  // h rounded once to bf16
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * G + gl;
            if (v < nvec) st_stream(a.res + base + (int64_t)v * VEC, hv[c]);
            float hf[VEC];
            Elem<__nv_bfloat16>::unpack(hv[c], hf);
#pragma unroll
            for (int k = 0; k < VEC; ++k) ss = fmaf(hf[k], hf[k], ss);
        }
        ss = group_sum(ss, a.wpr, red, group, parity);
        parity ^= 1;
        const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, Hf), a.eps)));

#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * G + gl;
            const bool ok = v < nvec;  // uniform over each 16-lane block (H % 128 == 0)
            float nf[VEC], wf[VEC];
            Elem<__nv_bfloat16>::unpack(hv[c], nf);
            if (ok) {
                load_w<__nv_bfloat16, VEC>(a.w, (int64_t)v * VEC, wf);
            } else {
#pragma unroll
                for (int k = 0; k < VEC; ++k) wf[k] = 0.f;
            }
#pragma unroll
            for (int k = 0; k < VEC; ++k) nf[k] = __fmul_rn(__fmul_rn(nf[k], rs), wf[k]);
            const uint4 nv = Elem<__nv_bfloat16>::pack(nf);
            if (ok) st_stream(a.normed + base + (int64_t)v * VEC, nv);
            Elem<__nv_bfloat16>::unpack(nv, nf);  // the bf16-rounded normed values

            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < VEC; ++k) amax = fmaxf(amax, fabsf(nf[k]));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float scale = __fdiv_rn(amax, 448.0f);
            if (ok && (gl & 15) == 0) a.scale[(int64_t)(v >> 4) * a.ld + row] = scale;

            uint32_t packed[2];
#pragma unroll
            for (int k = 0; k < VEC; k += 4) {
                float qv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    qv[u] = (scale > 0.f) ? __fdiv_rn(nf[k + u], scale) : nf[k + u];
                packed[k / 4] = (uint32_t)to_e4m3x2(qv[0], qv[1]) |
                                ((uint32_t)to_e4m3x2(qv[2], qv[3]) << 16);
            }
            if (ok)
                __stcs(reinterpret_cast<uint2*>(a.q + base + (int64_t)v * VEC),
                       make_uint2(packed[0], packed[1]));
        }
    }
}

cudaError_t launch_fused(const Launch& L, const void* x, void* residual, const void* w,
                         uint8_t* q, float* block_scale, int64_t scale_ld, void* normed,
                         int64_t T, int64_t H, float eps, cudaStream_t s) {
    FusedArgs a{static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(residual),
                static_cast<const __nv_bfloat16*>(w), q, block_scale,
                static_cast<__nv_bfloat16*>(normed), T, scale_ld, (int)H, L.wpr, eps};
#define RMSN_FUSED_CASE(N)                                                                     \
    case N:                                                                                    \
        fused_add_rmsnorm_fp8_kernel<N><<<(unsigned)L.grid, L.threads, 0, s>>>(a);             \
        return cudaGetLastError();
    switch (L.nch) {
        RMSN_FUSED_CASE(1)
        RMSN_FUSED_CASE(2)
        RMSN_FUSED_CASE(3)
        RMSN_FUSED_CASE(4)
        RMSN_FUSED_CASE(6)
        RMSN_FUSED_CASE(8)
        default:
            return cudaErrorInvalidConfiguration;
    }
#undef RMSN_FUSED_CASE
}

}  // namespace rmsn
