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
// back q exactly.  With 16-byte vectors of 8 bf16 and lane-contiguous vectors
// (v = c * NC + t), a 128-column block is held by 16 consecutive lanes of one warp, so its
// amax is a register-only shuffle among those 16 lanes.
//
// The page's kernel runs one CTA per row in a single wave; here the grid is persistent:
// CTA b streams the rows b, b + G, ... (x and residual) through a shared-memory ring
// filled by bulk copies, and its consumer warps share one row at a time; w is copied to
// shared memory once per CTA.
#include "rmsn_device.cuh"
#include "rmsn_internal.h"
#include "rmsn_pipe.cuh"

namespace rmsn {

struct FusedArgs {
    const __nv_bfloat16* x;
    __nv_bfloat16* res;
    const __nv_bfloat16* w;
    uint8_t* q;
    float* scale;
    __nv_bfloat16* normed;
    unsigned* err;
    int64_t T;
    int64_t ld;
    uint64_t limit_ns;
    int H;
    int nw;
    int stages;
    uint32_t row_bytes;
    uint32_t stage_bytes;
    uint32_t w_bytes;
    uint32_t data_off;
    float eps;
};

// Round-to-nearest-even, saturating conversion of two floats to E4M3 (a in the low byte).
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

template <int NCH>
__global__ void __launch_bounds__(288, 3) fused_add_rmsnorm_fp8_kernel(FusedArgs a) {
    constexpr int VEC = 8;
    extern __shared__ __align__(128) uint8_t smem[];
    const Ring ring = ring_at(smem, a.stages, a.stage_bytes, a.data_off);
    const uint8_t* wsm = smem + kRingHeader;
    const int nw = a.nw;
    const int64_t G = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t nrows = (a.T - 1 - b) / G + 1;  // rows b, b + G, ... below T
    const uint32_t r_off = a.stage_bytes / 2;  // stage = [x row | residual row]
    stage_weights(a.w, smem + kRingHeader, a.w_bytes);
    ring_init(ring, nw);

    if ((int)(threadIdx.x >> 5) == nw) {  // producer warp
        if ((threadIdx.x & 31) == 0) {
            const uint8_t* X = reinterpret_cast<const uint8_t*>(a.x);
            const uint8_t* R = reinterpret_cast<const uint8_t*>(a.res);
            const int64_t issued = ring_produce(
                ring, nrows, a.limit_ns, a.err, [&](int64_t k, uint8_t* dst, uint64_t* full) {
                    const int64_t off = (b + k * G) * (int64_t)a.row_bytes;
                    mbar_arrive_expect_tx(full, 2 * a.row_bytes);
                    bulk_load(dst, X + off, a.row_bytes, full);
                    bulk_load(dst + r_off, R + off, a.row_bytes, full);
                });
            ring_drain(ring, issued, a.limit_ns, a.err);
        }
        return;
    }

    const int t = threadIdx.x;
    const int NC = nw * 32;
    const int H = a.H;
    const int nvec = H / VEC;
    const float Hf = (float)H;

    for (int64_t k = 0; k < nrows; ++k) {
        const int64_t row = b + k * G;
        const int64_t base = row * H;
        const bool ok = ring_wait_full(ring, k, a.limit_ns, a.err);
        const uint8_t* st = ring.stage((int)(k % ring.stages));
        uint4 hv[NCH];
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * NC + t;
            const bool in = ok && v < nvec;
            const uint4 xv = in ? lds128(st + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
            const uint4 rv = in ? lds128(st + r_off + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
            float xf[VEC], rf[VEC];
            Elem<__nv_bfloat16>::unpack(xv, xf);
            Elem<__nv_bfloat16>::unpack(rv, rf);
#pragma unroll
            for (int q = 0; q < VEC; ++q) rf[q] = __fadd_rn(xf[q], rf[q]);
            hv[c] = Elem<__nv_bfloat16>::pack(rf);  // h rounded once to bf16
        }
        if (__all_sync(0xffffffffu, ok)) ring_release(ring, k);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * NC + t;
            if (ok && v < nvec) st_stream(a.res + base + (int64_t)v * VEC, hv[c]);
            float hf[VEC];
            Elem<__nv_bfloat16>::unpack(hv[c], hf);
#pragma unroll
            for (int q = 0; q < VEC; ++q) ss = fmaf(hf[q], hf[q], ss);
        }
        if (!consumer_sum(smem, ss, ok, nw, (int)(k & 1))) break;
        const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, Hf), a.eps)));

#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * NC + t;
            const bool in = v < nvec;  // uniform over each 16-lane block (H % 128 == 0)
            float nf[VEC], wf[VEC];
            Elem<__nv_bfloat16>::unpack(hv[c], nf);
            if (in) {
                WSmem<__nv_bfloat16, VEC>::get(wsm, v, wf);
            } else {
#pragma unroll
                for (int q = 0; q < VEC; ++q) wf[q] = 0.f;
            }
#pragma unroll
            for (int q = 0; q < VEC; ++q) nf[q] = __fmul_rn(__fmul_rn(nf[q], rs), wf[q]);
            const uint4 nv = Elem<__nv_bfloat16>::pack(nf);
            if (in) st_stream(a.normed + base + (int64_t)v * VEC, nv);
            Elem<__nv_bfloat16>::unpack(nv, nf);  // the bf16-rounded normed values

            float amax = 0.f;
#pragma unroll
            for (int q = 0; q < VEC; ++q) amax = fmaxf(amax, fabsf(nf[q]));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float scale = __fdiv_rn(amax, 448.0f);
            if (in && (t & 15) == 0) a.scale[(int64_t)(v >> 4) * a.ld + row] = scale;

            uint32_t packed[2];
#pragma unroll
            for (int q = 0; q < VEC; q += 4) {
                float qv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    qv[u] = (scale > 0.f) ? __fdiv_rn(nf[q + u], scale) : nf[q + u];
                packed[q / 4] = to_e4m3x2(qv[0], qv[1]) | (to_e4m3x2(qv[2], qv[3]) << 16);
            }
            if (in)
                __stcs(reinterpret_cast<uint2*>(a.q + base + (int64_t)v * VEC),
                       make_uint2(packed[0], packed[1]));
        }
    }
}

template <int NCH>
static cudaError_t run(const Launch& L, const FusedArgs& a, cudaStream_t s) {
    auto k = fused_add_rmsnorm_fp8_kernel<NCH>;
    const int threads = L.nw * 32 + 32;
    int64_t grid = 0;
    cudaError_t e = fit_grid((const void*)k, L, threads, &grid);
    if (e != cudaSuccess) return e;
    k<<<(unsigned)grid, threads, (size_t)L.smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fused(const Launch& L, const void* x, void* residual, const void* w,
                         uint8_t* q, float* block_scale, int64_t scale_ld, void* normed,
                         int64_t T, int64_t H, float eps, cudaStream_t s) {
    FusedArgs a{static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(residual),
                static_cast<const __nv_bfloat16*>(w), q, block_scale,
                static_cast<__nv_bfloat16*>(normed), L.err, T, scale_ld, L.limit_ns, (int)H,
                L.nw, L.stages, L.row_bytes, L.stage_bytes, L.w_bytes, L.data_off, eps};
    switch (L.nch) {
        case 1: return run<1>(L, a, s);
        case 2: return run<2>(L, a, s);
        case 3: return run<3>(L, a, s);
        case 4: return run<4>(L, a, s);
        case 6: return run<6>(L, a, s);
        case 8: return run<8>(L, a, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace rmsn
