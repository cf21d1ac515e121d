// rmsn_fused_quant.cu -- residual add + RMSNorm + E4M3 1x128 block quantization in one
// pass (FlashInfer PR #4480 "Add FusedAddRMSNormFP8BlockQuant", Summary and Kernel).
//
// Per row (bf16 only):
//   h = bf16(x + residual)          -> written back to residual (pre-norm, in place)
//   rstd = 1/sqrt(mean(h^2) + eps)  (FP32, IEEE)
//   n = bf16((h * rstd) * w)        -> written to normed
//   per block b of 128 columns: amax = max|n|, scale = amax / 448 (IEEE FP32)
//                                   -> block_scale[b * ld + row]
//   q = e4m3_rn_satfinite(n / scale) (the code of the IEEE FP32 quotient; a block with
//                                   amax 0 keeps the signed zero of each element)
// The quantization reads the bf16-rounded n, so re-quantizing the normed output gives
// back q exactly.  With 16-byte vectors of 8 bf16 and lane-contiguous vectors
// (v = c * NC + t), a 128-column block is held by 16 consecutive lanes of one warp, so its
// amax is a register-only shuffle among those 16 lanes.
//
// The page's kernel runs one CTA per row in a single wave; here the grid is persistent:
// CTA b streams the rows b, b + G, ... (x and residual) through a shared-memory ring
// filled by bulk copies, and its consumer warps share one row at a time; w is copied to
// shared memory (as FP32) once per CTA.  The arithmetic runs on FP32 pairs (two IEEE
// operations per instruction, each rounded as its scalar form would be).
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

// scale = RN(amax / 448) for a bf16 value amax in [2^-100, max finite]: Markstein's
// correction of the product with c = RN(1/448) (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", 1990): q0 = RN(amax * c), the residual
// r = amax - 448 * q0 is exact in one FMA, and RN(q0 + r * c) is the correctly rounded
// quotient.  Checked exhaustively against the exact quotient for every bf16 value of that
// range (29184 values; tests/test_oracle_pins.py re-derives the check).  Outside it (0,
// tiny, inf) the IEEE division is used.
__device__ __forceinline__ float scale_of(float amax) {
    constexpr float c = 1.0f / 448.0f;  // RN(1/448)
    if (!(amax >= 0x1p-100f && amax <= 0x1.fep127f)) return __fdiv_rn(amax, 448.0f);
    const float q0 = __fmul_rn(amax, c);
    const float r = __fmaf_rn(-q0, 448.0f, amax);
    return __fmaf_rn(r, c, q0);
}

// y ~ 1/s for a normal s within 2^-23 relative: the approximate reciprocal followed by one
// Newton-Raphson step y1 = y0 + y0 * (1 - s * y0) (the step squares the relative error of
// y0 and adds at most one rounding).
__device__ __forceinline__ float recip_of(float s) {
    float y0;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(s));
    return __fmaf_rn(y0, __fmaf_rn(-s, y0, 1.0f), y0);
}

// E4M3 codes (round to nearest even, saturating) of two FP32 pairs, packed into one word:
// a.lo in byte 0, a.hi in byte 1, b.lo in byte 2, b.hi in byte 3.
__device__ __forceinline__ uint32_t e4m3x4(f2 a, f2 b) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(f2_lo(a)), "f"(f2_hi(a)), "f"(f2_lo(b)), "f"(f2_hi(b)));
    return r;
}

// E4M3 codes of RN(n / s) for the eight bf16-rounded normed values of a 16-byte vector
// (four pairs), s > 0 the block scale and y ~ 1/s within 2^-23 relative (s and y normal),
// packed as two words (element order).  The IEEE quotient Q = RN(n / s) is not formed
// directly: q0 = RN(n * y) satisfies |q0 - Q| < 4.01 * 2^-24 * |q0|, so
// lo = RN(q0 * (1 - 2^-21)) and hi = RN(q0 * (1 + 2^-21)) bracket Q.  The conversion is
// monotone, so where lo and hi give the same code it is the code of Q.  If any element of
// the vector differs (Q within a few units in the last place of an E4M3 rounding boundary:
// about one element in 10^5), the vector's codes are taken from the IEEE division itself.
__device__ __forceinline__ uint2 quotient_codes(const f2 (&n)[4], float y, float s) {
    const f2 y2 = f2_splat(y);
    const f2 dn = f2_splat(1.0f - 0x1p-21f), up = f2_splat(1.0f + 0x1p-21f);
    f2 q0[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q0[i] = mul2(n[i], y2);
    const uint32_t lo0 = e4m3x4(mul2(q0[0], dn), mul2(q0[1], dn));
    const uint32_t lo1 = e4m3x4(mul2(q0[2], dn), mul2(q0[3], dn));
    const uint32_t hi0 = e4m3x4(mul2(q0[0], up), mul2(q0[1], up));
    const uint32_t hi1 = e4m3x4(mul2(q0[2], up), mul2(q0[3], up));
    if (((lo0 ^ hi0) | (lo1 ^ hi1)) == 0) return make_uint2(lo0, lo1);
    f2 qd[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        qd[i] = f2_make(__fdiv_rn(f2_lo(n[i]), s), __fdiv_rn(f2_hi(n[i]), s));
    return make_uint2(e4m3x4(qd[0], qd[1]), e4m3x4(qd[2], qd[3]));
}

// MAXT / MINB: the launch bound (8 consumer warps + producer at 3 CTAs per SM, 72 registers
// per thread; or 16 + producer at one CTA per SM for long rows, 120 registers).
template <int NCH, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) fused_add_rmsnorm_fp8_kernel(FusedArgs a) {
    constexpr int VEC = 8;
    extern __shared__ __align__(128) uint8_t smem[];
    const Ring ring = ring_at(smem, a.stages, a.stage_bytes, a.data_off);
    const uint8_t* wsm = smem + kRingHeader;
    const int nw = a.nw;
    const int64_t G = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t nrows = (a.T - 1 - b) / G + 1;  // rows b, b + G, ... below T
    const uint32_t r_off = a.stage_bytes / 2;  // stage = [x row | residual row]
    stage_weights_f32<VEC>(a.w, a.H, smem + kRingHeader);
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
    constexpr int NP = 4;  // FP32 pairs per 16-byte vector of bf16

    Slot at;
    for (int64_t k = 0; k < nrows; ++k, at.advance(ring.stages)) {
        const int64_t row = b + k * G;
        const int64_t base = row * H;
        const bool ok = ring_wait_full(ring, at, a.limit_ns, a.err);
        const uint8_t* st = ring.stage(at.s);
        // h = bf16(x + residual), written back to residual; sum of h^2 in two chains (even
        // and odd elements) added at the end
        uint4 hv[NCH];
        f2 ss2 = f2_splat(0.f);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * NC + t;
            const bool in = ok && v < nvec;
            f2 xp[NP], rp[NP];
            Pairs<__nv_bfloat16>::get(in ? lds128(st + (size_t)v * 16) : make_uint4(0, 0, 0, 0), xp);
            Pairs<__nv_bfloat16>::get(in ? lds128(st + r_off + (size_t)v * 16) : make_uint4(0, 0, 0, 0), rp);
#pragma unroll
            for (int i = 0; i < NP; ++i) rp[i] = add2(xp[i], rp[i]);
            hv[c] = Pairs<__nv_bfloat16>::put(rp);  // h rounded once to bf16
            if (in) st_stream(a.res + base + (int64_t)v * VEC, hv[c]);
            Pairs<__nv_bfloat16>::get(hv[c], rp);
#pragma unroll
            for (int i = 0; i < NP; ++i) ss2 = fma2(rp[i], rp[i], ss2);
        }
        if (__all_sync(0xffffffffu, ok)) ring_release(ring, at);
        float ss = __fadd_rn(f2_lo(ss2), f2_hi(ss2));
        if (!consumer_sum<(MAXT > 288 ? 16 : 8)>(smem, ss, ok, nw, (int)(k & 1))) break;
        const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, Hf), a.eps)));
        const f2 rs2 = f2_splat(rs);

#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * NC + t;
            const bool in = v < nvec;  // uniform over each 16-lane block (H % 128 == 0)
            f2 np_[NP], wp[NP];
            Pairs<__nv_bfloat16>::get(hv[c], np_);
            if (in) {
                w_pairs<NP>(wsm, nvec, v, wp);
            } else {
#pragma unroll
                for (int i = 0; i < NP; ++i) wp[i] = f2_splat(0.f);
            }
#pragma unroll
            for (int i = 0; i < NP; ++i) np_[i] = mul2(mul2(np_[i], rs2), wp[i]);
            const uint4 nv = Pairs<__nv_bfloat16>::put(np_);
            if (in) st_stream(a.normed + base + (int64_t)v * VEC, nv);
            Pairs<__nv_bfloat16>::get(nv, np_);  // the bf16-rounded normed values

            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < NP; ++i)
                amax = fmaxf(amax, fmaxf(fabsf(f2_lo(np_[i])), fabsf(f2_hi(np_[i]))));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float scale = scale_of(amax);
            if (in && (t & 15) == 0) a.scale[(int64_t)(v >> 4) * a.ld + row] = scale;

            uint2 codes;
            if (amax >= 0x1p-100f && amax <= 0x1.fep127f) {
                codes = quotient_codes(np_, recip_of(scale), scale);
            } else if (scale > 0.f) {  // tiny or infinite amax: the IEEE division
                f2 qd[NP];
#pragma unroll
                for (int i = 0; i < NP; ++i)
                    qd[i] = f2_make(__fdiv_rn(f2_lo(np_[i]), scale), __fdiv_rn(f2_hi(np_[i]), scale));
                codes = make_uint2(e4m3x4(qd[0], qd[1]), e4m3x4(qd[2], qd[3]));
            } else {  // amax == 0: the signed zero of each element
                codes = make_uint2(e4m3x4(np_[0], np_[1]), e4m3x4(np_[2], np_[3]));
            }
            if (in) __stcs(reinterpret_cast<uint2*>(a.q + base + (int64_t)v * VEC), codes);
        }
    }
}

template <int NCH, int MAXT = 288, int MINB = 3>
static cudaError_t run(const Launch& L, const FusedArgs& a, cudaStream_t s) {
    auto k = fused_add_rmsnorm_fp8_kernel<NCH, MAXT, MINB>;
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
    if (L.nw > 8) {  // 16 consumer warps: rows of 1024-2048 vectors
        switch (L.nch) {
            case 2: return run<2, 544, 1>(L, a, s);
            case 3: return run<3, 544, 1>(L, a, s);
            case 4: return run<4, 544, 1>(L, a, s);
            default: return cudaErrorInvalidConfiguration;
        }
    }
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
