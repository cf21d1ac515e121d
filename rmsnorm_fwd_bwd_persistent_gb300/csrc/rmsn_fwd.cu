// rmsn_fwd.cu -- persistent RMSNorm forward (FlashInfer PR #5741 "cake_rmsnorm_train",
// Design/Forward: FP32 sum of squares, two-level shuffle/shared reduce, IEEE rsqrt in
// FP32, one pass that writes y and the FP32 rstd).
//
// CTA b takes the rows b, b + G, b + 2G, ... (G = grid size), so at any moment the whole
// grid streams one window of consecutive rows.  Its producer thread streams those rows
// into a shared-memory ring with bulk copies; the consumer warps take a row out of the
// ring into registers (16-byte vectors, lane-contiguous so every warp access is 512
// contiguous bytes), release the stage, reduce sum(x^2) across the consumer warps, and
// write y straight from registers.  w is copied to shared memory (as FP32) once per CTA.
// The arithmetic runs on FP32 pairs (two IEEE operations per instruction, each rounded as
// its scalar form would be).  x is read from HBM exactly once.
//
// Residual variant (RES; FlashInfer PR #5741 "cake_rmsnorm_train", Design/Forward and API:
// the forward optionally fused with a residual add): the stage holds the x row and the
// residual row, h_new = x + residual is rounded once to x's dtype and written out, and the
// row that is normalized is h_new.
#include "rmsn_device.cuh"
#include "rmsn_internal.h"
#include "rmsn_pipe.cuh"

namespace rmsn {

struct FwdArgs {
    const void* x;
    const void* w;
    void* y;
    float* rstd;
    const void* res;  // residual variant: the residual rows (x's dtype)
    void* h;          // residual variant: h_new = x + residual, rounded to x's dtype
    unsigned* err;
    int64_t T;
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

template <typename TX, typename TW, int NCH, bool RES>
__global__ void __launch_bounds__(288, 3) rmsnorm_fwd_kernel(FwdArgs a) {
    constexpr int VEC = Elem<TX>::VEC;
    extern __shared__ __align__(128) uint8_t smem[];
    const Ring ring = ring_at(smem, a.stages, a.stage_bytes, a.data_off);
    const uint8_t* wsm = smem + kRingHeader;
    const int nw = a.nw;
    const int64_t G = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t nrows = (a.T - 1 - b) / G + 1;  // rows b, b + G, ... below T
    stage_weights_f32<VEC>(static_cast<const TW*>(a.w), a.H, smem + kRingHeader);
    ring_init(ring, nw);

    if ((int)(threadIdx.x >> 5) == nw) {  // producer warp
        if ((threadIdx.x & 31) == 0) {
            const uint8_t* X = static_cast<const uint8_t*>(a.x);
            const int64_t issued = ring_produce(
                ring, nrows, a.limit_ns, a.err, [&](int64_t k, uint8_t* dst, uint64_t* full) {
                    const int64_t off = (b + k * G) * (int64_t)a.row_bytes;
                    if constexpr (RES) {  // stage = [x row | residual row]
                        mbar_arrive_expect_tx(full, 2 * a.row_bytes);
                        bulk_load(dst, X + off, a.row_bytes, full);
                        bulk_load(dst + a.stage_bytes / 2,
                                  static_cast<const uint8_t*>(a.res) + off, a.row_bytes, full);
                    } else {
                        mbar_arrive_expect_tx(full, a.row_bytes);
                        bulk_load(dst, X + off, a.row_bytes, full);
                    }
                });
            ring_drain(ring, issued, a.limit_ns, a.err);
        }
        return;
    }

    const int t = threadIdx.x;
    const int NC = nw * 32;
    const int nvec = a.H / VEC;
    const float Hf = (float)a.H;
    TX* __restrict__ Y = static_cast<TX*>(a.y);

    Slot at;
    for (int64_t k = 0; k < nrows; ++k, at.advance(ring.stages)) {
        const int64_t row = b + k * G;
        const bool ok = ring_wait_full(ring, at, a.limit_ns, a.err);
        const uint8_t* st = ring.stage(at.s);
        uint4 xv[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * NC + t;
            xv[c] = (ok && v < nvec) ? lds128(st + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
            if constexpr (RES) {  // h_new = x + residual, rounded once to x's dtype
                const uint4 rv = (ok && v < nvec) ? lds128(st + a.stage_bytes / 2 + (size_t)v * 16)
                                                  : make_uint4(0, 0, 0, 0);
                f2 hp[Pairs<TX>::NP], rp[Pairs<TX>::NP];
                Pairs<TX>::get(xv[c], hp);
                Pairs<TX>::get(rv, rp);
#pragma unroll
                for (int i = 0; i < Pairs<TX>::NP; ++i) hp[i] = add2(hp[i], rp[i]);
                xv[c] = Pairs<TX>::put(hp);
            }
        }
        if (__all_sync(0xffffffffu, ok)) ring_release(ring, at);
        if constexpr (RES) {
            TX* hr = static_cast<TX*>(a.h) + row * a.H;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const int v = c * NC + t;
                if (ok && v < nvec) st_stream(hr + (int64_t)v * VEC, xv[c]);
            }
        }

        // sum of squares in two chains (even and odd elements), one pair instruction per two
        // elements; the chains are added at the end (a fixed order, same on every run)
        constexpr int NP = Pairs<TX>::NP;
        f2 ss2 = f2_splat(0.f);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            f2 p[NP];
            Pairs<TX>::get(xv[c], p);
#pragma unroll
            for (int i = 0; i < NP; ++i) ss2 = fma2(p[i], p[i], ss2);
        }
        float ss = __fadd_rn(f2_lo(ss2), f2_hi(ss2));
        if (!consumer_sum(smem, ss, ok, nw, (int)(k & 1))) break;
        const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, Hf), a.eps)));
        if (t == 0) a.rstd[row] = rs;

        // y = (x * rstd) * w, two elements per instruction, rounded once to x's type
        const f2 rs2 = f2_splat(rs);
        TX* yr = Y + row * a.H;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int v = c * NC + t;
            if (v < nvec) {
                f2 p[NP], wp[NP];
                Pairs<TX>::get(xv[c], p);
                w_pairs<NP>(wsm, nvec, v, wp);
#pragma unroll
                for (int i = 0; i < NP; ++i) p[i] = mul2(mul2(p[i], rs2), wp[i]);
                st_stream(yr + (int64_t)v * VEC, Pairs<TX>::put(p));
            }
        }
    }
}

template <typename TX, typename TW, int NCH>
static cudaError_t run(const Launch& L, const FwdArgs& a, cudaStream_t s) {
    auto k = a.res ? rmsnorm_fwd_kernel<TX, TW, NCH, true> : rmsnorm_fwd_kernel<TX, TW, NCH, false>;
    const int threads = L.nw * 32 + 32;
    int64_t grid = 0;
    cudaError_t e = fit_grid((const void*)k, L, threads, &grid);
    if (e != cudaSuccess) return e;
    k<<<(unsigned)grid, threads, (size_t)L.smem, s>>>(a);
    return cudaGetLastError();
}

template <typename TX, typename TW>
static cudaError_t dispatch(const Launch& L, const FwdArgs& a, cudaStream_t s) {
    switch (L.nch) {
        case 1: return run<TX, TW, 1>(L, a, s);
        case 2: return run<TX, TW, 2>(L, a, s);
        case 3: return run<TX, TW, 3>(L, a, s);
        case 4: return run<TX, TW, 4>(L, a, s);
        case 6: return run<TX, TW, 6>(L, a, s);
        case 8: return run<TX, TW, 8>(L, a, s);
        case 16: return run<TX, TW, 16>(L, a, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

cudaError_t launch_fwd(const Launch& L, const void* x, int x_dt, const void* w, int w_dt,
                       void* y, float* rstd, int64_t T, int64_t H, float eps, cudaStream_t s,
                       const void* residual, void* h_new) {
    FwdArgs a{x, w, y, rstd, residual, h_new, L.err, T, L.limit_ns, (int)H, L.nw, L.stages,
              L.row_bytes, L.stage_bytes, L.w_bytes, L.data_off, eps};
    if (x_dt == 1 && w_dt == 1) return dispatch<__nv_bfloat16, __nv_bfloat16>(L, a, s);
    if (x_dt == 1 && w_dt == 0) return dispatch<__nv_bfloat16, float>(L, a, s);
    if (x_dt == 0 && w_dt == 0) return dispatch<float, float>(L, a, s);
    if (x_dt == 0 && w_dt == 1) return dispatch<float, __nv_bfloat16>(L, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
