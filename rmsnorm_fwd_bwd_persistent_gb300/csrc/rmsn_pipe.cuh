// rmsn_pipe.cuh -- the shared-memory row ring that feeds every kernel (sm_90+ PTX:
// mbarrier, cp.async.bulk).
//
// One producer thread per CTA streams whole rows from HBM into an S-stage ring of shared
// memory with 1-D bulk copies (the TMA engine), each stage guarded by two mbarriers:
//   full[s]   completes when the copies of the row in stage s have landed
//             (arrive.expect_tx by the producer + complete_tx by the copy engine);
//   empty[s]  completes when every consumer warp has taken the row out of stage s
//             (one arrive per consumer warp), so the producer may refill it.
// The bytes in flight are set by the ring depth, not by registers or warp count.
//
// Every wait is bounded in time.  A wait that runs out sets a bit in the caller's error
// word and the kernel leaves its row loop; before the CTA exits, the producer waits
// (again bounded) for the copies it issued.  No wait spins forever and nothing traps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

enum : unsigned {
    ERR_WAIT_FULL = 1u,   // a consumer waited too long for a row to land
    ERR_WAIT_EMPTY = 2u,  // the producer waited too long for a stage to be released
    ERR_WAIT_DRAIN = 4u,  // copies still in flight when the CTA gave up
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase of `bar` with parity `parity` to complete.  Gives up (returns
// false) after `limit_ns` of %globaltimer time or after kMaxPolls polls, whichever comes
// first, so the wait ends even if the timer does not advance.  Polls after the first few
// back off with __nanosleep.
constexpr uint32_t kMaxPolls = 1u << 22;

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 1; n < kMaxPolls; ++n) {
        if (mbar_test(bar, parity)) return true;
        if (n > 64) __nanosleep(256);
        if (global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// 1-D bulk copy global -> shared of `bytes` (multiple of 16, both addresses 16-byte
// aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Copies the H weights into shared memory as FP32 (bf16 weights are widened exactly), all
// threads of the CTA cooperating; made visible by the __syncthreads in ring_init.
// Layout for a row split into 16-byte vectors of VEC elements: P = VEC / 4 planes of
// 16-byte slots; slot (plane q, vector v) at float4 index q * (H / VEC) + v holds weights
// v*VEC + 4q .. v*VEC + 4q + 3, so consecutive lanes read consecutive 16-byte slots.
template <int VEC>
__device__ __forceinline__ void stage_weights_f32(const float* w, int H, uint8_t* dst) {
    constexpr int P = VEC / 4;
    const int nvec = H / VEC;
    const float4* src = reinterpret_cast<const float4*>(w);
    float4* d = reinterpret_cast<float4*>(dst);
    for (int g = threadIdx.x; g < H / 4; g += blockDim.x) d[(g % P) * nvec + g / P] = __ldg(src + g);
}
template <int VEC>
__device__ __forceinline__ void stage_weights_f32(const __nv_bfloat16* w, int H, uint8_t* dst) {
    constexpr int P = VEC / 4;
    const int nvec = H / VEC;
    const uint2* src = reinterpret_cast<const uint2*>(w);
    float4* d = reinterpret_cast<float4*>(dst);
    for (int g = threadIdx.x; g < H / 4; g += blockDim.x) {
        const uint2 u = __ldg(src + g);
        d[(g % P) * nvec + g / P] =
            make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                        __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    }
}

// Ring bookkeeping shared by the kernels: `stages` stages of `stage_bytes` each, placed
// after the barrier block at the start of dynamic shared memory.
struct Ring {
    uint64_t* full;
    uint64_t* empty;
    uint8_t* data;
    int stages;
    uint32_t stage_bytes;

    __device__ __forceinline__ uint8_t* stage(int s) const { return data + (size_t)s * stage_bytes; }
};

// Dynamic shared memory layout: [full[S] | empty[S] | reduce slots (2 x 32 floats) |
// abort flags (2 x 32 ints)] (kRingHeader bytes) [weights, padded to 128] [S stages].
constexpr int kRingHeader = 1024;  // bytes reserved before the weights (S <= 32)

__device__ __forceinline__ Ring ring_at(uint8_t* smem, int stages, uint32_t stage_bytes,
                                        uint32_t data_offset) {
    Ring r;
    r.full = reinterpret_cast<uint64_t*>(smem);
    r.empty = r.full + 32;
    r.data = smem + data_offset;
    r.stages = stages;
    r.stage_bytes = stage_bytes;
    return r;
}

__device__ __forceinline__ float* ring_red(uint8_t* smem) {
    return reinterpret_cast<float*>(smem + 512);  // [2][32] per-warp partial sums
}
__device__ __forceinline__ int* ring_abort(uint8_t* smem) {
    return reinterpret_cast<int*>(smem + 768);    // [2][32] per-warp "gave up" flags
}

// Initializes the barriers (thread 0) and makes them visible to the CTA.
__device__ __forceinline__ void ring_init(const Ring& r, int consumer_warps) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < r.stages; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], consumer_warps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
}

// The producer loop (one thread).  `issue(k, stage_ptr, full_bar)` issues the bulk copies
// of the CTA's k-th row and returns their total byte count after arming the barrier.
// Returns the number of rows issued.
template <typename Issue>
__device__ __forceinline__ int64_t ring_produce(const Ring& r, int64_t nrows, uint64_t limit_ns,
                                                unsigned* err, Issue issue) {
    int64_t k = 0;
    for (; k < nrows; ++k) {
        const int s = (int)(k % r.stages);
        if (k >= r.stages) {
            const uint32_t par = (uint32_t)(((k / r.stages) & 1) ^ 1);
            if (!mbar_wait(&r.empty[s], par, limit_ns)) {
                atomicOr(err, ERR_WAIT_EMPTY);
                break;
            }
        }
        issue(k, r.stage(s), &r.full[s]);
    }
    return k;
}

// After the producer stops (normally or not): every copy it issued must land before the
// CTA may exit.  Waits on the last `stages` full barriers it armed.
__device__ __forceinline__ void ring_drain(const Ring& r, int64_t issued, uint64_t limit_ns,
                                           unsigned* err) {
    const int64_t first = issued > r.stages ? issued - r.stages : 0;
    for (int64_t k = first; k < issued; ++k) {
        const int s = (int)(k % r.stages);
        if (!mbar_wait(&r.full[s], (uint32_t)((k / r.stages) & 1), limit_ns)) {
            atomicOr(err, ERR_WAIT_DRAIN);
            return;
        }
    }
}

// Consumer side: wait for row k's stage.  The decision to go on is taken together by
// all consumer warps at the next named barrier (see consumer_sync), so a warp that gave
// up never leaves the others waiting at a barrier.
__device__ __forceinline__ bool ring_wait_full(const Ring& r, int64_t k, uint64_t limit_ns,
                                               unsigned* err) {
    const int s = (int)(k % r.stages);
    if (mbar_wait(&r.full[s], (uint32_t)((k / r.stages) & 1), limit_ns)) return true;
    atomicOr(err, ERR_WAIT_FULL);
    return false;
}

__device__ __forceinline__ void ring_release(const Ring& r, int64_t k) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[(int)(k % r.stages)]);
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Row-wide sum over the consumer warps (warps 0 .. nw-1), combined with the "keep going"
// vote: every consumer warp posts its warp sum and whether its wait succeeded, one named
// barrier, then every lane adds the posts in warp order (same bits on every lane).
// Returns false if any consumer warp gave up on this row.
__device__ __forceinline__ bool consumer_sum(uint8_t* smem, float& v, bool ok, int nw,
                                             int parity) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    float* red = ring_red(smem) + parity * 32;
    int* ab = ring_abort(smem) + parity * 32;
    const int warp = threadIdx.x >> 5;
    const bool warp_ok = __all_sync(0xffffffffu, ok);
    if ((threadIdx.x & 31) == 0) {
        red[warp] = v;
        ab[warp] = warp_ok ? 0 : 1;
    }
    named_bar(1, nw * 32);
    float s = red[0];
    int bad = ab[0];
    for (int k = 1; k < nw; ++k) {
        s += red[k];
        bad |= ab[k];
    }
    v = s;
    return bad == 0;
}

}  // namespace rmsn
