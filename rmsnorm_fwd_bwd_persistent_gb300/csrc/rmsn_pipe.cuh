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

// One poll of the phase with parity `parity`.  While the phase is incomplete the thread
// may be suspended for up to kSuspendNs (it resumes as soon as the phase completes), so a
// waiting warp takes few issue slots.
constexpr uint32_t kSuspendNs = 20000;

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "n"(kSuspendNs)
        : "memory");
    return done != 0;
}

// Waits for the phase of `bar` with parity `parity` to complete.  Gives up (returns
// false) after `limit_ns` of %globaltimer time or after kMaxPolls polls (each suspends for
// at most kSuspendNs), whichever comes first, so the wait ends even if the timer does not
// advance.  Polls after the first few back off with __nanosleep.
constexpr uint32_t kMaxPolls = 1u << 16;

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

// Prefetch `bytes` (multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 16-byte global load that is not kept in L1 (read once).
__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
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

// Position of the k-th row in the ring: stage s = k mod S and the parity ph = (k div S) mod 2
// of that stage's current phase, advanced row by row (no division in the row loops).
struct Slot {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void advance(int stages) {
        if (++s == stages) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Dynamic shared memory layout (kRingHeader bytes of bookkeeping, then the weights padded
// to 128 bytes, then the stages):
//   [0, 256)      full[32]      mbarriers, one per stage
//   [256, 512)    empty[32]     mbarriers, one per stage
//   [512, 768)    red[2][32]    per-warp partial sums (one value per row)
//   [768, 832)    abort[2][32]  per-warp "gave up" flags, one byte each
//   [1024, 1536)  red2[2][32]   per-warp partial sums (two values, two rows at a time)
constexpr int kRingHeader = 2048;  // bytes reserved before the weights (S <= 32)

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
__device__ __forceinline__ uint8_t* ring_abort(uint8_t* smem) {
    return smem + 768;                              // [2][32] per-warp "gave up" bytes
}
__device__ __forceinline__ float2* ring_red2(uint8_t* smem) {
    return reinterpret_cast<float2*>(smem + 1024);  // [2][32] per-warp partial sum pairs
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
    Slot at;
    for (; k < nrows; ++k, at.advance(r.stages)) {
        // a stage is refilled once every consumer warp has released its previous row
        if (k >= r.stages && !mbar_wait(&r.empty[at.s], at.ph ^ 1u, limit_ns)) {
            atomicOr(err, ERR_WAIT_EMPTY);
            break;
        }
        issue(k, r.stage(at.s), &r.full[at.s]);
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

// Consumer side: wait for the row in stage `at`.  The decision to go on is taken together
// by all consumer warps at the next named barrier (consumer_sum), so a warp that gave up
// never leaves the others waiting at a barrier.
__device__ __forceinline__ bool ring_wait_full(const Ring& r, const Slot& at, uint64_t limit_ns,
                                               unsigned* err) {
    if (mbar_wait(&r.full[at.s], at.ph, limit_ns)) return true;
    atomicOr(err, ERR_WAIT_FULL);
    return false;
}

__device__ __forceinline__ void ring_release(const Ring& r, const Slot& at) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[at.s]);
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// True if any of the first nw (1 .. 16) "gave up" bytes at f (16-byte aligned) is set.
__device__ __forceinline__ bool any_gave_up(const uint8_t* f, int nw) {
    const uint64_t* w = reinterpret_cast<const uint64_t*>(f);
    auto bytes = [](int n) { return n >= 8 ? ~0ull : ((1ull << (8 * n)) - 1ull); };
    if (nw <= 8) return (w[0] & bytes(nw)) != 0;
    return (w[0] | (w[1] & bytes(nw - 8))) != 0;
}

// r[0] + r[1] + ... + r[nw-1], left to right, for nw in {1, 2, 4, 8} and, when MAXW is
// 16, also 16 (r 16-byte aligned).
template <int MAXW = 8>
__device__ __forceinline__ float sum_posts(const float* r, int nw) {
    if (nw >= 4) {
        const float4 a = *reinterpret_cast<const float4*>(r);
        float s = a.x + a.y + a.z + a.w;
        if (nw == 8 || (MAXW >= 16 && nw == 16)) {
            const float4 b = *reinterpret_cast<const float4*>(r + 4);
            s = s + b.x + b.y + b.z + b.w;
        }
        if constexpr (MAXW >= 16) {
            if (nw == 16) {
                const float4 c = *reinterpret_cast<const float4*>(r + 8);
                const float4 d = *reinterpret_cast<const float4*>(r + 12);
                s = s + c.x + c.y + c.z + c.w + d.x + d.y + d.z + d.w;
            }
        }
        return s;
    }
    return nw == 2 ? r[0] + r[1] : r[0];
}

// Row-wide sum over the consumer warps (warps 0 .. nw-1), combined with the "keep going"
// vote: every consumer warp reduces its value by a butterfly of shuffles and posts it with
// whether its wait succeeded, one named barrier, then every lane adds the posts in warp
// order (same bits on every lane).  Returns false if any consumer warp gave up on this row.
template <int MAXW = 8>
__device__ __forceinline__ bool consumer_sum(uint8_t* smem, float& v, bool ok, int nw,
                                             int parity) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    float* red = ring_red(smem) + parity * 32;
    uint8_t* ab = ring_abort(smem) + parity * 32;
    const int warp = threadIdx.x >> 5;
    const bool warp_ok = __all_sync(0xffffffffu, ok);
    if ((threadIdx.x & 31) == 0) {
        red[warp] = v;
        ab[warp] = warp_ok ? 0 : 1;
    }
    named_bar(1, nw * 32);
    v = sum_posts<MAXW>(red, nw);
    return !any_gave_up(ab, nw);
}

// Two row-wide sums at once (two rows share one barrier).  The first shuffle pairs the
// lanes so that even lanes go on with v0 and odd lanes with v1; four more butterfly levels
// among lanes of the same parity finish both warp sums (lane 0 holds v0's, lane 1 v1's).
// Each warp posts its sums times m0 and m1 (rounded), and the posts are added in warp
// order.  The order is fixed, so the bits depend only on the data.  nw is 1 .. 16 (the
// powers of two read the posts as float4s; the order is the same either way).
__device__ __forceinline__ bool consumer_sum2(uint8_t* smem, float& v0, float& v1, float m0,
                                              float m1, bool ok, int nw, int parity) {
    const int lane = threadIdx.x & 31;
    const bool odd = (lane & 1) != 0;
    float mine = odd ? v1 : v0;
    mine += __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
#pragma unroll
    for (int o = 16; o > 1; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    float* red = reinterpret_cast<float*>(ring_red2(smem) + parity * 32);
    uint8_t* ab = ring_abort(smem) + parity * 32;
    const int warp = threadIdx.x >> 5;
    const bool warp_ok = __all_sync(0xffffffffu, ok);
    if (lane < 2) red[2 * warp + lane] = __fmul_rn(mine, odd ? m1 : m0);
    if (lane == 0) ab[warp] = warp_ok ? 0 : 1;
    named_bar(1, nw * 32);
    const float4* r4 = reinterpret_cast<const float4*>(red);
    float s0, s1;
    if (nw == 16) {
        const float4 q0 = r4[0];
        s0 = q0.x + q0.z;
        s1 = q0.y + q0.w;
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            const float4 q = r4[i];
            s0 = s0 + q.x + q.z;
            s1 = s1 + q.y + q.w;
        }
    } else if (nw == 8) {
        const float4 a = r4[0], b = r4[1], c = r4[2], d = r4[3];
        s0 = a.x + a.z + b.x + b.z + c.x + c.z + d.x + d.z;
        s1 = a.y + a.w + b.y + b.w + c.y + c.w + d.y + d.w;
    } else if (nw == 4) {
        const float4 a = r4[0], b = r4[1];
        s0 = a.x + a.z + b.x + b.z;
        s1 = a.y + a.w + b.y + b.w;
    } else if (nw == 2) {
        const float4 a = r4[0];
        s0 = a.x + a.z;
        s1 = a.y + a.w;
    } else {
        s0 = red[0];
        s1 = red[1];
        for (int i = 1; i < nw; ++i) {
            s0 = s0 + red[2 * i];
            s1 = s1 + red[2 * i + 1];
        }
    }
    v0 = s0;
    v1 = s1;
    return !any_gave_up(ab, nw);
}

}  // namespace rmsn
