// rmsn_device.cuh -- device helpers shared by the RMSNorm kernels (sm_103a).
//
// Row geometry used by every kernel: a "row group" of G = 32 * wpr consecutive threads
// owns one row at a time.  The row is split into 16-byte vectors; lane l of the group
// holds vectors v = c * G + l for c = 0 .. NCH-1 (NCH is a compile-time count, vectors
// past the end of the row are masked), so one warp-wide access touches 512 contiguous
// bytes and every load is a coalesced 16-byte access.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

// ------------------------------------------------------------------ element traits
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int VEC = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// two floats -> packed bf16x2 (round to nearest even), a in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int VEC = 8;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                          pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    }
};

// ------------------------------------------------------------------ memory access
// Streamed operands (read or written once per call): evict-first cache policy.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// The weight is re-read by every row: read-only path, default (L1-resident) policy.
// Loads the VEC weights that sit beside a 16-byte vector of x (VEC = 16 / sizeof(x)).
template <typename TW, int VEC>
__device__ __forceinline__ void load_w(const TW* w, int64_t col0, float (&f)[VEC]);

template <>
__device__ __forceinline__ void load_w<float, 4>(const float* w, int64_t col0, float (&f)[4]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(w + col0));
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
}
template <>
__device__ __forceinline__ void load_w<float, 8>(const float* w, int64_t col0, float (&f)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(w + col0));
    float4 b = __ldg(reinterpret_cast<const float4*>(w + col0 + 4));
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
template <>
__device__ __forceinline__ void load_w<__nv_bfloat16, 8>(const __nv_bfloat16* w, int64_t col0,
                                                         float (&f)[8]) {
    uint4 a = __ldg(reinterpret_cast<const uint4*>(w + col0));
    Elem<__nv_bfloat16>::unpack(a, f);
}
template <>
__device__ __forceinline__ void load_w<__nv_bfloat16, 4>(const __nv_bfloat16* w, int64_t col0,
                                                         float (&f)[4]) {
    uint2 a = __ldg(reinterpret_cast<const uint2*>(w + col0));
    f[0] = bf16_lo(a.x); f[1] = bf16_hi(a.x);
    f[2] = bf16_lo(a.y); f[3] = bf16_hi(a.y);
}

// ------------------------------------------------------------------ reductions
// Butterfly sum over a warp.  IEEE addition is commutative, so every lane ends with the
// same bits.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Sum over the wpr warps of one row group.  `red` is a shared array of 2 * (CTA warps)
// floats; `parity` alternates per row so that a warp that moves on to the next row never
// overwrites a slot another warp of its group has not read yet.  Groups synchronize on
// their own named barrier (id 1 + group), never on the CTA barrier.  The warp sums are
// added in warp order, so the result is the same on every lane of the group.
__device__ __forceinline__ float group_sum(float v, int wpr, float* red, int group, int parity) {
    v = warp_sum(v);
    if (wpr == 1) return v;
    const int warp = threadIdx.x >> 5;
    float* slot = red + parity * (blockDim.x >> 5) + group * wpr;
    if ((threadIdx.x & 31) == 0) red[parity * (blockDim.x >> 5) + warp] = v;
    named_barrier(1 + group, 32 * wpr);
    float s = slot[0];
    for (int k = 1; k < wpr; ++k) s += slot[k];
    return s;
}

// ------------------------------------------------------------------ compensated sums
// Error-free transformation of a + b (Knuth's TwoSum): s + e == a + b exactly.
// Written with the _rn intrinsics so that the compiler can neither contract nor
// reassociate any step.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) += v
__device__ __forceinline__ void comp_add(float& hi, float& lo, float v) {
    float s, e;
    two_sum(hi, v, s, e);
    hi = s;
    lo = __fadd_rn(lo, e);
}

// (hi, lo) += (h2, l2)
__device__ __forceinline__ void comp_merge(float& hi, float& lo, float h2, float l2) {
    float s, e;
    two_sum(hi, h2, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, l2));
}

}  // namespace rmsn
