// rmsn_device.cuh -- element conversions, register-resident weights and compensated sums
// shared by the RMSNorm kernels (sm_103a).
//
// Row geometry used by every kernel: the NC consumer threads of a CTA share one row at a
// time.  The row is split into 16-byte vectors; consumer thread t holds the vectors
// v = c * NC + t for c = 0 .. NCH-1 (NCH is a compile-time count, vectors past the end of
// the row are masked), so one warp-wide access touches 512 contiguous bytes.
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
// Streamed outputs (written once per call): evict-first cache policy.
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// The weights beside one 16-byte vector v of x, read from the copy of w in shared memory
// (VEC = 16 / sizeof(x) weights of type TW, at byte offset v * VEC * sizeof(TW)).
template <typename TW, int VEC>
struct WSmem;

template <>
struct WSmem<__nv_bfloat16, 8> {
    __device__ __forceinline__ static void get(const uint8_t* w, int v, float (&f)[8]) {
        uint4 u;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                     : "r"((uint32_t)__cvta_generic_to_shared(w + (size_t)v * 16)));
        Elem<__nv_bfloat16>::unpack(u, f);
    }
};
template <>
struct WSmem<__nv_bfloat16, 4> {
    __device__ __forceinline__ static void get(const uint8_t* w, int v, float (&f)[4]) {
        uint32_t a, b;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                     : "=r"(a), "=r"(b)
                     : "r"((uint32_t)__cvta_generic_to_shared(w + (size_t)v * 8)));
        f[0] = bf16_lo(a); f[1] = bf16_hi(a);
        f[2] = bf16_lo(b); f[3] = bf16_hi(b);
    }
};
template <>
struct WSmem<float, 8> {
    __device__ __forceinline__ static void get(const uint8_t* w, int v, float (&f)[8]) {
        const uint32_t addr = (uint32_t)__cvta_generic_to_shared(w + (size_t)v * 32);
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3])
                     : "r"(addr));
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(f[4]), "=f"(f[5]), "=f"(f[6]), "=f"(f[7])
                     : "r"(addr + 16));
    }
};
template <>
struct WSmem<float, 4> {
    __device__ __forceinline__ static void get(const uint8_t* w, int v, float (&f)[4]) {
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3])
                     : "r"((uint32_t)__cvta_generic_to_shared(w + (size_t)v * 16)));
    }
};

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
