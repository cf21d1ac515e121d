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

// ------------------------------------------------------------------ paired FP32 arithmetic
// Blackwell executes two IEEE binary32 operations per instruction on a 64-bit register
// pair (mul/fma/add/sub .rn.f32x2).  Each half is rounded exactly as the scalar operation
// would be, so the results are bit-identical to __fmul_rn / fmaf / __fadd_rn / __fsub_rn
// element by element; only the instruction count halves.  A pair holds (even, odd)
// elements in (low, high) halves.
using f2 = uint64_t;

__device__ __forceinline__ f2 f2_make(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ f2 f2_splat(float v) { return f2_make(v, v); }
__device__ __forceinline__ float f2_lo(f2 v) {
    float lo;
    asm("{\n\t.reg .f32 t;\n\tmov.b64 {%0, t}, %1;\n\t}" : "=f"(lo) : "l"(v));
    return lo;
}
__device__ __forceinline__ float f2_hi(f2 v) {
    float hi;
    asm("{\n\t.reg .f32 t;\n\tmov.b64 {t, %0}, %1;\n\t}" : "=f"(hi) : "l"(v));
    return hi;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// A 16-byte vector of x as FP32 pairs (NP pairs) and back (one rounding to x's type).
template <typename T>
struct Pairs;

template <>
struct Pairs<float> {
    static constexpr int NP = 2;
    __device__ __forceinline__ static void get(const uint4& v, f2 (&p)[2]) {
        p[0] = f2_make(__uint_as_float(v.x), __uint_as_float(v.y));
        p[1] = f2_make(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    __device__ __forceinline__ static uint4 put(const f2 (&p)[2]) {
        return make_uint4(__float_as_uint(f2_lo(p[0])), __float_as_uint(f2_hi(p[0])),
                          __float_as_uint(f2_lo(p[1])), __float_as_uint(f2_hi(p[1])));
    }
    // elementwise products a * b, rounded to FP32
    __device__ __forceinline__ static void prod(const uint4& a, const uint4& b, f2 (&p)[2]) {
        f2 x[2], y[2];
        get(a, x);
        get(b, y);
        p[0] = mul2(x[0], y[0]);
        p[1] = mul2(x[1], y[1]);
    }
};

template <>
struct Pairs<__nv_bfloat16> {
    static constexpr int NP = 4;
    __device__ __forceinline__ static f2 word(uint32_t u) { return f2_make(bf16_lo(u), bf16_hi(u)); }
    __device__ __forceinline__ static void get(const uint4& v, f2 (&p)[4]) {
        p[0] = word(v.x);
        p[1] = word(v.y);
        p[2] = word(v.z);
        p[3] = word(v.w);
    }
    __device__ __forceinline__ static uint32_t round_word(f2 v) {
        return pack_bf16x2(f2_lo(v), f2_hi(v));
    }
    __device__ __forceinline__ static uint4 put(const f2 (&p)[4]) {
        return make_uint4(round_word(p[0]), round_word(p[1]), round_word(p[2]), round_word(p[3]));
    }
    // Elementwise products of two words of bf16 pairs, each by one mixed-precision FMA
    // (bf16 operands, FP32 addend +0 and result).  A product of two bf16 values has at most
    // 16 significant bits, so it is exact in FP32 unless it leaves FP32's normal range.
    __device__ __forceinline__ static f2 word_prod(uint32_t a, uint32_t b) {
        float lo, hi;
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
            "mov.b32 {a0, a1}, %2;\n\t"
            "mov.b32 {b0, b1}, %3;\n\t"
            "fma.rn.f32.bf16 %0, a0, b0, 0f00000000;\n\t"
            "fma.rn.f32.bf16 %1, a1, b1, 0f00000000;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(a), "r"(b));
        return f2_make(lo, hi);
    }
    __device__ __forceinline__ static void prod(const uint4& a, const uint4& b, f2 (&p)[4]) {
        p[0] = word_prod(a.x, b.x);
        p[1] = word_prod(a.y, b.y);
        p[2] = word_prod(a.z, b.z);
        p[3] = word_prod(a.w, b.w);
    }
};

// The weights beside 16-byte vector v of x as FP32 pairs, read from the planar FP32 copy
// of w in shared memory (stage_weights_f32): plane q holds pairs 2q and 2q+1 of every
// vector at byte offset (q * nvec + v) * 16.
template <int NP>
__device__ __forceinline__ void w_pairs(const uint8_t* wsm, int nvec, int v, f2 (&p)[NP]) {
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(wsm);
#pragma unroll
    for (int q = 0; q < NP / 2; ++q)
        asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];"
                     : "=l"(p[2 * q]), "=l"(p[2 * q + 1])
                     : "r"(base + (uint32_t)(q * nvec + v) * 16));
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

// TwoSum on both halves of a pair: s + e == a + b exactly, per half.
__device__ __forceinline__ void two_sum2(f2 a, f2 b, f2& s, f2& e) {
    s = add2(a, b);
    const f2 bb = sub2(s, a);
    e = add2(sub2(a, sub2(s, bb)), sub2(b, bb));
}

// (hi, lo) += v on both halves
__device__ __forceinline__ void comp_add2(f2& hi, f2& lo, f2 v) {
    f2 s, e;
    two_sum2(hi, v, s, e);
    hi = s;
    lo = add2(lo, e);
}

}  // namespace rmsn
