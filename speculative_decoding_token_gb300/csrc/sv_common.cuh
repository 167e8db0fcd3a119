// sv_common.cuh -- device-side building blocks of the verify-step kernels.
//
// Counter-based uniforms (Philox4x32-10, Salmon et al., "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11), float-float arithmetic (Knuth's
// TwoSum, FMA-based exact products) and packed f32x2 helpers. The table-driven
// float-float exponential of the draw (P. T. P. Tang, "Table-driven
// implementation of the exponential function in IEEE floating-point
// arithmetic", ACM TOMS 15(2), 1989) lives in sv_draw.cu.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "sv_internal.h"

namespace sv {

// ---------------------------------------------------------------------------
// Philox4x32-10: ten rounds of two 32x32->64 multiplies, xor of the high
// halves into the odd counter words with the round key, and a word
// permutation; the key advances by the two Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x;
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

__device__ __forceinline__ uint4 seeded_block(uint64_t seed, uint32_t b, uint32_t i,
                                              uint32_t purpose) {
    return philox4x32_10(make_uint4(b, i, purpose, 0u),
                         make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}

// accept-test uniform of sequence b at 1-based position i: (2*(w>>9)+1)*2^-24,
// an odd multiple of 2^-24 below 1 and so exact in float
__device__ __forceinline__ float accept_uniform(uint64_t seed, uint32_t b, uint32_t i) {
    const uint32_t w = seeded_block(seed, b, i, 0u).x;
    return (float)(2u * (w >> 9) + 1u) * 0x1p-24f;
}

// final-draw uniform at 1-based position i: (2*k+1)*2^-53, k = (w0<<20)|(w1>>12)
__device__ __forceinline__ double draw_uniform(uint64_t seed, uint32_t b, uint32_t i) {
    const uint4 w = seeded_block(seed, b, i, 1u);
    const uint64_t k = ((uint64_t)w.x << 20) | (uint64_t)(w.y >> 12);
    return (double)(2ull * k + 1ull) * 0x1p-53;
}

// ---------------------------------------------------------------------------
// float-float helpers. A pair (h, l) stands for the unevaluated sum h + l.

// ln 2 split into a float head and a float tail
constexpr float kLn2Hi = 0.693147182464599609375f;
constexpr float kLn2Lo = -1.904654323148236017e-09f;

// s + e = a + b exactly (Knuth TwoSum)
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// acc += (xh, xl), keeping the rounding error of the head addition
__device__ __forceinline__ void ff_accumulate(float &ah, float &al, float xh, float xl) {
    float s, e;
    two_sum(ah, xh, s, e);
    ah = s;
    al += xl + e;
}

// (ah, al) + (bh, bl), renormalised
__device__ __forceinline__ void ff_add(float ah, float al, float bh, float bl, float &rh,
                                       float &rl) {
    float s, e;
    two_sum(ah, bh, s, e);
    e += al + bl;
    rh = s + e;
    rl = e - (rh - s);
}

// (ah, al) * (bh, bl), renormalised (the head product's error from an FMA)
__device__ __forceinline__ void ff_mul(float ah, float al, float bh, float bl, float &rh,
                                       float &rl) {
    const float p = ah * bh;
    float e = fmaf(ah, bh, -p);
    e = fmaf(ah, bl, e);
    e = fmaf(al, bh, e);
    rh = p + e;
    rl = e - (rh - p);
}

// (ah, al) / (bh, bl): the float quotient and one correction from its remainder
__device__ __forceinline__ void ff_div(float ah, float al, float bh, float bl, float &rh,
                                       float &rl) {
    const float q1 = ah / bh;
    float ph, pl, dh, dl;
    ff_mul(q1, 0.0f, bh, bl, ph, pl);
    ff_add(ah, al, -ph, -pl, dh, dl);
    const float q2 = dh / bh;
    two_sum(q1, q2, rh, rl);
}

__device__ __forceinline__ double ff_to_double(float h, float l) {
    return (double)h + (double)l;
}

// the final-draw uniform (2k+1) 2^-53 as a float-float: the top 24 bits of
// the odd integer m = 2k+1 exactly, its other 29 bits rounded to 24
__device__ __forceinline__ void draw_uniform_ff(uint64_t seed, uint32_t b, uint32_t i, float &uh,
                                                float &ul) {
    const uint4 w = seeded_block(seed, b, i, 1u);
    const uint64_t k = ((uint64_t)w.x << 20) | (uint64_t)(w.y >> 12);
    const uint64_t m = 2ull * k + 1ull;
    const float hi = (float)(uint32_t)(m >> 29) * 0x1p-24f;
    const float lo = (float)(uint32_t)(m & ((1ull << 29) - 1ull)) * 0x1p-53f;
    two_sum(hi, lo, uh, ul);
}

// ---------------------------------------------------------------------------
// bf16 <-> fp32 (bf16 is the top half of a binary32)
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int DT>
__device__ __forceinline__ float load_logit(const char *row, int64_t v) {
    if (DT == SV_DT_FP32) return __ldg(reinterpret_cast<const float *>(row) + v);
    const uint16_t h = __ldg(reinterpret_cast<const unsigned short *>(row) + v);
    return __uint_as_float((uint32_t)h << 16);
}

// NaN-propagating max (a NaN input yields NaN)
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// packed pairs of floats for the f32x2 arithmetic of sm_100-class GPUs
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 unpack2(f32x2 v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return make_float2(lo, hi);
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---------------------------------------------------------------------------
// memory-model helpers for data handed between warps of one launch

// relaxed 64-bit store / load at GPU scope: single-copy atomic, no fence
__device__ __forceinline__ void st_relaxed_f2(float2 *p, float2 v) {
    const unsigned long long bits =
        ((unsigned long long)__float_as_uint(v.y) << 32) | __float_as_uint(v.x);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(bits) : "memory");
}

__device__ __forceinline__ float2 ld_relaxed_f2(const float2 *p) {
    unsigned long long bits;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(bits) : "l"(p) : "memory");
    return make_float2(__uint_as_float((uint32_t)bits), __uint_as_float((uint32_t)(bits >> 32)));
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

}  // namespace sv
