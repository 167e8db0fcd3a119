// sv_common.cuh -- device-side building blocks of the verify-step kernels.
//
// Counter-based uniforms (Philox4x32-10, Salmon et al., "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11), float-float arithmetic (Knuth's
// TwoSum, Dekker's Fast2Sum, FMA-based exact products) and a table-driven
// base-2 exponential in float-float precision (P. T. P. Tang, "Table-driven
// implementation of the exponential function in IEEE floating-point
// arithmetic", ACM TOMS 15(2), 1989): reduce y = k/256 + f with |f| <= 1/512,
// read 2^(j/256) from a 256-entry float-float table and evaluate 2^f - 1 by a
// short Taylor polynomial of (f ln 2).
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

// accept-test uniform of sequence b at 1-based position i: (2*(w>>9)+1)*2^-24
__device__ __forceinline__ double accept_uniform(uint64_t seed, uint32_t b, uint32_t i) {
    const uint32_t w = seeded_block(seed, b, i, 0u).x;
    return (double)(2u * (w >> 9) + 1u) * 0x1p-24;
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

__device__ __forceinline__ double ff_to_double(float h, float l) {
    return (double)h + (double)l;
}

// y = (l - M) * c as a float-float, c = (ch, cl); exact difference by TwoSum
__device__ __forceinline__ void scaled_gap(float l, float M, float ch, float cl, float &yh,
                                           float &yl) {
    float dh, dl;
    two_sum(l, -M, dh, dl);
    yh = dh * ch;
    float e = fmaf(dh, ch, -yh);
    e = fmaf(dh, cl, e);
    yl = fmaf(dl, ch, e);
}

// 2^(yh + yl) for yh <= 0 as a float-float with relative error near 2^-43;
// tab[j] = 2^(j/256) as (head, tail). Results below 2^-125 flush to zero.
__device__ __forceinline__ void ff_exp2(float yh, float yl, const float2 *__restrict__ tab,
                                        float &eh, float &el) {
    const float kf = rintf(yh * 256.0f);
    const float f = fmaf(kf, -0.00390625f, yh);  // exact: |f| <= 1/512
    const int k = (int)kf;
    const int j = k & 255;
    const int i = k >> 8;                        // floor(k / 256)
    // a = (f + yl) ln2 as (ah, al)
    const float ah = f * kLn2Hi;
    float al = fmaf(f, kLn2Hi, -ah);
    al = fmaf(f, kLn2Lo, al);
    al = fmaf(yl, kLn2Hi, al);
    // e^(ah+al) - 1 = ah + [ah^2 (1/2 + ah/6 + ah^2/24) + al (1 + ah + ah^2/2)]
    // to O(ah^5, al^2) < 1e-16; the bracket is below 1e-6 and is rounded once
    const float poly = fmaf(fmaf(ah, 1.0f / 24.0f, 1.0f / 6.0f), ah, 0.5f);
    const float qal = fmaf(fmaf(ah, 0.5f, 1.0f), ah, 1.0f);
    const float tail = fmaf(al, qal, (ah * ah) * poly);
    const float2 t = tab[j];
    // t * (1 + ah + tail)
    const float p = t.x * ah;
    const float pe = fmaf(t.x, ah, -p);
    const float s = t.x + p;
    const float se = (t.x - s) + p;
    const float lo = se + (pe + fmaf(t.x, tail, fmaf(t.y, ah, t.y)));
    if (i < -125) {
        eh = 0.0f;
        el = 0.0f;
    } else {
        const float sc = __int_as_float((i + 127) << 23);
        eh = s * sc;
        el = lo * sc;
    }
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

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

}  // namespace sv
