// sv_draw.cuh -- the final-token draw of the verify step, as warp-level tasks.
//
// "DistillSpec" Algorithm A.1 ("sample from the adjusted distribution"
// norm(max(0, p_{n+1} - q_{n+1})) after a rejection, otherwise sample the
// bonus token from p_{gamma+1}); "Speculative Decoding and Distillation"
// (Kadimisetty notes) Part 1 steps 4-5. The draw is the inverse CDF in token
// index order: k = min{k : C_k > u * R}.
//
// Exactness of the decision needs the CDF to roughly 40 bits, far beyond
// fp32 sums of fp32 exponentials, so every weight is a float-float
// e = 2^(l log2(e)/T - I) (relative error near 2^-40; I is a per-row integer
// shift, usually 0) and every sum is compensated. With rho = S_p / S_q the
// residual weight of token v is proportional to max(0, e_p(v) - rho e_q(v)).
// For bf16 rows without shift the weights come from the call's bf16 weight
// table, which holds the same float-float values.
//
// Pass task: one warp per (sequence, a span of task_chunks draw chunks of
// kDrawChunk tokens), walking them in blocks of 256 tokens with lane L on
// tokens 8L .. 8L + 7 of each block; the blocks arrive through the warp's
// shared-memory ring by per-lane asynchronous copies, several blocks ahead
// of the arithmetic. Each lane accumulates S_p, S_q and, over the tokens
// whose sign is certain under the row-statistics estimate of rho (window
// 2^-15), P_A = sum e_p and Q_A = sum e_q of the positive ones; the few
// tokens inside the window are listed. Output: each chunk's four totals, as
// float-float pairs.
//
// Finalize task: one warp per sequence forms the exact rho, the chunk masses
// P_A - rho Q_A (+ the listed tokens, settled exactly), locates t = u R among
// the chunks and rescans that chunk block by block with exact weights. With
// the chunk totals staged in the warp's ring it works in float-float on the
// FP32 pipe; otherwise (or with many listed tokens) in double. A list
// overflow or an estimate outside the window makes it compute the masses
// from exact weights instead (slow path, flagged).
#pragma once

#include "sv_stream.cuh"

namespace sv {


// ---------------------------------------------------------------------------
// packed helpers

__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f32x2 splat2(float x) { return pack2(x, x); }

// (ah, al) += (xh, xl) on both halves, keeping the head's rounding error
__device__ __forceinline__ void acc2(f32x2 &ah, f32x2 &al, f32x2 xh, f32x2 xl) {
    const f32x2 s = add2(ah, xh);
    const f32x2 bb = sub2(s, ah);
    const f32x2 e = add2(sub2(ah, sub2(s, bb)), sub2(xh, bb));
    ah = s;
    al = add2(al, add2(xl, e));
}

// Per-row constants of the exponential: c = log2(e)/T as (h, l) on both
// halves and the integer shifts of the two halves.
struct ExpRow {
    f32x2 ch, cl, shift;
    f32x2 lmin;  // logits below M - 1000/c are clamped (their weight is exactly 0)
};

// e = 2^(l c - I) on both halves, as float-float pairs (eh, el).
// y = l c is an exact product split (l is exact); with kShift the integer
// shift is subtracted by TwoSum. Then y = k/4096 + f with |f| <= 2^-13:
// 2^(k/4096) = 2^i T_j from the 4096-entry table, and
// 2^f = 1 + ah + [al + ah (ah/2 + al)] with a = f ln2 as (ah, al). Values
// below 2^-126 are returned as exact zeros; a logit more than 1000/c below
// the row reference M is clamped first (so -inf gives weight 0, not NaN).
template <bool kShift>
__device__ __forceinline__ void exp2_pair(f32x2 lraw, const ExpRow &r,
                                          const float2 *__restrict__ tab, f32x2 &eh, f32x2 &el) {
    const f32x2 z = 0ull;
    f32x2 l;
    {
        const float2 x = unpack2(lraw), lm = unpack2(r.lmin);
        l = pack2(fmaxf(x.x, lm.x), fmaxf(x.y, lm.y));
    }
    f32x2 yh = mul2(l, r.ch);
    f32x2 yl = fma2(l, r.ch, sub2(z, yh));
    yl = fma2(l, r.cl, yl);
    if (kShift) {
        const f32x2 ns = sub2(z, r.shift);
        const f32x2 s = add2(yh, ns);
        const f32x2 bb = sub2(s, yh);
        const f32x2 e = add2(sub2(yh, sub2(s, bb)), sub2(ns, bb));
        yh = s;
        yl = add2(yl, e);
    }
    const f32x2 t = fma2(yh, splat2(4096.0f), splat2(12582912.0f));
    const f32x2 kf = sub2(t, splat2(12582912.0f));
    const f32x2 f = fma2(kf, splat2(-1.0f / 4096.0f), yh);  // exact, |f| <= 2^-13
    const f32x2 ah = mul2(f, splat2(kLn2Hi));
    f32x2 al = fma2(f, splat2(kLn2Hi), sub2(z, ah));
    al = fma2(f, splat2(kLn2Lo), al);
    al = fma2(yl, splat2(kLn2Hi), al);
    const f32x2 elo = fma2(ah, fma2(ah, splat2(0.5f), al), al);
    const float2 tf = unpack2(t);
    const int k0 = __float_as_int(tf.x) - 0x4B400000;
    const int k1 = __float_as_int(tf.y) - 0x4B400000;
    const float2 T0 = tab[k0 & 4095];
    const float2 T1 = tab[k1 & 4095];
    const int i0 = k0 >> 12, i1 = k1 >> 12;
    const f32x2 tx = pack2(T0.x, T1.x);
    const f32x2 ty = pack2(T0.y, T1.y);
    const f32x2 lo = fma2(tx, ah, fma2(tx, elo, fma2(ty, ah, ty)));
    const f32x2 sc = pack2(i0 < -126 ? 0.0f : __int_as_float((i0 + 127) << 23),
                           i1 < -126 ? 0.0f : __int_as_float((i1 + 127) << 23));
    eh = mul2(tx, sc);
    el = mul2(lo, sc);
}

// exact-rho residual weight max(0, e_p - rho e_q) as a float-float
__device__ __forceinline__ void residual_weight(float eph, float epl, float eqh, float eql,
                                                float rh, float rl, float &wh, float &wl) {
    const float ph = rh * eqh;
    float pe = fmaf(rh, eqh, -ph);
    pe = fmaf(rh, eql, pe);
    pe = fmaf(rl, eqh, pe);
    float s, e;
    two_sum(eph, -ph, s, e);
    e += epl - pe;
    wh = s + e;
    wl = e - (wh - s);
    if (!(wh > 0.0f)) {
        wh = 0.0f;
        wl = 0.0f;
    }
}

// L1-bypassing loads of records written by another kernel of this call
__device__ __forceinline__ Quad ld_quad(const ChunkTot *p) {
    const float4 s = __ldcg(&p->s);
    const float4 a = __ldcg(&p->a);
    return Quad{ff_to_double(s.x, s.y), ff_to_double(s.z, s.w), ff_to_double(a.x, a.y),
                ff_to_double(a.z, a.w)};
}

__device__ __forceinline__ ZoneEntry ld_zone(const ZoneEntry *p) {
    ZoneEntry z;
    *reinterpret_cast<int4 *>(&z) = __ldcg(reinterpret_cast<const int4 *>(p));
    *(reinterpret_cast<int4 *>(&z) + 1) = __ldcg(reinterpret_cast<const int4 *>(p) + 1);
    return z;
}

// Eight consecutive logits starting at token v (v a multiple of 8), as floats;
// tokens at or past V read as -inf.
template <int DT>
__device__ __forceinline__ void load8(const char *row, int64_t v, int64_t V, float *x) {
    if (v + 8 <= V) {
        if (DT == SV_DT_BF16) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(row + v * 2));
            x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x);
            x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
            x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z);
            x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
        } else {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(row + v * 4));
            const float4 b = __ldg(reinterpret_cast<const float4 *>(row + v * 4) + 1);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = v + e < V ? load_logit<DT>(row, v + e) : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// per-sequence setup

struct DrawRows {
    const char *prow, *qrow;
    ExpRow er;         // residual: halves (p, q); bonus: both halves p
    bool shift;        // some row needs the general (shifted) exponential
    float rho_est;     // row-statistics estimate of S_p / S_q in the shifted scale
};

__device__ __forceinline__ DrawRows draw_rows(const Params &P, const DrawDesc &d) {
    DrawRows r;
    r.prow = P.target + d.p_phys * P.stride_bytes;
    r.qrow = d.residual ? P.draft + d.q_phys * P.stride_bytes : r.prow;
    r.shift = d.shift != 0;
    r.er.ch = splat2(P.c2h);
    r.er.cl = splat2(P.c2l);
    r.er.shift = pack2(d.ip, d.residual ? d.iq : d.ip);
    r.er.lmin = pack2(d.Mp - P.lspan, d.residual ? d.Mq - P.lspan : d.Mp - P.lspan);
    r.rho_est = d.rho_est;
    return r;
}

__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Sum of a packed float-float pair over the warp (butterfly of float-float
// additions; every lane ends with a total, lane 0's in a fixed order).
__device__ __forceinline__ void warp_sum_ff2(f32x2 &h, f32x2 &l) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const f32x2 oh = __shfl_xor_sync(0xffffffffu, h, off);
        const f32x2 ol = __shfl_xor_sync(0xffffffffu, l, off);
        acc2(h, l, oh, ol);
    }
}

// Inclusive prefix sum of a float-float value over the warp (Hillis-Steele).
__device__ __forceinline__ void warp_incl_scan_ff(float &h, float &l, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float yh = __shfl_up_sync(0xffffffffu, h, off);
        const float yl = __shfl_up_sync(0xffffffffu, l, off);
        if (lane >= off) ff_add(yh, yl, h, l, h, l);
    }
}

__device__ __forceinline__ double warp_incl_scan_d(double x, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    return x;
}

// ---------------------------------------------------------------------------
// raw groups of 8 tokens and the bf16 weight table

template <int DT>
struct Raw {
    uint4 w[DT == SV_DT_BF16 ? 1 : 2];
};

// the 8 logits starting at token v (v + 8 <= V, v a multiple of 8)
template <int DT>
__device__ __forceinline__ void load_raw(const char *row, int64_t v, Raw<DT> &r) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row + v * (DT == SV_DT_BF16 ? 2 : 4));
    r.w[0] = __ldg(p);
    if (DT == SV_DT_FP32) r.w[DT == SV_DT_FP32 ? 1 : 0] = __ldg(p + 1);
}

template <int DT>
__device__ __forceinline__ void raw_floats(const Raw<DT> &r, float *x) {
    if (DT == SV_DT_BF16) {
        const uint4 w = r.w[0];
        x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x);
        x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
        x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z);
        x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
    } else {
        const uint4 a = r.w[0], b = r.w[DT == SV_DT_FP32 ? 1 : 0];
        x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
        x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
        x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
        x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
    }
}

// table offset of a bf16 code (low 16 bits of c): < kCodeHalf inside the table
__device__ __forceinline__ uint32_t code_offset(uint32_t c) { return (c & 0x7FFFu) - kCodeBase; }
__device__ __forceinline__ uint32_t code_index(uint32_t c) {
    return code_offset(c) | ((c >> 4) & (uint32_t)kCodeHalf);
}

// the 8 bf16 codes of a raw group; true when all lie in the table
__device__ __forceinline__ bool raw_codes(const uint4 &w, uint32_t *c) {
    c[0] = w.x & 0xFFFFu; c[1] = w.x >> 16;
    c[2] = w.y & 0xFFFFu; c[3] = w.y >> 16;
    c[4] = w.z & 0xFFFFu; c[5] = w.z >> 16;
    c[6] = w.w & 0xFFFFu; c[7] = w.w >> 16;
    uint32_t out = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) out |= code_offset(c[e]);
    return out < (uint32_t)kCodeHalf;
}

// The bf16 weight table of a call: entry i holds the weight that the
// exponential above gives for the bf16 logit of code
// (i mod kCodeHalf) + kCodeBase, negated when i >= kCodeHalf, in a row
// without shift; stored planar, the kCodeTab float heads then the tails. Entries whose exponent l c lies outside [-1000, 127] are 0:
// the exponential gives 0 below (a row without shift has every l c in
// [M c - 1000, 60]) and no such row reads the entries above.
__device__ inline void build_code_table(float2 *ct, const float2 *tab, float c2h, float c2l, int tid,
                                        int nthreads) {
    ExpRow er;
    er.ch = splat2(c2h);
    er.cl = splat2(c2l);
    er.shift = 0ull;
    er.lmin = splat2(-INFINITY);
    for (int i = tid; i < kCodeTab / 2; i += nthreads) {
        const uint32_t c0 = (uint32_t)(2 * i) % kCodeHalf + kCodeBase;
        const uint32_t s0 = (2 * i) >= kCodeHalf ? 0x8000u : 0u;
        const float l0 = __uint_as_float((c0 | s0) << 16);
        const float l1 = __uint_as_float(((c0 + 1) | s0) << 16);
        f32x2 eh, el;
        exp2_pair<false>(pack2(l0, l1), er, tab, eh, el);
        const float2 h = unpack2(eh), l = unpack2(el);
        const float y0 = l0 * c2h, y1 = l1 * c2h;
        const bool ok0 = y0 >= -1000.0f && y0 <= 127.0f;
        const bool ok1 = y1 >= -1000.0f && y1 <= 127.0f;
        float *heads = reinterpret_cast<float *>(ct), *tails = heads + kCodeTab;
        heads[2 * i] = ok0 ? h.x : 0.0f;
        tails[2 * i] = ok0 ? l.x : 0.0f;
        heads[2 * i + 1] = ok1 ? h.y : 0.0f;
        tails[2 * i + 1] = ok1 ? l.y : 0.0f;
    }
}

// ---------------------------------------------------------------------------
// pass task

// Two independent sets of accumulators (tokens alternate between them) for
// instruction-level parallelism; merged at the end of the chunk.
struct PassAcc {
    f32x2 sh, sl;  // (S_p, S_q), or two halves of S_p for a bonus draw
    f32x2 ah, al;  // (P_A, Q_A)
};

// List a token whose residual sign the estimated rho cannot decide (rare).
static __device__ __noinline__ void list_token(const Params &P, int b, int64_t v, f32x2 eh, f32x2 el) {
    const uint32_t slot = atomicAdd(&P.zone_cnt[b], 1u);
    if (slot < (uint32_t)kZoneMax) {
        const float2 h = unpack2(eh), lw = unpack2(el);
        ZoneEntry zz;
        zz.v = (int32_t)v;
        zz.eph = h.x;
        zz.epl = lw.x;
        zz.eqh = h.y;
        zz.eql = lw.y;
        zz.pad[0] = zz.pad[1] = zz.pad[2] = 0;
        P.zone[(int64_t)b * kZoneMax + slot] = zz;
    }
}

// one token of a residual pass: S_p, S_q always; P_A, Q_A when the sign of
// e_p - rho e_q is certain under the estimated rho (a 0/1 factor, no
// branch). Returns whether the token must be listed (its sign undecided).
__device__ __forceinline__ bool residual_token(f32x2 eh, f32x2 el, float rhi, float rlo,
                                               PassAcc &a) {
    acc2(a.sh, a.sl, eh, el);
    const float2 h = unpack2(eh);
    const bool pos = h.x > rhi * h.y;
    const float k = pos ? 1.0f : 0.0f;
    const f32x2 k2 = pack2(k, k);
    acc2(a.ah, a.al, mul2(eh, k2), mul2(el, k2));
    return !pos && h.y > 0.0f && h.x >= rlo * h.y;
}

// 8 tokens from their logits (tokens at or past V read as -inf: weight 0)
template <bool kShift, bool kRes>
__device__ __forceinline__ void pass_floats(const Params &P, const DrawRows &r, int b, int64_t v,
                                            const float *xp, const float *xq, const float2 *tab,
                                            float rhi, float rlo, PassAcc *a) {
    if (kRes) {
        f32x2 eh[8], el[8];
        uint32_t listed = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            exp2_pair<kShift>(pack2(xp[e], xq[e]), r.er, tab, eh[e], el[e]);
            listed |= residual_token(eh[e], el[e], rhi, rlo, a[e & 1]) ? 1u << e : 0u;
        }
        if (listed) {  // rare: outside the unrolled group, one branch per group
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (listed & (1u << e)) list_token(P, b, v + e, eh[e], el[e]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            f32x2 eh, el;
            exp2_pair<kShift>(pack2(xp[e], xp[e + 1]), r.er, tab, eh, el);
            acc2(a[(e >> 1) & 1].sh, a[(e >> 1) & 1].sl, eh, el);
        }
    }
}

// Byte offsets into the planar bf16 weight heads of the two bf16 codes in
// word w, in the two 16-bit halves of the result; bits of 0xF800F800 in *out
// are set when a code lies outside the table. Both halves at once: the
// magnitudes minus kCodeBase (a half below kCodeBase borrows and so flags
// itself), the sign bit moved to bit 11 of its half, times 4.
__device__ __forceinline__ uint32_t code_offsets2(uint32_t w, uint32_t &out) {
    const uint32_t d = (w & 0x7FFF7FFFu) - (kCodeBase | (kCodeBase << 16));
    out |= d;
    return (d | ((w >> 4) & 0x08000800u)) << 2;
}

// head and tail of the table weight at byte offset off
__device__ __forceinline__ float head_at(const float2 *ct, uint32_t off) {
    return *reinterpret_cast<const float *>(reinterpret_cast<const char *>(ct) + off);
}
__device__ __forceinline__ float tail_at(const float2 *ct, uint32_t off) {
    return *reinterpret_cast<const float *>(reinterpret_cast<const char *>(ct) + off +
                                            kCodeTab * sizeof(float));
}

// 8 tokens from raw words; kTab: weights from the bf16 table when all codes
// of the group lie in it (the same values the exponential gives)
template <int DT, bool kShift, bool kTab, bool kRes>
__device__ __forceinline__ void pass_raw(const Params &P, const DrawRows &r, int b, int64_t v,
                                         const Raw<DT> &rp, const Raw<DT> &rq, const float2 *tab,
                                         const float2 *ct, float rhi, float rlo, PassAcc *a) {
    if (kTab) {
        const uint32_t wp[4] = {rp.w[0].x, rp.w[0].y, rp.w[0].z, rp.w[0].w};
        const uint32_t wq[4] = {rq.w[0].x, rq.w[0].y, rq.w[0].z, rq.w[0].w};
        uint32_t out = 0, op[4], oq[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            op[k] = code_offsets2(wp[k], out);
            if (kRes) oq[k] = code_offsets2(wq[k], out);
        }
        if ((out & 0xF800F800u) == 0u) {
            uint32_t listed = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t p0 = op[k] & 0xFFFFu, p1 = op[k] >> 16;
                if (kRes) {
                    const uint32_t q0 = oq[k] & 0xFFFFu, q1 = oq[k] >> 16;
                    const f32x2 h0 = pack2(head_at(ct, p0), head_at(ct, q0));
                    const f32x2 l0 = pack2(tail_at(ct, p0), tail_at(ct, q0));
                    const f32x2 h1 = pack2(head_at(ct, p1), head_at(ct, q1));
                    const f32x2 l1 = pack2(tail_at(ct, p1), tail_at(ct, q1));
                    listed |= residual_token(h0, l0, rhi, rlo, a[0]) ? 1u << (2 * k) : 0u;
                    listed |= residual_token(h1, l1, rhi, rlo, a[1]) ? 2u << (2 * k) : 0u;
                } else {
                    acc2(a[k & 1].sh, a[k & 1].sl, pack2(head_at(ct, p0), head_at(ct, p1)),
                         pack2(tail_at(ct, p0), tail_at(ct, p1)));
                }
            }
            if (kRes && listed) {  // rare: outside the unrolled group
#pragma unroll
                for (int k = 0; k < 4; ++k) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (!(listed & (1u << (2 * k + h)))) continue;
                        const uint32_t pk = h ? op[k] >> 16 : op[k] & 0xFFFFu;
                        const uint32_t qk = h ? oq[k] >> 16 : oq[k] & 0xFFFFu;
                        list_token(P, b, v + 2 * k + h, pack2(head_at(ct, pk), head_at(ct, qk)),
                                   pack2(tail_at(ct, pk), tail_at(ct, qk)));
                    }
                }
            }
            return;
        }
    }
    float xp[8], xq[8];
    raw_floats<DT>(rp, xp);
    if (kRes) raw_floats<DT>(rq, xq);
    pass_floats<kShift, kRes>(P, r, b, v, xp, xq, tab, rhi, rlo, a);
}

// ---------------------------------------------------------------------------
// the warp's draw ring: per-lane asynchronous copies

// 16 bytes global -> shared, cached in L2 only; completes with its group
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// waits until at most N of this thread's groups are pending
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A warp's ring of kPassRingBytes holds D blocks of 256 tokens of both draw
// rows. Lane L copies its own 8 tokens of each row and reads back only those,
// so the ring needs no barrier: a lane's wait on its own copy groups is
// enough. Row r's 16-byte word w of lane L in slot s lies at
// s * kSlot + ((r * W + w) * 32 + L) * 16 (a warp's reads of one word are
// 512 contiguous bytes).
template <int DT>
struct DrawRing {
    static constexpr int W = DT == SV_DT_BF16 ? 1 : 2;  // words per lane per row
    static constexpr int kSlot = 2 * W * 512;
    static constexpr int D = kPassRingBytes / kSlot;    // blocks in flight
    static_assert(D >= 2, "at least double buffering");
};

// issue the copies of token group v (v + 8 <= V) of row p (and q) into slot s
template <int DT, bool kRes>
__device__ __forceinline__ void ring_copy(uint32_t ring, int s, const DrawRows &r, int64_t v,
                                          int lane) {
    using R = DrawRing<DT>;
    constexpr int ESZ = DT == SV_DT_FP32 ? 4 : 2;
    const uint32_t base = ring + (uint32_t)(s * R::kSlot + lane * 16);
#pragma unroll
    for (int w = 0; w < R::W; ++w) {
        cp_async16(base + w * 512, r.prow + v * ESZ + 16 * w);
        if (kRes) cp_async16(base + (R::W + w) * 512, r.qrow + v * ESZ + 16 * w);
    }
}

// read back this lane's words of row `row` from slot s
template <int DT>
__device__ __forceinline__ void ring_read(const uint8_t *ring, int s, int row, int lane,
                                          Raw<DT> &out) {
    using R = DrawRing<DT>;
    const uint8_t *p = ring + s * R::kSlot + lane * 16 + row * R::W * 512;
#pragma unroll
    for (int w = 0; w < R::W; ++w) out.w[w] = *reinterpret_cast<const uint4 *>(p + w * 512);
}

// The chunk totals in float-float: the two accumulator sets, then the 32
// lanes (butterfly; lane 0's result is the chunk's), stored to draw_chunk;
// the accumulators restart at zero.
__device__ __forceinline__ void store_chunk_totals(const Params &P, int b, int c, bool residual,
                                                   PassAcc *a, int lane) {
    acc2(a[0].sh, a[0].sl, a[1].sh, a[1].sl);
    warp_sum_ff2(a[0].sh, a[0].sl);
    if (residual) {
        acc2(a[0].ah, a[0].al, a[1].ah, a[1].al);
        warp_sum_ff2(a[0].ah, a[0].al);
    }
    if (lane == 0) {
        const float2 h = unpack2(a[0].sh), l = unpack2(a[0].sl);
        ChunkTot tot;
        if (residual) {
            const float2 g = unpack2(a[0].ah), m = unpack2(a[0].al);
            tot.s = make_float4(h.x, l.x, h.y, l.y);
            tot.a = make_float4(g.x, m.x, g.y, m.y);
        } else {  // a bonus pass: the two halves are two parts of S_p
            float sh, sl;
            ff_add(h.x, l.x, h.y, l.y, sh, sl);
            tot.s = make_float4(sh, sl, 0.0f, 0.0f);
            tot.a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        P.draw_chunk[(int64_t)b * P.nch3 + c] = tot;
    }
    a[0] = a[1] = PassAcc{0ull, 0ull, 0ull, 0ull};
}

// The pass over draw chunks [c_begin, c_end) of sequence b: the blocks of
// 256 tokens in order, D of them in flight through the warp's ring; each
// lane takes tokens 8L .. 8L + 7 of every block, so the summation order is
// that of a chunk-by-chunk walk.
template <int DT, bool kShift, bool kTab, bool kRes>
__device__ void pass_span(const Params &P, const DrawRows &r, int b, int c_begin, int c_end,
                          const float2 *tab, const float2 *ct, uint8_t *ring, int lane) {
    constexpr int D = DrawRing<DT>::D;
    constexpr int kBlkPerChunk = kDrawChunk / kDrawBlock;
    const float rhi = r.rho_est * (float)(1.0 + kRhoWindow);
    const float rlo = r.rho_est * (float)(1.0 - kRhoWindow);
    const int64_t v0 = (int64_t)c_begin * kDrawChunk + 8 * lane;  // this lane's first token
    const int64_t vend = min(P.V, (int64_t)c_end * kDrawChunk);
    const int nblk = (int)((vend - (int64_t)c_begin * kDrawChunk + kDrawBlock - 1) / kDrawBlock);
    const uint32_t rs = smem_u32(ring);
    auto issue = [&](int j) {
        const int64_t v = v0 + (int64_t)j * kDrawBlock;
        if (j < nblk && v + 8 <= vend) ring_copy<DT, kRes>(rs, j % D, r, v, lane);
        cp_async_commit();  // one group per block, empty or not
    };
#pragma unroll
    for (int j = 0; j < D - 1; ++j) issue(j);
    PassAcc a[2] = {{0ull, 0ull, 0ull, 0ull}, {0ull, 0ull, 0ull, 0ull}};
    for (int j = 0; j < nblk; ++j) {
        issue(j + D - 1);
        cp_async_wait<D - 1>();  // block j has landed
        const int64_t v = v0 + (int64_t)j * kDrawBlock;
        if (v + 8 <= vend) {
            Raw<DT> rp, rq;
            ring_read<DT>(ring, j % D, 0, lane, rp);
            if (kRes) ring_read<DT>(ring, j % D, 1, lane, rq);
            pass_raw<DT, kShift, kTab, kRes>(P, r, b, v, rp, rq, tab, ct, rhi, rlo, a);
        } else if (v < vend) {  // the ragged end of the row
            float xp[8], xq[8];
            load8<DT>(r.prow, v, P.V, xp);
            if (kRes) load8<DT>(r.qrow, v, P.V, xq);
            pass_floats<kShift, kRes>(P, r, b, v, xp, xq, tab, rhi, rlo, a);
        }
        if ((j + 1) % kBlkPerChunk == 0 || j + 1 == nblk)
            store_chunk_totals(P, b, c_begin + j / kBlkPerChunk, kRes, a, lane);
    }
    cp_async_wait<0>();  // the trailing empty groups
}

// Pass task t of sequence b: chunks t * task_chunks .. (t + 1) * task_chunks
// - 1 (those that exist), each chunk's S_p, S_q, P_A, Q_A to draw_chunk.
// ct: the bf16 weight table of this call, or null. ring: the warp's
// kPassRingBytes of shared memory (16-byte aligned).
template <int DT>
__device__ void pass_task(const Params &P, int b, int t, const DrawDesc &d, const float2 *tab,
                          const float2 *ct, uint8_t *ring, int lane) {
    const DrawRows r = draw_rows(P, d);
    const int c0 = t * P.task_chunks;
    const int c1 = min(P.nch3, (t + 1) * P.task_chunks);
    if (c0 >= c1) return;
    if constexpr (DT == SV_DT_BF16) {
        if (ct != nullptr && !r.shift) {
            if (d.residual)
                pass_span<DT, false, true, true>(P, r, b, c0, c1, tab, ct, ring, lane);
            else
                pass_span<DT, false, true, false>(P, r, b, c0, c1, tab, ct, ring, lane);
            return;
        }
    }
    // bf16 rows without the weight table take the shifted exponential (with
    // a zero shift it gives the same weights): one variant fewer in the code
    if (r.shift || DT == SV_DT_BF16) {
        if (d.residual)
            pass_span<DT, true, false, true>(P, r, b, c0, c1, tab, ct, ring, lane);
        else
            pass_span<DT, true, false, false>(P, r, b, c0, c1, tab, ct, ring, lane);
    } else {
        if (d.residual)
            pass_span<DT, false, false, true>(P, r, b, c0, c1, tab, ct, ring, lane);
        else
            pass_span<DT, false, false, false>(P, r, b, c0, c1, tab, ct, ring, lane);
    }
}

// A draw descriptor written by another kernel of this call (L1 bypassed)
__device__ __forceinline__ DrawDesc load_desc(const DrawDesc *p) {
    static_assert(sizeof(DrawDesc) % 16 == 0, "DrawDesc is loaded as 16-byte words");
    DrawDesc d;
    const int4 *src = reinterpret_cast<const int4 *>(p);
    int4 *dst = reinterpret_cast<int4 *>(&d);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(DrawDesc) / 16); ++i) dst[i] = __ldcg(src + i);
    return d;
}

// ---------------------------------------------------------------------------
// finalize task

// Exact weights of the 8 tokens v .. v + 7 under the final rho (tokens at or
// past V weigh 0): e_p for a bonus draw, max(0, e_p - rho e_q) otherwise.
// staged_p, staged_q: the raw words already in registers (v + 8 <= V), or
// null to load them here.
template <int DT, bool kShift, bool kTab>
__device__ __forceinline__ void exact_group(const Params &P, const DrawRows &r, int64_t v,
                                            bool residual, float rh, float rl, const float2 *tab,
                                            const float2 *ct, float *wh, float *wl,
                                            const Raw<DT> *staged_p = nullptr,
                                            const Raw<DT> *staged_q = nullptr) {
    float eph[8], epl[8], eqh[8], eql[8];
    bool done = false;
    float xp[8], xq[8];
    if (v + 8 <= P.V) {
        Raw<DT> rp, rq;
        if (staged_p != nullptr) {
            rp = *staged_p;
            if (residual) rq = *staged_q;
        } else {
            load_raw<DT>(r.prow, v, rp);
            if (residual) load_raw<DT>(r.qrow, v, rq);
        }
        if (kTab && ct != nullptr) {
            uint32_t cp[8], cq[8];
            bool in = raw_codes(rp.w[0], cp);
            if (residual) in &= raw_codes(rq.w[0], cq);
            if (in) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float *heads = reinterpret_cast<const float *>(ct);
                    const uint32_t ip = code_index(cp[e]);
                    eph[e] = heads[ip];
                    epl[e] = heads[kCodeTab + ip];
                    eqh[e] = 0.0f;
                    eql[e] = 0.0f;
                    if (residual) {
                        const uint32_t iq = code_index(cq[e]);
                        eqh[e] = heads[iq];
                        eql[e] = heads[kCodeTab + iq];
                    }
                }
                done = true;
            }
        }
        if (!done) {
            raw_floats<DT>(rp, xp);
            if (residual) raw_floats<DT>(rq, xq);
        }
    } else {
        load8<DT>(r.prow, v, P.V, xp);
        if (residual) load8<DT>(r.qrow, v, P.V, xq);
    }
    if (!done) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            f32x2 eh, el;
            exp2_pair<kShift>(pack2(xp[e], residual ? xq[e] : xp[e]), r.er, tab, eh, el);
            const float2 h = unpack2(eh), l = unpack2(el);
            eph[e] = h.x;
            epl[e] = l.x;
            eqh[e] = h.y;
            eql[e] = l.y;
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if (residual) {
            residual_weight(eph[e], epl[e], eqh[e], eql[e], rh, rl, wh[e], wl[e]);
        } else {
            wh[e] = eph[e];
            wl[e] = epl[e];
        }
    }
}

// Sum of the exact weights of chunk c (slow path), by the whole warp.
template <int DT, bool kShift, bool kTab>
__device__ double exact_chunk_sum(const Params &P, const DrawRows &r, int c, bool residual, float rh,
                                  float rl, const float2 *tab, const float2 *ct, int lane) {
    const int64_t c0 = (int64_t)c * kDrawChunk;
    const int64_t cend = min(P.V, c0 + kDrawChunk);
    float sh = 0.0f, sl = 0.0f;
    for (int64_t v = c0 + 8 * lane; v < cend; v += kDrawBlock) {
        float wh[8], wl[8];
        exact_group<DT, kShift, kTab>(P, r, v, residual, rh, rl, tab, ct, wh, wl);
#pragma unroll
        for (int e = 0; e < 8; ++e) ff_accumulate(sh, sl, wh[e], wl[e]);
    }
    return warp_sum_d(ff_to_double(sh, sl));
}

// a > b for normalised float-float values (a head plus a tail of at most
// half its unit in the last place)
__device__ __forceinline__ bool ff_gt(float ah, float al, float bh, float bl) {
    return ah > bh || (ah == bh && al > bl);
}

// Sum of a float-float value over the warp (butterfly); every lane returns
// lane 0's total, so all lanes take the same decisions.
__device__ __forceinline__ void warp_sum_ff(float &h, float &l) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, h, off);
        const float ol = __shfl_xor_sync(0xffffffffu, l, off);
        ff_add(h, l, oh, ol, h, l);
    }
    h = __shfl_sync(0xffffffffu, h, 0);
    l = __shfl_sync(0xffffffffu, l, 0);
}

// The chunk stage of a finalize when every chunk total of the sequence fits
// in the warp's ring and at most 32 tokens were listed: the totals are
// staged in shared memory, and S_p, S_q, rho, the listed tokens' weights, the
// chunk masses, R and the chunk c* that holds t = u R are all formed in
// float-float on the FP32 pipe (FP64 runs at a small fraction of its rate).
// Returns false, having decided nothing, in the cases the general path
// handles: an estimate of rho outside the window, or a residual mass that
// rounds to zero. cstar stays -1 when t lies at or past the end.
static __device__ __noinline__ bool finalize_fast(const Params &P, int b, const DrawDesc &d,
                                           const DrawRows &r, int nch, const ChunkTot *chunk,
                                           const ZoneEntry *zs, int zc, uint8_t *ring, int lane,
                                           float &rh, float &rl, int &cstar, int &lastpos_chunk,
                                           float &tlh, float &tll) {
    const uint32_t rs = smem_u32(ring);
    const char *src = reinterpret_cast<const char *>(chunk);
    for (int i = lane; i < 2 * nch; i += 32) cp_async16(rs + 16u * (uint32_t)i, src + 16 * i);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    ChunkTot *cs = reinterpret_cast<ChunkTot *>(ring);
    const bool residual = d.residual != 0;
    rh = 1.0f;
    rl = 0.0f;
    if (residual) {
        // S_p, S_q in a fixed order (lane-strided, then the butterfly)
        float sph = 0.0f, spl = 0.0f, sqh = 0.0f, sql = 0.0f;
        for (int c = lane; c < nch; c += 32) {
            const float4 v = cs[c].s;
            ff_add(sph, spl, v.x, v.y, sph, spl);
            ff_add(sqh, sql, v.z, v.w, sqh, sql);
        }
        warp_sum_ff(sph, spl);
        warp_sum_ff(sqh, sql);
        // rho = S_p / S_q: a first quotient, then the quotient of its
        // remainder S_p - q1 S_q (formed with an exact product)
        const float q1 = sph / sqh;
        const float ph = q1 * sqh;
        float pl = fmaf(q1, sqh, -ph);
        pl = fmaf(q1, sql, pl);
        const float r1 = ((sph - ph) - pl) + spl;
        const float q2 = r1 / sqh;
        rh = q1 + q2;
        rl = q2 - (rh - q1);
        if (!(fabsf(rh / r.rho_est - 1.0f) <= (float)(0.5 * kRhoWindow))) return false;
        // each listed token's exact weight joins P_A of its chunk, in token order
        if (zc > 0) {
            int zv = INT_MAX, zchunk = 0;
            float zwh = 0.0f, zwl = 0.0f;
            if (lane < zc) {
                const ZoneEntry z = ld_zone(&zs[lane]);
                zv = z.v;
                zchunk = z.v / kDrawChunk;
                residual_weight(z.eph, z.epl, z.eqh, z.eql, rh, rl, zwh, zwl);
            }
            int rank = 0;
            for (int j = 0; j < 32; ++j) rank += __shfl_sync(0xffffffffu, zv, j) < zv ? 1 : 0;
            for (int k = 0; k < zc; ++k) {
                const int who = __ffs(__ballot_sync(0xffffffffu, lane < zc && rank == k)) - 1;
                const int c = __shfl_sync(0xffffffffu, zchunk, who);
                const float wh = __shfl_sync(0xffffffffu, zwh, who);
                const float wl = __shfl_sync(0xffffffffu, zwl, who);
                if (lane == 0 && wh > 0.0f) {
                    float4 a = cs[c].a;
                    ff_add(a.x, a.y, wh, wl, a.x, a.y);
                    cs[c].a = a;
                }
                __syncwarp();
            }
        }
    }
    // the mass of chunk c: P_A - rho Q_A, or S_p for a bonus draw
    auto mass_of = [&](int c, float &mh, float &ml) {
        if (residual) {
            const float4 a = cs[c].a;
            const float xh = rh * a.z;
            float xl = fmaf(rh, a.z, -xh);
            xl = fmaf(rh, a.w, xl);
            xl = fmaf(rl, a.z, xl);
            ff_add(a.x, a.y, -xh, -xl, mh, ml);
        } else {
            const float4 v = cs[c].s;
            mh = v.x;
            ml = v.y;
        }
    };
    // the chunk masses, a contiguous run of chunks a lane: each lane's total,
    // one warp scan (its last prefix is R), then the lane whose prefix
    // passes t = u R walks its chunks
    const int per = (nch + 31) / 32;
    const int cb = min(nch, lane * per), ce = min(nch, cb + per);
    float sh = 0.0f, sl = 0.0f;
    int lastp = -1;
    for (int c = cb; c < ce; ++c) {
        float mh, ml;
        mass_of(c, mh, ml);
        ff_add(sh, sl, mh, ml, sh, sl);
        if (mh > 0.0f || (mh == 0.0f && ml > 0.0f)) lastp = c;
    }
    float ih = sh, il = sl;
    warp_incl_scan_ff(ih, il, lane);
    const float Rh = __shfl_sync(0xffffffffu, ih, 31), Rl = __shfl_sync(0xffffffffu, il, 31);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lastp = max(lastp, __shfl_xor_sync(0xffffffffu, lastp, off));
    lastpos_chunk = lastp;
    if (!(Rh > 0.0f) || !isfinite(Rh)) return false;
    // t = u R, u the draw uniform (both float-float)
    float th, tl;
    {
        float uh, ul;
        draw_uniform_ff(P.seed, (uint32_t)b, (uint32_t)(d.n + 1), uh, ul);
        ff_mul(uh, ul, Rh, Rl, th, tl);
    }
    const uint32_t hit = __ballot_sync(0xffffffffu, cb < ce && ff_gt(ih, il, th, tl));
    if (!hit) {  // t at or past the end through rounding
        ff_add(th, tl, -Rh, -Rl, tlh, tll);
        return true;
    }
    const int L = __ffs(hit) - 1;
    int cpick = -1;
    float eh = 0.0f, el = 0.0f;  // C before chunk cpick
    if (lane == L) {
        ff_add(ih, il, -sh, -sl, eh, el);  // C before this lane's chunks
        int lastc = -1;
        float lh = 0.0f, ll = 0.0f;  // C before lastc
        for (int c = cb; c < ce; ++c) {
            float mh, ml, nh, nl;
            mass_of(c, mh, ml);
            ff_add(eh, el, mh, ml, nh, nl);
            if (ff_gt(nh, nl, th, tl)) {
                cpick = c;
                break;
            }
            if (mh > 0.0f || (mh == 0.0f && ml > 0.0f)) {
                lastc = c;
                lh = eh;
                ll = el;
            }
            eh = nh;
            el = nl;
        }
        // summed in this order the lane can round below t: its last chunk of
        // positive mass then holds it
        if (cpick < 0) {
            cpick = lastc >= 0 ? lastc : ce - 1;
            if (lastc >= 0) {
                eh = lh;
                el = ll;
            }
        }
    }
    cstar = __shfl_sync(0xffffffffu, cpick, L);
    eh = __shfl_sync(0xffffffffu, eh, L);
    el = __shfl_sync(0xffffffffu, el, L);
    ff_add(th, tl, -eh, -el, tlh, tll);
    return true;
}

// What the chunk stage of a finalize hands to its rescan.
struct FinState {
    float rh, rl;        // rho = S_p / S_q as a float-float (1 for a bonus draw)
    float tlh, tll;      // t - C before chunk c*, t = u R
    int cstar;           // the chunk that holds t, -1 when t lies at or past the end
    int lastpos_chunk;   // the last chunk of positive mass
    int residual;        // 0 once a zero residual mass fell back to p_{n+1}
};

// The general chunk stage (FP64 chunk masses; exact chunk sums when rho left
// the window or too many tokens were listed). Out of line, like the other
// finalize stages, so that each is register-allocated on its own.
template <int DT>
__device__ __noinline__ void finalize_general(const Params &P, int b, const DrawDesc &d,
                                              const DrawRows &r, const float2 *tab,
                                              const float2 *ct, int lane, FinState &f) {
    const int nch = P.nch3;
    const ChunkTot *chunk = P.draw_chunk + (int64_t)b * nch;
    double *mass = P.draw_mass + (int64_t)b * nch;
    ZoneEntry *zs = P.zone + (int64_t)b * kZoneMax;
    const int zc_all = d.residual ? (int)__ldcg(&P.zone_cnt[b]) : 0;
    int residual = d.residual;
    int cstar = -1, lastpos_chunk = -1;
    float rh, rl, tlh, tll;
    double before = 0.0;
    double sp = 0.0, sq = 0.0;
    for (int c = lane; c < nch; c += 32) {
        const Quad q = ld_quad(&chunk[c]);
        sp += q.x;
        sq += q.y;
    }
    sp = warp_sum_d(sp);
    sq = warp_sum_d(sq);
    const double rho = residual ? sp / sq : 1.0;
    rh = (float)rho;
    rl = (float)(rho - (double)rh);
    const bool slow = residual && (zc_all > kZoneMax ||
                                   !(fabs(rho / (double)r.rho_est - 1.0) <= 0.5 * kRhoWindow));
    const int zc = slow ? 0 : min(zc_all, kZoneMax);
    if (zc > 1 && lane == 0) {
        // sort the ambiguous tokens by index (in place): a fixed summation order
        for (int i = 1; i < zc; ++i) {
            const ZoneEntry z = ld_zone(&zs[i]);
            int j = i - 1;
            ZoneEntry y = ld_zone(&zs[j]);
            while (y.v > z.v) {
                zs[j + 1] = y;
                if (--j < 0) break;
                y = ld_zone(&zs[j]);
            }
            zs[j + 1] = z;
        }
    }
    __syncwarp();
    if (slow && lane == 0) atomicOr(P.status, SPECVERIFY_STATUS_DRAW_SLOW);

    // chunk masses (in the scratch row `mass`) and their total R
    double R = 0.0;
    if (slow) {
        for (int c = 0; c < nch; ++c) {
            const double m = exact_chunk_sum<DT, true, true>(P, r, c, true, rh, rl, tab, ct, lane);
            if (lane == 0) __stcg(&mass[c], m);
            R += m;
        }
    } else {
        double part_r = 0.0;
        for (int c = lane; c < nch; c += 32) {
            const Quad q = ld_quad(&chunk[c]);
            double m = q.x;
            if (residual) {
                m = q.z - rho * q.w;
                for (int i = 0; i < zc; ++i) {
                    const ZoneEntry z = ld_zone(&zs[i]);
                    if (z.v / kDrawChunk == c) {
                        const double w =
                            ff_to_double(z.eph, z.epl) - rho * ff_to_double(z.eqh, z.eql);
                        if (w > 0.0) m += w;
                    }
                }
            }
            __stcg(&mass[c], m);
            part_r += m;
        }
        R = warp_sum_d(part_r);
    }
    if (!(R > 0.0) || !isfinite(R)) {
        // zero residual mass through rounding: draw from p_{n+1}
        residual = 0;
        if (lane == 0) atomicOr(P.status, SPECVERIFY_STATUS_DRAW_ZERO_MASS);
        double part_r = 0.0;
        for (int c = lane; c < nch; c += 32) {
            const double m = ld_quad(&chunk[c]).x;
            __stcg(&mass[c], m);
            part_r += m;
        }
        R = warp_sum_d(part_r);
    }
    __syncwarp();
    const double u = draw_uniform(P.seed, (uint32_t)b, (uint32_t)(d.n + 1));
    const double t = u * R;

    // the chunk: first c with C_c > t
    for (int c0 = 0; c0 < nch && cstar < 0; c0 += 32) {
        const double m = c0 + lane < nch ? __ldcg(&mass[c0 + lane]) : 0.0;
        const double incl = before + warp_incl_scan_d(m, lane);
        const uint32_t hit = __ballot_sync(0xffffffffu, c0 + lane < nch && incl > t);
        const uint32_t pos = __ballot_sync(0xffffffffu, m > 0.0);
        if (pos) lastpos_chunk = c0 + 31 - __clz(pos);
        if (hit) {
            const int l = __ffs(hit) - 1;
            cstar = c0 + l;
            before = __shfl_sync(0xffffffffu, incl - m, l);
        } else {
            before = __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    // t - C before chunk c*, as a float-float: the rescan compares in
    // float-float on the FP32 pipe
    const double tld = t - before;
    tlh = (float)tld;
    tll = (float)(tld - (double)tlh);
    f.rh = rh;
    f.rl = rl;
    f.tlh = tlh;
    f.tll = tll;
    f.cstar = cstar;
    f.lastpos_chunk = lastpos_chunk;
    f.residual = residual;
}

// The rescan of chunk c* with exact weights: the token where C crosses t.
template <int DT>
__device__ __noinline__ void finalize_rescan(const Params &P, int b, const DrawDesc &d,
                                             const DrawRows &r, const float2 *tab,
                                             const float2 *ct, uint8_t *ring, int lane,
                                             const FinState &f) {
    const float rh = f.rh, rl = f.rl, tlh = f.tlh, tll = f.tll;
    const int residual = f.residual;
    int cstar = f.cstar;
    const int lastpos_chunk = f.lastpos_chunk;
    const bool takelast = cstar < 0;  // t at or past the end through rounding
    if (takelast) cstar = lastpos_chunk < 0 ? 0 : lastpos_chunk;

    // rescan chunk c* in blocks of 256 tokens with exact weights, D blocks
    // in flight through the warp's ring
    const int64_t c0 = (int64_t)cstar * kDrawChunk;
    const int64_t cend = min(P.V, c0 + kDrawChunk);
    const int nblk = (int)((cend - c0 + kDrawBlock - 1) / kDrawBlock);
    constexpr int D = DrawRing<DT>::D;
    const uint32_t rs = smem_u32(ring);
    auto issue = [&](int j) {
        const int64_t v = c0 + (int64_t)j * kDrawBlock + 8 * lane;
        if (j < nblk && v + 8 <= cend) {
            if (residual)
                ring_copy<DT, true>(rs, j % D, r, v, lane);
            else
                ring_copy<DT, false>(rs, j % D, r, v, lane);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < D - 1; ++j) issue(j);
    float runh = 0.0f, runl = 0.0f;  // mass of the blocks before this one
    int k = -1, lastpos = -1;
    for (int j = 0; j < nblk && k < 0; ++j) {
        issue(j + D - 1);
        cp_async_wait<D - 1>();  // block j has landed
        const int64_t v = c0 + (int64_t)j * kDrawBlock + 8 * lane;
        float wh[8], wl[8];
        float mh = 0.0f, ml = 0.0f;  // this lane's 8 weights, float-float
        if (v < cend) {
            if (v + 8 <= cend) {
                Raw<DT> rp, rq;
                ring_read<DT>(ring, j % D, 0, lane, rp);
                if (residual) ring_read<DT>(ring, j % D, 1, lane, rq);
                exact_group<DT, true, true>(P, r, v, residual, rh, rl, tab, ct, wh, wl, &rp, &rq);
            } else {
                exact_group<DT, true, true>(P, r, v, residual, rh, rl, tab, ct, wh, wl);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                ff_accumulate(mh, ml, wh[e], wl[e]);
                if (wh[e] > 0.0f && v + e < cend) lastpos = (int)(v + e);
            }
        }
        float ih = mh, il = ml;
        warp_incl_scan_ff(ih, il, lane);
        ff_add(runh, runl, ih, il, ih, il);  // C at the end of this lane's 8 tokens
        if (!takelast) {
            const uint32_t hit = __ballot_sync(0xffffffffu, v < cend && ff_gt(ih, il, tlh, tll));
            if (hit) {
                const int L = __ffs(hit) - 1;
                int kk = -1;
                if (lane == L) {
                    float ch, cl;  // C before this lane's 8 tokens
                    ff_add(ih, il, -mh, -ml, ch, cl);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        ff_add(ch, cl, wh[e], wl[e], ch, cl);
                        if (kk < 0 && v + e < cend && ff_gt(ch, cl, tlh, tll)) kk = (int)(v + e);
                    }
                    // summed in this order the group can round below tl: its
                    // last positive token then holds the crossing
                    int lastp = -1;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (wh[e] > 0.0f && v + e < cend) lastp = (int)(v + e);
                    if (kk < 0) kk = lastp >= 0 ? lastp : (int)v;
                }
                k = __shfl_sync(0xffffffffu, kk, L);
            }
        }
        runh = __shfl_sync(0xffffffffu, ih, 31);
        runl = __shfl_sync(0xffffffffu, il, 31);
    }
    cp_async_wait<0>();  // copies still in flight after an early stop
    int lp = lastpos;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, off));
    if (lane == 0)
        P.tok_out[(int64_t)b * (P.gamma_max + 1) + d.n] = k >= 0 ? k : (lp >= 0 ? lp : (int)c0);
}

// The finalize of sequence b, once all its pass tasks are done: the chunk
// stage (float-float when the totals fit the ring, else the general one),
// then the rescan of chunk c*. The weights come from the bf16 weight table
// (ct, rows without shift only) where the codes lie in it, else from the
// exponential with the row's shift (0 for a row without shift, where it
// gives the table's values bit for bit): one instantiation of each stage
// keeps the kernel's code, and so its instruction-cache footprint, small.
// ring: the warp's kPassRingBytes of shared memory (16-byte aligned).
template <int DT>
__device__ __noinline__ void finalize_task(const Params &P, int b, const DrawDesc &d,
                                           const float2 *tab, const float2 *ct_call,
                                           uint8_t *ring, int lane) {
    const DrawRows r = draw_rows(P, d);
    const float2 *ct = r.shift ? nullptr : ct_call;
    const int nch = P.nch3;
    const int zc_all = d.residual ? (int)__ldcg(&P.zone_cnt[b]) : 0;
    FinState f;
    f.rh = 1.0f;
    f.rl = 0.0f;
    f.tlh = f.tll = 0.0f;
    f.cstar = -1;
    f.lastpos_chunk = -1;
    f.residual = d.residual;
    bool done = false;
    if (nch * (int)sizeof(ChunkTot) <= kPassRingBytes && zc_all <= 32) {
        done = finalize_fast(P, b, d, r, nch, P.draw_chunk + (int64_t)b * nch,
                             P.zone + (int64_t)b * kZoneMax, zc_all, ring, lane, f.rh, f.rl,
                             f.cstar, f.lastpos_chunk, f.tlh, f.tll);
    }
    if (!done) finalize_general<DT>(P, b, d, r, tab, ct, lane, f);
    finalize_rescan<DT>(P, b, d, r, tab, ct, ring, lane, f);
}

}  // namespace sv
