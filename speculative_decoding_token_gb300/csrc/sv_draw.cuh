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
//
// Pass task: one warp per (sequence, chunk of 8192 tokens); lane L owns the
// contiguous span of 256 tokens starting at chunk + 256 L. Each lane
// accumulates S_p, S_q and, over the tokens whose sign is certain under the
// row-statistics estimate of rho (window 2^-15), P_A = sum e_p and
// Q_A = sum e_q of the positive ones; the few tokens inside the window are
// listed. The p and q exponentials run on packed f32x2 pairs (a bonus draw
// pairs two tokens of the p row). Outputs: one record per lane span and the
// chunk's totals.
//
// Finalize task: one warp per sequence forms the exact rho, the chunk masses
// P_A - rho Q_A (+ the listed tokens, settled exactly), locates t = u R among
// the chunks, then among the 32 lane spans of that chunk, and rescans the one
// 256-token span token by token. A list overflow or an estimate outside the
// window makes it recompute the masses with the exact rho instead (slow path,
// flagged).
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
__device__ __forceinline__ Quad ld_quad(const Quad *p) {
    const double2 a = __ldcg(reinterpret_cast<const double2 *>(p));
    const double2 b = __ldcg(reinterpret_cast<const double2 *>(p) + 1);
    return Quad{a.x, a.y, b.x, b.y};
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
// per-sequence setup shared by the two kernels

struct DrawRows {
    const char *prow, *qrow;
    ExpRow er;         // residual: halves (p, q); bonus: both halves p
    bool shift;        // some row needs the general (shifted) exponential
    double rho_est;    // row-statistics estimate of S_p / S_q in the shifted scale
};

__device__ __forceinline__ DrawRows draw_rows(const Params &P, const DrawDesc &d) {
    DrawRows r;
    r.prow = P.target + d.p_phys * P.stride_bytes;
    r.qrow = d.residual ? P.draft + d.q_phys * P.stride_bytes : r.prow;
    const double c2 = (double)P.c2h + (double)P.c2l;
    const double mp = (double)d.Mp * c2;
    const double mq = d.residual ? (double)d.Mq * c2 : mp;
    // logits far from 0 in the 2^(l c) scale take an integer shift
    r.shift = !(fabs(mp) <= 60.0 && fabs(mq) <= 60.0);
    const float ip = r.shift ? (float)rint(mp) : 0.0f;
    const float iq = r.shift ? (float)rint(mq) : 0.0f;
    r.er.ch = splat2(P.c2h);
    r.er.cl = splat2(P.c2l);
    r.er.shift = pack2(ip, d.residual ? iq : ip);
    const float span = (float)(1000.0 / c2);
    r.er.lmin = pack2(d.Mp - span, d.residual ? d.Mq - span : d.Mp - span);
    // S' = S * 2^(M c - I) in the shifted scale of each row
    r.rho_est = d.residual ? ((double)d.Sp / (double)d.Sq) *
                                 exp2((mp - (double)ip) - (mq - (double)iq))
                           : 1.0;
    return r;
}

// ---------------------------------------------------------------------------
// pass task

__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ double warp_incl_scan_d(double x, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    return x;
}

// one token of a residual pass: S_p, S_q always; P_A, Q_A when the sign of
// e_p - rho e_q is certain under the estimated rho; else list the token
__device__ __forceinline__ void residual_token(const Params &P, int b, int64_t v, f32x2 eh, f32x2 el,
                                               float rhi, float rlo, f32x2 &sh, f32x2 &sl,
                                               f32x2 &ah, f32x2 &al) {
    acc2(sh, sl, eh, el);
    const float2 h = unpack2(eh);
    if (h.x > rhi * h.y) {
        acc2(ah, al, eh, el);
    } else if (h.y > 0.0f && h.x >= rlo * h.y) {
        const uint32_t slot = atomicAdd(&P.zone_cnt[b], 1u);
        if (slot < (uint32_t)kZoneMax) {
            const float2 lw = unpack2(el);
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
}

// weights of a group of 8 tokens from their logits, then accumulated
template <bool kShift>
__device__ __forceinline__ void group_general(const Params &P, const DrawRows &r, int b, int64_t v,
                                              const float *xp, const float *xq, bool residual,
                                              const float2 *tab, float rhi, float rlo, f32x2 &sh,
                                              f32x2 &sl, f32x2 &ah, f32x2 &al) {
    if (residual) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            f32x2 eh, el;
            exp2_pair<kShift>(pack2(xp[e], xq[e]), r.er, tab, eh, el);
            residual_token(P, b, v + e, eh, el, rhi, rlo, sh, sl, ah, al);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            f32x2 eh, el;
            exp2_pair<kShift>(pack2(xp[e], xp[e + 1]), r.er, tab, eh, el);
            acc2(sh, sl, eh, el);
        }
    }
}

__device__ __forceinline__ Quad span_record(bool residual, f32x2 sh, f32x2 sl, f32x2 ah, f32x2 al) {
    const float2 h = unpack2(sh), l = unpack2(sl);
    if (residual) {
        const float2 a = unpack2(ah), b2 = unpack2(al);
        return Quad{ff_to_double(h.x, l.x), ff_to_double(h.y, l.y), ff_to_double(a.x, b2.x),
                    ff_to_double(a.y, b2.y)};
    }
    return Quad{ff_to_double(h.x, l.x) + ff_to_double(h.y, l.y), 0.0, 0.0, 0.0};
}

// The pass over tokens [v0, v1) of one lane, computing every weight.
template <int DT, bool kShift>
__device__ void pass_span(const Params &P, const DrawRows &r, int b, int64_t v0, int64_t v1,
                          const float2 *tab, bool residual, Quad &rec) {
    f32x2 sh = 0ull, sl = 0ull;  // (S_p, S_q), or two halves of S_p for a bonus draw
    f32x2 ah = 0ull, al = 0ull;  // (P_A, Q_A)
    const float rhi = (float)(r.rho_est * (1.0 + kRhoWindow));
    const float rlo = (float)(r.rho_est * (1.0 - kRhoWindow));
    float xp[8], xq[8];
    if (v0 < v1) {
        load8<DT>(r.prow, v0, P.V, xp);
        if (residual) load8<DT>(r.qrow, v0, P.V, xq);
    }
    for (int64_t v = v0; v < v1; v += 8) {
        float np[8], nq[8];
        const bool more = v + 8 < v1;
        if (more) {  // the next group's loads are in flight while this one computes
            load8<DT>(r.prow, v + 8, P.V, np);
            if (residual) load8<DT>(r.qrow, v + 8, P.V, nq);
        }
        group_general<kShift>(P, r, b, v, xp, xq, residual, tab, rhi, rlo, sh, sl, ah, al);
        if (more) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                xp[e] = np[e];
                if (residual) xq[e] = nq[e];
            }
        }
    }
    rec = span_record(residual, sh, sl, ah, al);
}

// table index of the bf16 code in the low 16 bits of c; >= kCodeHalf (after
// masking with kCodeHalf - 1 removed) when outside the table
__device__ __forceinline__ uint32_t code_offset(uint32_t c) { return (c & 0x7FFFu) - kCodeBase; }
__device__ __forceinline__ uint32_t code_index(uint32_t c) {
    return code_offset(c) | ((c >> 4) & (uint32_t)kCodeHalf);
}

__device__ __forceinline__ void codes8(const uint4 &w, uint32_t *c) {
    c[0] = w.x & 0xFFFFu; c[1] = w.x >> 16;
    c[2] = w.y & 0xFFFFu; c[3] = w.y >> 16;
    c[4] = w.z & 0xFFFFu; c[5] = w.z >> 16;
    c[6] = w.w & 0xFFFFu; c[7] = w.w >> 16;
}

__device__ __forceinline__ void floats8(const uint4 &w, float *x) {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x);
    x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z);
    x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
}

// The pass over tokens [v0, v1) of a bf16 row pair without shift: a group of
// 8 tokens whose codes all lie in the weight table reads its weights from it
// (the same float-float values the exponential gives); other groups compute
// them. Accumulation order is the same either way.
template <bool kRes>
__device__ void pass_span_bf16(const Params &P, const DrawRows &r, int b, int64_t v0, int64_t v1,
                               const float2 *tab, const float2 *ct, Quad &rec) {
    f32x2 sh = 0ull, sl = 0ull, ah = 0ull, al = 0ull;
    const float rhi = (float)(r.rho_est * (1.0 + kRhoWindow));
    const float rlo = (float)(r.rho_est * (1.0 - kRhoWindow));
    // end of the full groups (a lane whose span starts at or past V has none)
    const int64_t vend = v1 > v0 ? v0 + ((v1 - v0) & ~(int64_t)7) : v1;
    const uint4 *pp = reinterpret_cast<const uint4 *>(r.prow);
    const uint4 *qq = reinterpret_cast<const uint4 *>(r.qrow);
    uint4 wp = make_uint4(0, 0, 0, 0), wq = make_uint4(0, 0, 0, 0);
    if (v0 < vend) {
        wp = __ldg(pp + v0 / 8);
        if (kRes) wq = __ldg(qq + v0 / 8);
    }
    for (int64_t v = v0; v < vend; v += 8) {
        uint4 np, nq;
        const bool more = v + 8 < vend;
        if (more) {
            np = __ldg(pp + v / 8 + 1);
            if (kRes) nq = __ldg(qq + v / 8 + 1);
        }
        uint32_t cp[8], cq[8];
        codes8(wp, cp);
        if (kRes) codes8(wq, cq);
        uint32_t out = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            out |= code_offset(cp[e]);
            if (kRes) out |= code_offset(cq[e]);
        }
        if (out < (uint32_t)kCodeHalf) {
            if (kRes) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 a = ct[code_index(cp[e])];
                    const float2 c = ct[code_index(cq[e])];
                    residual_token(P, b, v + e, pack2(a.x, c.x), pack2(a.y, c.y), rhi, rlo, sh, sl,
                                   ah, al);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 a = ct[code_index(cp[e])];
                    const float2 c = ct[code_index(cp[e + 1])];
                    acc2(sh, sl, pack2(a.x, c.x), pack2(a.y, c.y));
                }
            }
        } else {
            float xp[8], xq[8];
            floats8(wp, xp);
            if (kRes) floats8(wq, xq);
            group_general<false>(P, r, b, v, xp, xq, kRes, tab, rhi, rlo, sh, sl, ah, al);
        }
        if (more) {
            wp = np;
            if (kRes) wq = nq;
        }
    }
    if (vend < v1) {  // the ragged end of the row
        float xp[8], xq[8];
        load8<SV_DT_BF16>(r.prow, vend, P.V, xp);
        if (kRes) load8<SV_DT_BF16>(r.qrow, vend, P.V, xq);
        group_general<false>(P, r, b, vend, xp, xq, kRes, tab, rhi, rlo, sh, sl, ah, al);
    }
    rec = span_record(kRes, sh, sl, ah, al);
}

// The pass over chunk c of sequence b: lane records and the chunk totals.
// ct: the bf16 weight table of this call, or null.
template <int DT>
__device__ void pass_task(const Params &P, int b, int c, const DrawDesc &d, const float2 *tab,
                          const float2 *ct, int lane) {
    const DrawRows r = draw_rows(P, d);
    const int64_t v0 = (int64_t)c * kDrawChunk + (int64_t)lane * kDrawSpan;
    const int64_t v1 = min(P.V, v0 + kDrawSpan);
    Quad rec;
    if (DT == SV_DT_BF16 && ct != nullptr && !r.shift) {
        if (d.residual)
            pass_span_bf16<true>(P, r, b, v0, v1, tab, ct, rec);
        else
            pass_span_bf16<false>(P, r, b, v0, v1, tab, ct, rec);
    } else if (r.shift) {
        pass_span<DT, true>(P, r, b, v0, v1, tab, d.residual, rec);
    } else {
        pass_span<DT, false>(P, r, b, v0, v1, tab, d.residual, rec);
    }
    const int64_t item = (int64_t)b * P.nch3 + c;
    P.draw_part[item * 32 + lane] = rec;
    const Quad tot{warp_sum_d(rec.x), warp_sum_d(rec.y), warp_sum_d(rec.z), warp_sum_d(rec.w)};
    if (lane == 0) P.draw_chunk[item] = tot;
}

// The bf16 weight table of a call: entry i holds the weight that the
// exponential above gives for the bf16 logit of code
// (i mod kCodeHalf) + kCodeBase, negated when i >= kCodeHalf, in a row
// without shift. Entries whose exponent l c lies outside [-1000, 127] are 0:
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
        ct[2 * i] = ok0 ? make_float2(h.x, l.x) : make_float2(0.0f, 0.0f);
        ct[2 * i + 1] = ok1 ? make_float2(h.y, l.y) : make_float2(0.0f, 0.0f);
    }
}

// ---------------------------------------------------------------------------
// finalize task

// exact weight of token v (v in [0, V)) under the final rho
template <int DT, bool kShift>
__device__ __forceinline__ void exact_weight(const DrawRows &r, int64_t v, bool residual, float rh,
                                             float rl, const float2 *tab, float &wh, float &wl) {
    const float lp = load_logit<DT>(r.prow, v);
    if (!residual) {
        f32x2 eh, el;
        exp2_pair<kShift>(pack2(lp, lp), r.er, tab, eh, el);
        wh = unpack2(eh).x;
        wl = unpack2(el).x;
        return;
    }
    const float lq = load_logit<DT>(r.qrow, v);
    f32x2 eh, el;
    exp2_pair<kShift>(pack2(lp, lq), r.er, tab, eh, el);
    const float2 h = unpack2(eh), l = unpack2(el);
    residual_weight(h.x, l.x, h.y, l.y, rh, rl, wh, wl);
}

// Sum of the exact weights of tokens [v0, v1) by one lane.
template <int DT, bool kShift>
__device__ double exact_span_sum(const DrawRows &r, int64_t v0, int64_t v1, bool residual, float rh,
                                 float rl, const float2 *tab) {
    float sh = 0.0f, sl = 0.0f;
    for (int64_t v = v0; v < v1; ++v) {
        float wh, wl;
        exact_weight<DT, kShift>(r, v, residual, rh, rl, tab, wh, wl);
        ff_accumulate(sh, sl, wh, wl);
    }
    return ff_to_double(sh, sl);
}

template <int DT, bool kShift>
__device__ void finalize_seq(const Params &P, int b, const DrawDesc &d, const DrawRows &r,
                             const float2 *tab, int lane) {
    const int nch = P.nch3;
    const Quad *chunk = P.draw_chunk + (int64_t)b * nch;
    const Quad *part = P.draw_part + (int64_t)b * nch * 32;
    double *mass = P.draw_mass + (int64_t)b * nch;
    ZoneEntry *zs = P.zone + (int64_t)b * kZoneMax;
    double sp = 0.0, sq = 0.0;
    for (int c = lane; c < nch; c += 32) {
        const Quad q = ld_quad(&chunk[c]);
        sp += q.x;
        sq += q.y;
    }
    sp = warp_sum_d(sp);
    sq = warp_sum_d(sq);
    int residual = d.residual;
    const double rho = residual ? sp / sq : 1.0;
    const float rh = (float)rho;
    const float rl = (float)(rho - (double)rh);
    const int zc_all = residual ? (int)__ldcg(&P.zone_cnt[b]) : 0;
    const bool slow = residual && (zc_all > kZoneMax ||
                                   !(fabs(rho / r.rho_est - 1.0) <= 0.5 * kRhoWindow));
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
    auto zone_add = [&](int c, int L, double m) -> double {
        for (int i = 0; i < zc; ++i) {
            const ZoneEntry z = ld_zone(&zs[i]);
            if (z.v / kDrawChunk == c && (L < 0 || (z.v % kDrawChunk) / kDrawSpan == L)) {
                const double w = ff_to_double(z.eph, z.epl) - rho * ff_to_double(z.eqh, z.eql);
                if (w > 0.0) m += w;
            }
        }
        return m;
    };

    // chunk masses (in the scratch row `mass`) and their total R
    double R = 0.0;
    if (slow) {
        for (int c = 0; c < nch; ++c) {
            const int64_t v0 = (int64_t)c * kDrawChunk + (int64_t)lane * kDrawSpan;
            const double m = warp_sum_d(
                exact_span_sum<DT, kShift>(r, v0, min(P.V, v0 + kDrawSpan), true, rh, rl, tab));
            if (lane == 0) __stcg(&mass[c], m);
            R += m;
        }
    } else {
        double part_r = 0.0;
        for (int c = lane; c < nch; c += 32) {
            const Quad q = ld_quad(&chunk[c]);
            const double m = residual ? zone_add(c, -1, q.z - rho * q.w) : q.x;
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
    int cstar = -1, lastpos_chunk = -1;
    double before = 0.0;
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
    bool takelast = false;
    if (cstar < 0) {  // t at or past the end through rounding: the last positive mass
        takelast = true;
        cstar = lastpos_chunk < 0 ? 0 : lastpos_chunk;
    }
    double tl = t - before;
    // the lane span within chunk c*
    double lm;
    if (slow && residual) {
        const int64_t v0 = (int64_t)cstar * kDrawChunk + (int64_t)lane * kDrawSpan;
        lm = exact_span_sum<DT, kShift>(r, v0, min(P.V, v0 + kDrawSpan), true, rh, rl, tab);
    } else {
        const Quad q = ld_quad(&part[(int64_t)cstar * 32 + lane]);
        lm = residual ? zone_add(cstar, lane, q.z - rho * q.w) : q.x;
    }
    const double lincl = warp_incl_scan_d(lm, lane);
    const uint32_t lhit = takelast ? 0u : __ballot_sync(0xffffffffu, lincl > tl);
    const uint32_t lpos = __ballot_sync(0xffffffffu, lm > 0.0);
    int Lstar;
    if (lhit) {
        Lstar = __ffs(lhit) - 1;
        tl -= __shfl_sync(0xffffffffu, lincl - lm, Lstar);
    } else {
        takelast = true;
        Lstar = lpos ? 31 - __clz(lpos) : 0;
    }
    // rescan that span: lane j owns tokens s0 + 8j .. s0 + 8j + 7
    const int64_t s0 = (int64_t)cstar * kDrawChunk + (int64_t)Lstar * kDrawSpan;
    const int64_t v0 = s0 + 8 * lane, v1 = min(min(P.V, s0 + kDrawSpan), v0 + 8);
    float w8h[8], w8l[8];
    double mine = 0.0;
    int lastpos = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        w8h[e] = 0.0f;
        w8l[e] = 0.0f;
        if (v0 + e < v1) {
            exact_weight<DT, kShift>(r, v0 + e, residual, rh, rl, tab, w8h[e], w8l[e]);
            mine += ff_to_double(w8h[e], w8l[e]);
            if (w8h[e] > 0.0f) lastpos = (int)(v0 + e);
        }
    }
    const double incl = warp_incl_scan_d(mine, lane);
    int k = -1;
    if (!takelast) {
        const double start = incl - mine;
        if (start <= tl && tl < incl) {
            double C = start;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                C += ff_to_double(w8h[e], w8l[e]);
                if (k < 0 && v0 + e < v1 && C > tl) k = (int)(v0 + e);
            }
        }
    }
    int kk = k;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kk = max(kk, __shfl_xor_sync(0xffffffffu, kk, off));
    int lp = lastpos;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, off));
    if (lane == 0)
        P.tok_out[(int64_t)b * (P.gamma_max + 1) + d.n] = kk >= 0 ? kk : (lp >= 0 ? lp : (int)s0);
}

template <int DT>
__device__ void finalize_task(const Params &P, int b, const DrawDesc &d, const float2 *tab,
                              int lane) {
    const DrawRows r = draw_rows(P, d);
    if (r.shift)
        finalize_seq<DT, true>(P, b, d, r, tab, lane);
    else
        finalize_seq<DT, false>(P, b, d, r, tab, lane);
}

}  // namespace sv
