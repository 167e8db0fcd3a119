// sv_stream.cuh -- the streaming side of the verify step: per-warp rings of
// bulk asynchronous copies into shared memory, per-lane online softmax
// statistics (sampling) or first argmax (greedy), chunk partials, the row
// combine and the accept scans. Shared by the row-statistics kernels and the
// fused sampling kernel.
#pragma once

#include "sv_common.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// shared-memory barriers and bulk copies

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The waiting thread is suspended until the phase completes or about
// kSuspendNs pass, so a waiting warp issues almost nothing.
constexpr uint32_t kSuspendNs = 100000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// bounded wait: gives up after about two seconds of wall time
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > 2000000000ull) return false;
    }
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------------------
// per-lane accumulators

struct SampleAcc {
    float m;        // reference logit (a lane maximum; see sample_group)
    f32x2 p0, p1;   // four partial sums of 2^((l - m) c2), packed in pairs
    float sx;       // contributions of the ragged row tail
};

__device__ __forceinline__ SampleAcc sample_acc_init() {
    return SampleAcc{-INFINITY, 0ull, 0ull, 0.0f};
}

__device__ __forceinline__ float sample_acc_sum(const SampleAcc &a) {
    const float2 x = unpack2(a.p0), y = unpack2(a.p1);
    return ((x.x + x.y) + (y.x + y.y)) + a.sx;
}

struct GreedyAcc {
    float best;     // best raw logit (NaN once a NaN was seen)
    int32_t idx;    // its element index in the row
};

template <int DT>
struct Elem;
template <>
struct Elem<SV_DT_FP32> {
    static constexpr int kPerVec = 4;
};
template <>
struct Elem<SV_DT_BF16> {
    static constexpr int kPerVec = 8;
};

// unpack one 16-byte vector into floats
template <int DT>
__device__ __forceinline__ void unpack(const uint4 &w, float *f) {
    if (DT == SV_DT_FP32) {
        f[0] = __uint_as_float(w.x);
        f[1] = __uint_as_float(w.y);
        f[2] = __uint_as_float(w.z);
        f[3] = __uint_as_float(w.w);
    } else {
        f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
        f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
        f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
        f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
    }
}

// NaN-propagating max of n floats as a balanced tree (short dependency chains)
template <int N>
__device__ __forceinline__ float tree_max(const float *f) {
    float t[N];
#pragma unroll
    for (int e = 0; e < N; ++e) t[e] = f[e];
#pragma unroll
    for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
        for (int e = 0; e < w; ++e) t[e] = max_nan(t[e], t[e + w]);
    return t[0];
}

// Feed a group of NV 16-byte vectors (already in registers) to the sampling
// accumulator. The reference a.m need not be the running maximum: the sums
// hold sum 2^((l - a.m) c2) for any a.m, so only the first finite group of a
// lane in a chunk takes its exact maximum. A later element far above a.m
// overflows the sum to +inf, which the chunk end detects and redoes exactly;
// a NaN propagates into the sum (a bad row). The FMA and the additions run on
// packed float pairs.
template <int DT, int NV>
__device__ __forceinline__ void sample_group(SampleAcc &a, const uint4 *w, float c2) {
    constexpr int PV = Elem<DT>::kPerVec;
    if (a.m == -INFINITY) {
        float f[NV * PV];
#pragma unroll
        for (int u = 0; u < NV; ++u) unpack<DT>(w[u], f + u * PV);
        const float g = tree_max<NV * PV>(f);
        if (g != g || g == INFINITY) {  // NaN or +inf logit: poison the sum
            a.sx = __int_as_float(0x7fffffff);
            return;
        }
        if (g == -INFINITY) return;     // nothing but -inf so far
        a.m = g;
    }
    const float mc = a.m * c2;
    const f32x2 c2x2 = pack2(c2, c2);
    const f32x2 nmc = pack2(-mc, -mc);
    f32x2 acc0 = a.p0, acc1 = a.p1;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const uint32_t wd[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
        if (DT == SV_DT_BF16) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 x = unpack2(fma2(pack2(bf16_lo(wd[k]), bf16_hi(wd[k])), c2x2, nmc));
                const f32x2 e = pack2(ex2_approx(x.x), ex2_approx(x.y));
                if (k & 1) acc1 = add2(acc1, e); else acc0 = add2(acc0, e);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; k += 2) {
                const float2 x = unpack2(
                    fma2(pack2(__uint_as_float(wd[k]), __uint_as_float(wd[k + 1])), c2x2, nmc));
                const f32x2 e = pack2(ex2_approx(x.x), ex2_approx(x.y));
                if (k & 2) acc1 = add2(acc1, e); else acc0 = add2(acc0, e);
            }
        }
    }
    a.p0 = acc0;
    a.p1 = acc1;
}

// Exact (max, sum) of one chunk by the whole warp, lane-strided over the
// chunk's elements from global memory: the rare path taken when a lane's sum
// overflowed because an element lay far above its reference.
template <int DT>
__device__ void sample_chunk_exact(SampleAcc &a, const char *row, int64_t e_begin, int64_t e_end,
                                   int lane, float c2) {
    float m = -INFINITY;
    for (int64_t e = e_begin + lane; e < e_end; e += 32) m = max_nan(m, load_logit<DT>(row, e));
    float s = 0.0f;
    if (m != m || m == INFINITY) {
        s = __int_as_float(0x7fffffff);
    } else if (m != -INFINITY) {
        for (int64_t e = e_begin + lane; e < e_end; e += 32)
            s += ex2_approx((load_logit<DT>(row, e) - m) * c2);
    }
    a = sample_acc_init();
    a.m = m;
    a.sx = s;
}

template <int DT, int NV>
__device__ __forceinline__ void greedy_group(GreedyAcc &a, const uint4 *w, int64_t first_elem,
                                             int lane) {
    constexpr int PV = Elem<DT>::kPerVec;
    float f[NV * PV];
#pragma unroll
    for (int u = 0; u < NV; ++u) unpack<DT>(w[u], f + u * PV);
    const float g = tree_max<NV * PV>(f);
    if (g != g) {
        a.best = g;  // NaN: sticky
        return;
    }
    if (a.best != a.best) return;
    if (g > a.best || a.idx < 0) {
        // first element equal to the group max, in increasing index order
        int32_t hit = -1;
#pragma unroll
        for (int u = NV - 1; u >= 0; --u)
#pragma unroll
            for (int e = PV - 1; e >= 0; --e)
                if (f[u * PV + e] == g) hit = u * 32 * PV + e;
        a.best = g;
        a.idx = (int32_t)(first_elem + lane * PV + hit);
    }
}

// ---------------------------------------------------------------------------
// warp reductions of the accumulators

__device__ __forceinline__ float2 warp_combine_sample(float m, float s, float c2) {
    float M = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = max_nan(M, __shfl_xor_sync(0xffffffffu, M, off));
    float t = (m == -INFINITY) ? 0.0f : s * ex2_approx((m - M) * c2);
    if (M != M || s != s) t = __int_as_float(0x7fffffff);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    return make_float2(M, t);
}

__device__ __forceinline__ float2 warp_combine_greedy(float best, int32_t idx) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, off);
        const int32_t oi = __shfl_xor_sync(0xffffffffu, idx, off);
        const bool take = (ob != ob) ? true
                          : (best != best) ? false
                          : (oi >= 0 && (idx < 0 || ob > best || (ob == best && oi < idx)));
        if (take) {
            best = ob;
            idx = oi;
        }
    }
    return make_float2(best, __int_as_float(idx));
}

// ---------------------------------------------------------------------------
// accept scans (one warp per sequence)

// The acceptance threshold f(p_k(x), eps) / q_k(x) ("DistillSpec" Algorithm
// A.1; f(p) = p when lossless, the lenience functions of its Sec. 4
// "DistillSpec with lossy SD" otherwise) from the logits of x and the row
// statistics (M, S), p = exp((l - M)/T) / S. FP64 is a narrow pipe on this
// part, so the arithmetic is float and float-float: the logit differences are
// exact (TwoSum), their scaling by 1/T keeps ~44 bits, and only the logs of
// the sums (or of their quotient) and the final exponential round at float
// precision, ~1e-6 of the ratio, far inside the accept test's flag band.
// f_lin and f_sq add len_c = -log eps or -2 log eps to log p; f_exp scales
// log p by len_c = eps.
__device__ __forceinline__ float accept_ratio(const Params &P, float lp, float lq, float2 sp,
                                              float2 sq) {
    float dph, dpl, dqh, dql;  // l - M, exactly
    two_sum(lp, -sp.x, dph, dpl);
    two_sum(lq, -sq.x, dqh, dql);
    if (P.len_kind == SPECVERIFY_LENIENCE_EXP) {
        float aph, apl, aqh, aql, eh, el;
        ff_mul(dph, dpl, P.invTh, P.invTl, aph, apl);
        ff_mul(dqh, dql, P.invTh, P.invTl, aqh, aql);
        ff_add(aph, apl, -logf(sp.y), 0.0f, aph, apl);  // log p
        ff_add(aqh, aql, -logf(sq.y), 0.0f, aqh, aql);  // log q
        ff_mul(aph, apl, P.len_cf, 0.0f, aph, apl);
        ff_add(aph, apl, -aqh, -aql, eh, el);
        return expf(eh + el);
    }
    float xh, xl, dh, dl;
    ff_add(dph, dpl, -dqh, -dql, xh, xl);
    ff_mul(xh, xl, P.invTh, P.invTl, dh, dl);
    float d = (dh - logf(sp.y / sq.y)) + dl;
    if (P.len_kind != SPECVERIFY_LENIENCE_NONE) d += P.len_cf;
    return expf(d);
}

// The draw's exponent scale and rho estimate of d (Mp, Sp, Mq, Sq, residual
// set): rows whose max lies far from 0 in the 2^(l c) scale (c = log2(e)/T)
// take integer shifts, and rho_est is S_p / S_q from the row statistics in
// that scale. The products M c are float-float, so the exponent difference
// stays exact to ~1e-12 whatever the logits' magnitude.
__device__ __forceinline__ void set_draw_scale(const Params &P, DrawDesc &d) {
    float mph, mpl, mqh, mql;
    ff_mul(d.Mp, 0.0f, P.c2h, P.c2l, mph, mpl);
    if (d.residual) {
        ff_mul(d.Mq, 0.0f, P.c2h, P.c2l, mqh, mql);
    } else {
        mqh = mph;
        mql = mpl;
    }
    d.shift = !(fabsf(mph) <= 60.0f && fabsf(mqh) <= 60.0f);
    d.ip = d.shift ? rintf(mph) : 0.0f;
    d.iq = d.shift ? rintf(mqh) : 0.0f;
    d.pad = 0;
    d.pad2 = 0;
    // (mp - ip) - (mq - iq): both heads lie within 1/2 of their integer, so
    // the head differences are exact
    const float e = ((mph - d.ip) - (mqh - d.iq)) + (mpl - mql);
    d.rho_est = d.residual ? (d.Sp / d.Sq) * exp2f(e) : 1.0f;
}

template <int DT>
__device__ void accept_scan_sampling(const Params &P, int b, int lane) {
    const int g = P.gamma[b];
    const int base = P.seq_base[b];
    const int gm = P.gamma_max;
    bool bad = false;
    for (int r = lane; r < 2 * g + 1; r += 32) {
        const float2 st = __ldcg(&P.row_stat[base + r]);
        bad |= (st.y != st.y);
    }
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) atomicOr(P.status, SPECVERIFY_STATUS_BAD_LOGIT);
        return;  // n_out, tokens and draw stay -1 from the plan kernel
    }
    int n = g;
    for (int i0 = 0; i0 < g; i0 += 32) {
        const int i = i0 + lane;
        bool rej = false;
        if (i < g) {
            const int32_t x = __ldg(&P.tokens[(int64_t)b * gm + i]);
            const float2 sp = __ldcg(&P.row_stat[base + i]);
            const float2 sq = __ldcg(&P.row_stat[base + g + 1 + i]);
            const int64_t rp = P.rows[base + i].phys;
            const int64_t rq = P.rows[base + g + 1 + i].phys;
            const float lp = load_logit<DT>(P.target + rp * P.stride_bytes, x);
            const float lq = load_logit<DT>(P.draft + rq * P.stride_bytes, x);
            const float ratio = accept_ratio(P, lp, lq, sp, sq);
            rej = accept_uniform(P.seed, (uint32_t)b, (uint32_t)(i + 1)) > ratio;
        }
        const uint32_t mask = __ballot_sync(0xffffffffu, rej);
        if (mask) {
            n = i0 + __ffs(mask) - 1;
            break;
        }
    }
    for (int i = lane; i < n; i += 32)
        P.tok_out[(int64_t)b * (gm + 1) + i] = __ldg(&P.tokens[(int64_t)b * gm + i]);
    if (lane == 0) {
        DrawDesc d;
        d.n = n;
        d.residual = n < g ? 1 : 0;
        const float2 sp = __ldcg(&P.row_stat[base + n]);
        d.p_phys = P.rows[base + n].phys;
        d.Mp = sp.x;
        d.Sp = sp.y;
        if (n < g) {
            const float2 sq = __ldcg(&P.row_stat[base + g + 1 + n]);
            d.q_phys = P.rows[base + g + 1 + n].phys;
            d.Mq = sq.x;
            d.Sq = sq.y;
        } else {
            d.q_phys = -1;
            d.Mq = 0.0f;
            d.Sq = 1.0f;
        }
        set_draw_scale(P, d);
        P.draw[b] = d;
        P.n_out[b] = n;
    }
}

__device__ inline void accept_scan_greedy(const Params &P, int b, int lane) {
    const int g = P.gamma[b];
    const int base = P.seq_base[b];
    const int gm = P.gamma_max;
    bool bad = false;
    for (int r = lane; r <= g; r += 32) {
        const float2 st = __ldcg(&P.row_stat[base + r]);
        bad |= (st.x != st.x);
    }
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) atomicOr(P.status, SPECVERIFY_STATUS_BAD_LOGIT);
        return;
    }
    int n = g;
    for (int i0 = 0; i0 < g; i0 += 32) {
        const int i = i0 + lane;
        bool mism = false;
        if (i < g) {
            const int32_t a = __float_as_int(__ldcg(&P.row_stat[base + i]).y);
            mism = __ldg(&P.tokens[(int64_t)b * gm + i]) != a;
        }
        const uint32_t mask = __ballot_sync(0xffffffffu, mism);
        if (mask) {
            n = i0 + __ffs(mask) - 1;
            break;
        }
    }
    for (int i = lane; i < n; i += 32)
        P.tok_out[(int64_t)b * (gm + 1) + i] = __ldg(&P.tokens[(int64_t)b * gm + i]);
    if (lane == 0) {
        P.tok_out[(int64_t)b * (gm + 1) + n] = __float_as_int(__ldcg(&P.row_stat[base + n]).y);
        P.n_out[b] = n;
    }
}

// ---------------------------------------------------------------------------
// row combine: one warp folds the chunk partials of logical row lrow, in a
// fixed order, into the row statistics (and the optional lse output)

template <int MODE>
__device__ void combine_row(const Params &P, int lrow, int lane) {
    const RowRef rr = P.rows[lrow];
    float2 res;
    if (MODE == 0) {
        float m = -INFINITY, s = 0.0f;
        for (int c = lane; c < P.cpr; c += 32) {
            const float2 pc = __ldcg(&P.partials[(int64_t)lrow * P.cpr + c]);
            if (pc.x != pc.x || pc.y != pc.y) {
                m = pc.x;
                s = __int_as_float(0x7fffffff);
            } else if (pc.x > m) {
                s = (m == -INFINITY ? 0.0f : s * ex2_approx((m - pc.x) * P.c2)) + pc.y;
                m = pc.x;
            } else if (pc.x != -INFINITY) {
                s += pc.y * ex2_approx((pc.x - m) * P.c2);
            }
        }
        res = warp_combine_sample(m, s, P.c2);
        const bool bad = !(res.x > -INFINITY && res.x < INFINITY) || !(res.y > 0.0f) ||
                         res.y == INFINITY;
        if (bad) res = make_float2(__int_as_float(0x7fffffff), __int_as_float(0x7fffffff));
        if (lane == 0) {
            float *lse_out = rr.j >= 0 ? P.p_lse : P.q_lse;
            if (lse_out)
                lse_out[rr.phys] = bad ? __int_as_float(0x7fffffff)
                                       : (float)((double)res.x * P.invT + log((double)res.y));
        }
    } else {
        float best = -INFINITY;
        int32_t idx = -1;
        for (int c = lane; c < P.cpr; c += 32) {
            const float2 pc = __ldcg(&P.partials[(int64_t)lrow * P.cpr + c]);
            const int32_t pi = __float_as_int(pc.y);
            if (pc.x != pc.x) {
                best = pc.x;
            } else if (best == best && pi >= 0 &&
                       (idx < 0 || pc.x > best)) {  // chunks visited in index order
                best = pc.x;
                idx = pi;
            }
        }
        res = warp_combine_greedy(best, idx);
    }
    if (lane == 0) P.row_stat[lrow] = res;
}

// One step of the chunk-order combine of a row's (max, sum) partials.
__device__ __forceinline__ void combine_step(float2 pc, float c2, float &m, float &s, bool &nan) {
    if (pc.x != pc.x || pc.y != pc.y) {
        nan = true;
    } else if (pc.x > m) {
        s = (m == -INFINITY ? 0.0f : s * ex2_approx((m - pc.x) * c2)) + pc.y;
        m = pc.x;
    } else if (pc.x != -INFINITY) {
        s += pc.y * ex2_approx((pc.x - m) * c2);
    }
}

// Stores the statistics of logical row lrow (NaN: bad row) and, when
// requested, its logsumexp; returns them.
__device__ __forceinline__ float2 finish_row(const Params &P, int lrow, float m, float s, bool nan) {
    const bool bad = nan || !(m > -INFINITY && m < INFINITY) || !(s > 0.0f) || s == INFINITY;
    const float qnan = __int_as_float(0x7fffffff);
    const float2 st = bad ? make_float2(qnan, qnan) : make_float2(m, s);
    P.row_stat[lrow] = st;
    if (P.p_lse || P.q_lse) {
        const RowRef rr = P.rows[lrow];
        float *lse_out = rr.j >= 0 ? P.p_lse : P.q_lse;
        if (lse_out) lse_out[rr.phys] = bad ? qnan : (float)((double)m * P.invT + log((double)s));
    }
    return st;
}

// The (max, sum) statistics of logical row lrow by one thread, combining
// the row's chunk partials in chunk order.
__device__ inline float2 combine_one_row(const Params &P, int lrow) {
    const int cpr = P.cpr;
    const float2 *pp = P.partials + (int64_t)lrow * cpr;
    float m = -INFINITY, s = 0.0f;
    bool nan = false;
    for (int c0 = 0; c0 < cpr; c0 += 8) {
        float2 pc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            pc[k] = c0 + k < cpr ? __ldcg(&pp[c0 + k]) : make_float2(-INFINITY, 0.0f);
#pragma unroll
        for (int k = 0; k < 8; ++k) combine_step(pc[k], P.c2, m, s, nan);
    }
    return finish_row(P, lrow, m, s, nan);
}

// The statistics of rows base .. base + rows - 1, one lane per row.
__device__ inline void combine_rows_sample(const Params &P, int base, int rows, int lane) {
    for (int r = lane; r < rows; r += 32) combine_one_row(P, base + r);
}

// ---------------------------------------------------------------------------
// hand-offs inside the fused kernel (bounded waits; a wait that gives up
// marks the call aborted so that every other wait returns at once)

// Default bound of a wait on another warp of the fused kernel (the call's
// Params.wait_ns; specverify_set_wait_limit changes it). The waits of a warp
// on its own bulk copies keep their fixed two-second bound, so no kernel
// exits with a copy in flight.
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ bool call_aborted(const Params &P) {
    return *reinterpret_cast<const volatile uint32_t *>(P.abort_flag) == P.epoch;
}

__device__ __forceinline__ void abort_call(const Params &P) {
    atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
    atomicExch(P.abort_flag, P.epoch);
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t *p) {
    return *reinterpret_cast<const volatile uint32_t *>(p);
}

__device__ __forceinline__ void publish(uint32_t *flag, uint32_t epoch, int lane) {
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        st_release_u32(flag, epoch);
    }
}

// Appends item v to a queue (lane 0 only): reserve a slot, then publish it
// as one 64-bit word (this call's epoch, the item) with release order.
__device__ __forceinline__ void queue_push(const Params &P, unsigned long long *slots,
                                           int tail_ctr, uint32_t v) {
    const uint32_t slot = atomicAdd(&P.ctr[tail_ctr * kCtrStride], 1u);
    st_release_u64(&slots[slot], ((unsigned long long)P.epoch << 32) | v);
}

// A warp's claim on one queue slot. Slots are claimed by ticket (an atomic
// increment of the queue's head) only while the head is behind the tail, so
// claims spread over the slots without retries; a claimed slot is served
// once its pusher has published it.
struct Ticket {
    uint32_t slot;
    bool held;
    bool dead;  // the queue is exhausted for this warp
};

constexpr uint32_t kNoItem = 0xFFFFFFFFu;

__device__ __forceinline__ void ticket_take(const Params &P, int head_ctr, int tail_ctr,
                                            uint32_t capacity, Ticket &t, int lane) {
    if (t.held || t.dead) return;
    uint32_t s = kNoItem;
    if (lane == 0 && ld_volatile_u32(&P.ctr[head_ctr * kCtrStride]) < ld_volatile_u32(&P.ctr[tail_ctr * kCtrStride]))
        s = atomicAdd(&P.ctr[head_ctr * kCtrStride], 1u);
    s = __shfl_sync(0xffffffffu, s, 0);
    if (s == kNoItem) return;
    if (s >= capacity) {
        t.dead = true;
    } else {
        t.slot = s;
        t.held = true;
    }
}

// The item of the warp's ticket once its slot is published, else kNoItem.
__device__ __forceinline__ uint32_t ticket_item(const Params &P, const unsigned long long *slots,
                                                Ticket &t, int lane) {
    if (!t.held) return kNoItem;
    uint32_t v = kNoItem;
    if (lane == 0) {
        const unsigned long long w = ld_acquire_u64(&slots[t.slot]);
        if ((uint32_t)(w >> 32) == P.epoch) v = (uint32_t)w;
    }
    v = __shfl_sync(0xffffffffu, v, 0);
    if (v != kNoItem) t.held = false;
    return v;
}

// A ticket taken without looking at the tail (the slot may be pushed later).
__device__ __forceinline__ void ticket_take_ahead(const Params &P, int head_ctr, uint32_t capacity,
                                                  Ticket &t, int lane) {
    if (t.held || t.dead) return;
    uint32_t s = 0;
    if (lane == 0) s = atomicAdd(&P.ctr[head_ctr * kCtrStride], 1u);
    s = __shfl_sync(0xffffffffu, s, 0);
    if (s >= capacity) {
        t.dead = true;
    } else {
        t.slot = s;
        t.held = true;
    }
}

// Stream the items gw, gw + NW, ... of the batch through this warp's ring of
// NS shared-memory stages of SB bytes (wbuf, barriers at bar0, initialised by the
// caller) and store one partial per item: (max, sum) in sampling mode
// (MODE 0), (best value, argmax) in greedy mode (MODE 1). The store is a
// relaxed 64-bit store over the sentinel the plan kernel wrote, so a consumer
// in the same launch can poll for it; the warp never waits on other warps.
template <int DT, int MODE, int NS, int SB>
__device__ void stream_items(const Params &P, uint8_t *wbuf, uint32_t bar0, int64_t gw,
                             int64_t NW, int lane) {
    constexpr int ESZ = DT == SV_DT_FP32 ? 4 : 2;
    constexpr int PV = Elem<DT>::kPerVec;
    constexpr int kVecPerLane = SB / 16 / 32;
    const int32_t cpr = P.cpr;
    const int64_t total_rows = *P.total_rows;
    // item = lrow * cpr + chunk; the warp visits items gw, gw + NW, ... as
    // (row, chunk) cursors advanced by NW without divisions
    const int64_t dq = NW / cpr;
    const int32_t dr = (int32_t)(NW - dq * cpr);
    auto advance = [&](int64_t &lrow, int32_t &chunk) {
        lrow += dq;
        chunk += dr;
        if (chunk >= cpr) {
            chunk -= cpr;
            ++lrow;
        }
    };
    const int64_t lrow0 = gw / cpr;
    const int32_t chunk0 = (int32_t)(gw - lrow0 * cpr);
    if (lrow0 >= total_rows) return;

    auto row_base = [&](const RowRef &rr) -> const char * {
        return (rr.j >= 0 ? P.target : P.draft) + rr.phys * P.stride_bytes;
    };
    auto item_bytes = [&](int32_t chunk) -> int32_t {
        return (int32_t)min((int64_t)kItemBytes, P.row_bytes - (int64_t)chunk * kItemBytes);
    };

    // Producer cursor, identical in every lane. The row descriptor of the
    // warp's next item is loaded one item ahead, so issuing a stage never
    // waits on a global load.
    int64_t p_lrow = lrow0, n_lrow = 0;
    int32_t p_chunk = chunk0, n_chunk = 0;
    bool p_live = true;
    int p_st = 0, p_nst = 0, p_slot = 0;
    const char *p_src = nullptr;
    int32_t p_bytes = 0;
    RowRef p_next{};
    auto p_enter = [&](const RowRef &rr) {
        p_src = row_base(rr) + (int64_t)p_chunk * kItemBytes;
        p_bytes = item_bytes(p_chunk);
        p_nst = (p_bytes + SB - 1) / SB;
        p_st = 0;
        n_lrow = p_lrow;
        n_chunk = p_chunk;
        advance(n_lrow, n_chunk);
        if (n_lrow < total_rows) p_next = P.rows[n_lrow];
    };
    p_enter(P.rows[p_lrow]);
    uint32_t pcnt = 0;
    auto issue_next = [&]() {
        if (!p_live) return;
        const int32_t off = p_st * SB;
        const uint32_t tma = (uint32_t)min(SB, p_bytes - off) & ~15u;
        if (lane == 0) {
            const uint32_t bar = bar0 + 8 * p_slot;
            if (tma > 0) {
                mbar_arrive_expect_tx(bar, tma);
                bulk_load(smem_u32(wbuf + p_slot * SB), p_src + off, tma, bar);
            } else {
                mbar_arrive(bar);
            }
        }
        ++pcnt;
        if (++p_slot == NS) p_slot = 0;
        if (++p_st == p_nst) {
            p_lrow = n_lrow;
            p_chunk = n_chunk;
            if (p_lrow < total_rows)
                p_enter(p_next);
            else
                p_live = false;
        }
    };
    for (int s = 0; s < NS; ++s) issue_next();

    SampleAcc sa = sample_acc_init();
    GreedyAcc ga{-INFINITY, -1};
    uint32_t ccnt = 0, c_phase = 0;
    int c_slot = 0;
    bool timed_out = false;
    int64_t lrow = lrow0;
    int32_t chunk = chunk0;
    for (; lrow < total_rows; advance(lrow, chunk)) {
        const int32_t ibytes = item_bytes(chunk);
        const int nst = (ibytes + SB - 1) / SB;
        const int64_t ebase = (int64_t)chunk * (kItemBytes / ESZ);
        for (int st = 0; st < nst; ++st) {
            if (!mbar_wait_bounded(bar0 + 8 * c_slot, c_phase)) {
                timed_out = true;
                break;
            }
            const int32_t bytes = min(SB, ibytes - st * SB);
            const int nvec = bytes >> 4;
            const uint4 *vb = reinterpret_cast<const uint4 *>(wbuf + c_slot * SB);
            const int64_t elem0 = ebase + (int64_t)st * (SB / ESZ);
            if (nvec == kVecPerLane * 32) {
#pragma unroll
                for (int t = 0; t < kVecPerLane; t += 4) {
                    uint4 w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) w[u] = vb[lane + 32 * (t + u)];
                    if (MODE == 0)
                        sample_group<DT, 4>(sa, w, P.c2);
                    else
                        greedy_group<DT, 4>(ga, w, elem0 + (int64_t)t * 32 * PV, lane);
                }
            } else {
#pragma unroll
                for (int t = 0; t < kVecPerLane; t += 4) {
                    uint4 w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int idx = lane + 32 * (t + u);
                        // padding: -inf (fp32 0xff800000, bf16 pair 0xff80ff80)
                        w[u] = idx < nvec ? vb[idx]
                                          : (DT == SV_DT_FP32
                                                 ? make_uint4(0xff800000u, 0xff800000u,
                                                              0xff800000u, 0xff800000u)
                                                 : make_uint4(0xff80ff80u, 0xff80ff80u,
                                                              0xff80ff80u, 0xff80ff80u));
                    }
                    if (MODE == 0)
                        sample_group<DT, 4>(sa, w, P.c2);
                    else
                        greedy_group<DT, 4>(ga, w, elem0 + (int64_t)t * 32 * PV, lane);
                }
                // ragged tail of the row (fewer than 16 bytes): plain loads
                const int rem = (bytes & 15) / ESZ;
                if (rem > 0 && lane < rem) {
                    const int64_t e = elem0 + (int64_t)nvec * PV + lane;
                    const float v = load_logit<DT>(row_base(P.rows[lrow]), e);
                    if (MODE == 0) {
                        if (v != v || v == INFINITY) {
                            sa.sx = __int_as_float(0x7fffffff);
                        } else if (v != -INFINITY) {
                            if (sa.m == -INFINITY) sa.m = v;
                            sa.sx += ex2_approx((v - sa.m) * P.c2);
                        }
                    } else if (v != v) {
                        ga.best = v;
                    } else if (ga.best == ga.best && (ga.idx < 0 || v > ga.best)) {
                        // tail elements come after every other element of this lane
                        ga.best = v;
                        ga.idx = (int32_t)e;
                    }
                }
            }
            __syncwarp();
            ++ccnt;
            if (++c_slot == NS) {
                c_slot = 0;
                c_phase ^= 1u;
            }
            issue_next();
        }
        if (timed_out) break;
        // chunk partial
        float2 part;
        if (MODE == 0) {
            float s = sample_acc_sum(sa);
            // a sum overflowed: an element lay far above its lane's reference
            if (__any_sync(0xffffffffu, s == INFINITY)) {
                sample_chunk_exact<DT>(sa, row_base(P.rows[lrow]), ebase, ebase + ibytes / ESZ,
                                       lane, P.c2);
                s = sample_acc_sum(sa);
            }
            part = warp_combine_sample(sa.m, s, P.c2);
        } else {
            part = warp_combine_greedy(ga.best, ga.idx);
        }
        sa = sample_acc_init();
        ga = GreedyAcc{-INFINITY, -1};
        if (lane == 0) st_relaxed_f2(&P.partials[lrow * cpr + chunk], part);
    }
    if (timed_out) {
        if (lane == 0) atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
        // drain the copies already issued into this warp's ring (bounded)
        while (ccnt < pcnt) {
            if (!mbar_wait_bounded(bar0 + 8 * c_slot, c_phase)) break;
            ++ccnt;
            if (++c_slot == NS) {
                c_slot = 0;
                c_phase ^= 1u;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// the fused kernel's stream: position-major rows, optional skipping

// What a ring slot holds, written by the producer (lane 0) before the copy
// and read by every lane after the slot's barrier completes.
struct __align__(16) StageMeta {
    int32_t lrow;   // logical row; -1: the stream has ended
    int32_t chunk;  // chunk of the row
    int32_t bytes;  // bytes in this stage
    int32_t e0;     // element index of the stage's first logit in the row
    int32_t b, pos; // sequence and position of the row
    int32_t need;   // chunk partials completing the position
    int32_t last;   // 1 on the chunk's last stage
};

// Streams items of the position-major order (item = order slot * cpr +
// chunk), claimed by ticket, through this warp's
// ring of NS stages of SB bytes and stores one chunk partial per streamed
// item (NW: the streaming warps of the grid). When P.skip is set,
// an item whose sequence is already known to be rejected at an earlier
// position is skipped: rows after a sequence's first rejection are never
// needed. The warp that stores the last partial of a position queues the
// position for its test. The warp never waits on other warps.
template <int DT, int NS, int SB>
__device__ void stream_needed(const Params &P, uint8_t *wbuf, StageMeta *meta, uint32_t bar0,
                              int64_t NW, int lane) {
    constexpr int ESZ = DT == SV_DT_FP32 ? 4 : 2;
    constexpr int PV = Elem<DT>::kPerVec;
    constexpr int kVecPerLane = SB / 16 / 32;
    const int32_t cpr = P.cpr;
    // the order holds every logical row of the call once (total_rows entries)
    const int64_t n_items = (int64_t)(*P.total_rows) * cpr;
    if (n_items == 0) return;

    // Items are handed out by ticket, kStreamWin items a ticket: dealt round
    // robin (streaming warp gw takes tickets gw, gw + NW, gw + 2 NW, ...) or
    // claimed one at a time from a shared counter (see take_ticket). The window holds two tickets, one item per lane:
    // lanes [0, K) the current ticket, lanes [K, 2K) the next one, whose order
    // entries are loaded a ticket ahead; the ticket after that is known too. Each lane keeps its item's row and
    // its sequence's first rejection, refreshed at every stage, so entering
    // an item never waits on memory.
    constexpr int K = kStreamWin;
    static_assert(2 * K <= 32, "two tickets of window items");
    const int32_t kNoRej = P.G + 1;
    int widx = K;
    OrderRef wr{};
    int32_t wchunk = 0, wrej = kNoRej;
    bool wvalid = false, wfresh = false;  // wfresh: wrej has been read
    // ticket c into lanes [lo, lo + K). Item indices of every realistic
    // batch fit in 31 bits, where 32-bit divisions replace the much slower
    // 64-bit ones (this runs once per ticket, on the streaming path).
    const bool narrow = n_items + 4 * (int64_t)K * NW < ((int64_t)1 << 31);
    const uint32_t nw32 = (uint32_t)NW, cpr32 = (uint32_t)cpr;
    auto load_ticket = [&](int64_t c, int lo) {
        if (lane >= lo && lane < lo + K) {
            int64_t t, oi;
            if (narrow) {
                const uint32_t c32 = (uint32_t)c;
                const uint32_t blk = c32 / nw32;
                t = (int64_t)(blk * (uint32_t)K * nw32 + (c32 - blk * nw32) +
                              (uint32_t)(lane - lo) * nw32);
            } else {
                const int64_t blk = c / NW;
                t = blk * K * NW + (c - blk * NW) + (int64_t)(lane - lo) * NW;
            }
            wvalid = t < n_items;
            wrej = kNoRej;
            wfresh = false;
            if (wvalid) {
                oi = narrow ? (int64_t)((uint32_t)t / cpr32) : t / cpr;
                wchunk = (int32_t)(t - oi * cpr);
                wr = P.order[oi];
            }
        }
    };
    uint32_t claim = 0;
    // Tickets are dealt round robin when each warp gets few items (no shared
    // counter: measured 2-5 % faster), and claimed from one counter when each
    // gets many (with over a hundred items a warp, the luck of the skips
    // leaves some warps far behind the others: measured 6 % slower dealt).
    const bool dealt = n_items <= (int64_t)kDealtItemsPerWarp * NW;
    uint32_t next_ticket = blockIdx.x * (uint32_t)(NW / gridDim.x) + (threadIdx.x >> 5);
    auto take_ticket = [&]() -> uint32_t {  // lane 0
        if (!dealt) return atomicAdd(&P.ctr[kCtrTicket * kCtrStride], 1u);
        const uint32_t c = next_ticket;
        next_ticket += (uint32_t)NW;
        return c;
    };
    if (lane == 0) claim = take_ticket();
    load_ticket((int64_t)__shfl_sync(0xffffffffu, claim, 0), K);
    if (lane == 0) claim = take_ticket();
    // the first rejection of every item still ahead (a load whose value is
    // used at a later item entry)
    auto refresh = [&](int from) {
        if (P.skip && lane >= from && lane < 2 * K && wvalid) {
            wrej = *reinterpret_cast<const volatile int32_t *>(&P.first_rej[wr.b]);
            wfresh = true;
        }
    };
    refresh(K);
    // the next ticket becomes the current one; returns false past the end
    auto refill = [&]() -> bool {
        const long long phys = __shfl_down_sync(0xffffffffu, (long long)wr.phys, K);
        const int32_t b = __shfl_down_sync(0xffffffffu, wr.b, K);
        const int32_t j = __shfl_down_sync(0xffffffffu, wr.j, K);
        const int32_t lrow = __shfl_down_sync(0xffffffffu, wr.lrow, K);
        const int32_t pos = __shfl_down_sync(0xffffffffu, wr.pos, K);
        const int32_t need = __shfl_down_sync(0xffffffffu, wr.need, K);
        const int32_t ch = __shfl_down_sync(0xffffffffu, wchunk, K);
        const int32_t rj = __shfl_down_sync(0xffffffffu, wrej, K);
        const bool v = __shfl_down_sync(0xffffffffu, wvalid ? 1 : 0, K) != 0;
        const bool fr = __shfl_down_sync(0xffffffffu, wfresh ? 1 : 0, K) != 0;
        if (lane < K) {
            wr.phys = phys;
            wr.b = b;
            wr.j = j;
            wr.lrow = lrow;
            wr.pos = pos;
            wr.need = need;
            wchunk = ch;
            wrej = rj;
            wvalid = v;
            wfresh = fr;
            // skipped tickets in a row leave no stage to refresh in: read now
            if (P.skip && v && !fr) {
                wrej = *reinterpret_cast<const volatile int32_t *>(&P.first_rej[wr.b]);
                wfresh = true;
            }
        }
        load_ticket((int64_t)__shfl_sync(0xffffffffu, claim, 0), K);
        if (lane == 0) claim = take_ticket();
        widx = 0;
        // the first item of a ticket past the end: every later ticket is too
        return __shfl_sync(0xffffffffu, wvalid ? 1 : 0, 0) != 0;
    };

    // producer, identical in every lane
    bool p_done = false, p_end_sent = false;
    int p_st = 0, p_nst = 0, p_slot = 0;
    const char *p_src = nullptr;
    int32_t p_bytes = 0, p_lrow = 0, p_chunk = 0, p_b = 0, p_pos = 0, p_need = 0;
    auto p_enter = [&]() {
        for (;;) {
            if (widx == K && !refill()) {
                p_done = true;
                return;
            }
            if (!__shfl_sync(0xffffffffu, wvalid ? 1 : 0, widx)) {  // past the end
                widx = K;
                continue;
            }
            const int k = widx++;
            const int32_t pos = __shfl_sync(0xffffffffu, wr.pos, k);
            // rejected at an earlier position: this row is not needed
            if (P.skip && __shfl_sync(0xffffffffu, wrej, k) < pos) continue;
            p_pos = pos;
            p_b = __shfl_sync(0xffffffffu, wr.b, k);
            p_lrow = __shfl_sync(0xffffffffu, wr.lrow, k);
            p_need = __shfl_sync(0xffffffffu, wr.need, k);
            p_chunk = __shfl_sync(0xffffffffu, wchunk, k);
            const int32_t j = __shfl_sync(0xffffffffu, wr.j, k);
            const long long phys = __shfl_sync(0xffffffffu, (long long)wr.phys, k);
            p_src = (j >= 0 ? P.target : P.draft) + (int64_t)phys * P.stride_bytes +
                    (int64_t)p_chunk * kItemBytes;
            p_bytes = (int32_t)min((int64_t)kItemBytes, P.row_bytes - (int64_t)p_chunk * kItemBytes);
            p_nst = (p_bytes + SB - 1) / SB;
            p_st = 0;
            return;
        }
    };
    p_enter();
    uint32_t pcnt = 0;
    auto issue_next = [&]() {
        if (p_done) {
            if (!p_end_sent) {  // the end marker takes one slot
                if (lane == 0) {
                    meta[p_slot].lrow = -1;
                    mbar_arrive(bar0 + 8 * p_slot);
                }
                p_end_sent = true;
                ++pcnt;
                if (++p_slot == NS) p_slot = 0;
            }
            return;
        }
        const int32_t off = p_st * SB;
        const int32_t bytes = min(SB, p_bytes - off);
        const uint32_t tma = (uint32_t)bytes & ~15u;
        if (lane == 0) {
            StageMeta m;
            m.lrow = p_lrow;
            m.chunk = p_chunk;
            m.bytes = bytes;
            m.e0 = (p_chunk * kItemBytes + off) / ESZ;
            m.b = p_b;
            m.pos = p_pos;
            m.need = p_need;
            m.last = p_st + 1 == p_nst ? 1 : 0;
            meta[p_slot] = m;
            const uint32_t bar = bar0 + 8 * p_slot;
            if (tma > 0) {
                mbar_arrive_expect_tx(bar, tma);
                bulk_load(smem_u32(wbuf + p_slot * SB), p_src + off, tma, bar);
            } else {
                mbar_arrive(bar);
            }
        }
        ++pcnt;
        if (++p_slot == NS) p_slot = 0;
        if (++p_st == p_nst) p_enter();
    };
    for (int s = 0; s < NS; ++s) issue_next();

    SampleAcc sa = sample_acc_init();
    uint32_t ccnt = 0, c_phase = 0;
    int c_slot = 0;
    bool timed_out = false;
    // The count of a finished item's position is read back one stage later
    // (lane 0), so the atomic's round trip overlaps the next stage; the warp
    // whose increment completed the position queues its test.
    uint32_t pend_pi = kNoItem, pend_old = 0u, pend_need = 0u;
    auto settle = [&]() {
        if (lane == 0 && pend_pi != kNoItem) {
            if (pend_old + 1u == pend_need) queue_push(P, P.rq_slot, kCtrRqTail, pend_pi);
            pend_pi = kNoItem;
        }
    };
    for (;;) {
        if (!mbar_wait_bounded(bar0 + 8 * c_slot, c_phase)) {
            timed_out = true;
            break;
        }
        const StageMeta m = meta[c_slot];
        if (m.lrow < 0) break;
        refresh(widx);
        const int nvec = m.bytes >> 4;
        const uint4 *vb = reinterpret_cast<const uint4 *>(wbuf + c_slot * SB);
        if (nvec == kVecPerLane * 32) {
#pragma unroll
            for (int t = 0; t < kVecPerLane; t += 4) {
                uint4 w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) w[u] = vb[lane + 32 * (t + u)];
                sample_group<DT, 4>(sa, w, P.c2);
            }
        } else {
#pragma unroll
            for (int t = 0; t < kVecPerLane; t += 4) {
                uint4 w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int idx = lane + 32 * (t + u);
                    // padding: -inf (fp32 0xff800000, bf16 pair 0xff80ff80)
                    w[u] = idx < nvec ? vb[idx]
                                      : (DT == SV_DT_FP32 ? make_uint4(0xff800000u, 0xff800000u,
                                                                       0xff800000u, 0xff800000u)
                                                          : make_uint4(0xff80ff80u, 0xff80ff80u,
                                                                       0xff80ff80u, 0xff80ff80u));
                }
                sample_group<DT, 4>(sa, w, P.c2);
            }
            // ragged tail of the row (fewer than 16 bytes): plain loads
            const int rem = (m.bytes & 15) / ESZ;
            if (rem > 0 && lane < rem) {
                const RowRef rr = P.rows[m.lrow];
                const char *row = (rr.j >= 0 ? P.target : P.draft) + rr.phys * P.stride_bytes;
                const float v = load_logit<DT>(row, (int64_t)m.e0 + (int64_t)nvec * PV + lane);
                if (v != v || v == INFINITY) {
                    sa.sx = __int_as_float(0x7fffffff);
                } else if (v != -INFINITY) {
                    if (sa.m == -INFINITY) sa.m = v;
                    sa.sx += ex2_approx((v - sa.m) * P.c2);
                }
            }
        }
        __syncwarp();
        ++ccnt;
        if (++c_slot == NS) {
            c_slot = 0;
            c_phase ^= 1u;
        }
        issue_next();
        settle();
        if (!m.last) continue;
        // chunk partial
        float s = sample_acc_sum(sa);
        if (__any_sync(0xffffffffu, s == INFINITY)) {
            // a sum overflowed: an element lay far above its lane's reference
            const RowRef rr = P.rows[m.lrow];
            const char *row = (rr.j >= 0 ? P.target : P.draft) + rr.phys * P.stride_bytes;
            const int64_t e_begin = (int64_t)m.chunk * (kItemBytes / ESZ);
            const int64_t e_end = min((int64_t)(m.chunk + 1) * (kItemBytes / ESZ), P.V);
            sample_chunk_exact<DT>(sa, row, e_begin, e_end, lane, P.c2);
            s = sample_acc_sum(sa);
        }
        const float2 part = warp_combine_sample(sa.m, s, P.c2);
        sa = sample_acc_init();
        if (lane == 0) {
            st_relaxed_f2(&P.partials[(int64_t)m.lrow * cpr + m.chunk], part);
            pend_pi = (uint32_t)m.b * (uint32_t)P.G + (uint32_t)(m.pos - 1);
            pend_need = (uint32_t)m.need;
            pend_old = atomicAdd(&P.pos_cnt[pend_pi], 1u);
        }
    }
    settle();
    if (timed_out) {
        if (lane == 0) abort_call(P);
        // drain the copies already issued into this warp's ring (bounded)
        while (ccnt < pcnt) {
            if (!mbar_wait_bounded(bar0 + 8 * c_slot, c_phase)) break;
            ++ccnt;
            if (++c_slot == NS) {
                c_slot = 0;
                c_phase ^= 1u;
            }
        }
    }
}

}  // namespace sv
