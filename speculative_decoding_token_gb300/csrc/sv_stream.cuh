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
            const double lp = load_logit<DT>(P.target + rp * P.stride_bytes, x);
            const double lq = load_logit<DT>(P.draft + rq * P.stride_bytes, x);
            // log p_i(x) - log q_i(x) with p = exp((l - M)/T) / S
            const double d = ((lp - (double)sp.x) - (lq - (double)sq.x)) * P.invT -
                             (log((double)sp.y) - log((double)sq.y));
            const double ratio = exp(d);
            const double r = accept_uniform(P.seed, (uint32_t)b, (uint32_t)(i + 1));
            rej = r > ratio;
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
        // Exponent scale of the draw: rows whose max lies far from 0 in the
        // 2^(l c) scale (c = log2(e)/T) take integer shifts; rho_est is
        // S_p / S_q from the row statistics, in that shifted scale.
        const double c2 = (double)P.c2h + (double)P.c2l;
        const double mp = (double)d.Mp * c2;
        const double mq = d.residual ? (double)d.Mq * c2 : mp;
        d.shift = !(fabs(mp) <= 60.0 && fabs(mq) <= 60.0);
        d.ip = d.shift ? (float)rint(mp) : 0.0f;
        d.iq = d.shift ? (float)rint(mq) : 0.0f;
        d.pad = 0;
        d.rho_est = d.residual ? ((double)d.Sp / (double)d.Sq) *
                                     exp2((mp - (double)d.ip) - (mq - (double)d.iq))
                               : 1.0;
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

// The (max, sum) statistics of rows base .. base + rows - 1, one lane per
// row combining that row's chunk partials in chunk order; writes row_stat
// and, when requested, the row's logsumexp.
__device__ inline void combine_rows_sample(const Params &P, int base, int rows, int lane) {
    const int cpr = P.cpr;
    for (int r = lane; r < rows; r += 32) {
        const int lrow = base + r;
        const float2 *pp = P.partials + (int64_t)lrow * cpr;
        float m = -INFINITY, s = 0.0f;
        bool nan = false;
        for (int c0 = 0; c0 < cpr; c0 += 8) {
            float2 pc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                pc[k] = c0 + k < cpr ? __ldcg(&pp[c0 + k]) : make_float2(-INFINITY, 0.0f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (pc[k].x != pc[k].x || pc[k].y != pc[k].y) {
                    nan = true;
                } else if (pc[k].x > m) {
                    s = (m == -INFINITY ? 0.0f : s * ex2_approx((m - pc[k].x) * P.c2)) + pc[k].y;
                    m = pc[k].x;
                } else if (pc[k].x != -INFINITY) {
                    s += pc[k].y * ex2_approx((pc[k].x - m) * P.c2);
                }
            }
        }
        const bool bad = nan || !(m > -INFINITY && m < INFINITY) || !(s > 0.0f) || s == INFINITY;
        const float qnan = __int_as_float(0x7fffffff);
        P.row_stat[lrow] = bad ? make_float2(qnan, qnan) : make_float2(m, s);
        const RowRef rr = P.rows[lrow];
        float *lse_out = rr.j >= 0 ? P.p_lse : P.q_lse;
        if (lse_out)
            lse_out[rr.phys] = bad ? qnan : (float)((double)m * P.invT + log((double)s));
    }
}

// ---------------------------------------------------------------------------
// hand-offs inside the fused kernel (bounded waits; a wait that gives up
// marks the call aborted so that every other wait returns at once)

constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ bool call_aborted(const Params &P) {
    return *reinterpret_cast<const volatile uint32_t *>(P.abort_flag) == P.epoch;
}

__device__ __forceinline__ void abort_call(const Params &P) {
    atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
    atomicExch(P.abort_flag, P.epoch);
}

// every lane polls its share of the chunk partials [begin, begin + count)
__device__ inline bool wait_partials(const Params &P, int64_t begin, int64_t count, int lane) {
    uint32_t ok = 1;
    const uint64_t t0 = global_ns();
    for (int64_t i = lane; i < count && ok; i += 32) {
        while (ld_relaxed_f2(&P.partials[begin + i]).y == kPartialPending) {
            __nanosleep(100);
            if (call_aborted(P) || global_ns() - t0 > kWaitNs) {
                ok = 0;
                break;
            }
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) abort_call(P);
    __threadfence();  // the polled partials are read again after this
    return ok != 0;
}

__device__ __forceinline__ void publish(uint32_t *flag, uint32_t epoch, int lane) {
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        st_release_u32(flag, epoch);
    }
}

// The accept step of sequence b inside the fused kernel, run by the warp
// that stored the sequence's last chunk partial: wait until every partial of
// its rows is visible, combine the rows, run the accept scan, publish.
template <int DT>
__device__ void accept_seq(const Params &P, int b, int lane) {
    const int rows = P.seq_rows[b];
    const int base = P.seq_base[b];
    if (rows > 0 && wait_partials(P, (int64_t)base * P.cpr, (int64_t)rows * P.cpr, lane)) {
        combine_rows_sample(P, base, rows, lane);
        __syncwarp();
        accept_scan_sampling<DT>(P, b, lane);
    }
    publish(&P.seq_flag[b], P.epoch, lane);
}

// Claims and runs the next accept step if its sequence is ready (accept
// steps are claimed in sequence order). Returns whether it ran one.
template <int DT>
__device__ bool try_accept(const Params &P, int lane) {
    uint32_t claimed = 0xFFFFFFFFu;
    if (lane == 0) {
        const uint32_t a = *reinterpret_cast<const volatile uint32_t *>(P.acc_next);
        if (a < (uint32_t)P.B && ld_acquire_u32(&P.seq_ready[a]) == P.epoch &&
            atomicCAS(P.acc_next, a, a + 1u) == a)
            claimed = a;
    }
    claimed = __shfl_sync(0xffffffffu, claimed, 0);
    if (claimed == 0xFFFFFFFFu) return false;
    accept_seq<DT>(P, (int)claimed, lane);
    return true;
}

// Waits (the whole warp) until *f holds this call's epoch, running ready
// accept steps meanwhile; false once the call is aborted or after about two
// seconds.
template <int DT>
__device__ bool wait_flag_helping(const Params &P, const uint32_t *f, int lane) {
    const uint64_t t0 = global_ns();
    for (;;) {
        uint32_t ok = 0;
        if (lane == 0) ok = ld_acquire_u32(f) == P.epoch ? 1u : 0u;
        if (__shfl_sync(0xffffffffu, ok, 0)) break;
        if (try_accept<DT>(P, lane)) continue;
        __nanosleep(200);
        uint32_t give_up = 0;
        if (lane == 0) give_up = (call_aborted(P) || global_ns() - t0 > kWaitNs) ? 1u : 0u;
        if (__shfl_sync(0xffffffffu, give_up, 0)) {
            if (lane == 0) abort_call(P);
            return false;
        }
    }
    __syncwarp();
    return true;
}

// Stream the items gw, gw + NW, ... of the batch through this warp's ring of
// NS shared-memory stages of SB bytes (wbuf, barriers at bar0, initialised by the
// caller) and store one partial per item: (max, sum) in sampling mode
// (MODE 0), (best value, argmax) in greedy mode (MODE 1). The store is a
// relaxed 64-bit store over the sentinel the plan kernel wrote, so a consumer
// in the same launch can poll for it; the warp never waits on other warps.
template <int DT, int MODE, int NS, int SB, bool kReady>
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
        if (kReady && lane == 0) {
            // the warp that stores a sequence's last chunk partial marks it ready
            const int32_t sb = P.rows[lrow].b;
            const uint32_t need = (uint32_t)P.seq_rows[sb] * (uint32_t)cpr;
            if (atomicAdd(&P.seq_cnt[sb], 1u) + 1u == need) st_release_u32(&P.seq_ready[sb], P.epoch);
        }
    }
    if (timed_out) {
        if (lane == 0) {
            if (kReady)
                abort_call(P);
            else
                atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
        }
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
