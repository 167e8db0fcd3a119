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

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait: gives up after about two seconds of wall time
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u && global_ns() - t0 > 2000000000ull) return false;
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

// Stream the items gw, gw + NW, ... of the batch through this warp's ring of
// kStages shared-memory stages (wbuf, barriers at bar0, initialised by the
// caller) and store one partial per item: (max, sum) in sampling mode
// (MODE 0), (best value, argmax) in greedy mode (MODE 1). The store is a
// relaxed 64-bit store over the sentinel the plan kernel wrote, so a consumer
// in the same launch can poll for it; the warp never waits on other warps.
template <int DT, int MODE>
__device__ void stream_items(const Params &P, uint8_t *wbuf, uint32_t bar0, int64_t gw,
                             int64_t NW, int lane) {
    constexpr int ESZ = DT == SV_DT_FP32 ? 4 : 2;
    constexpr int PV = Elem<DT>::kPerVec;
    constexpr int kVecPerLane = kStageBytes / 16 / 32;  // 8
    const int64_t cpr = P.cpr;
    const int64_t n_items = (int64_t)(*P.total_rows) * cpr;

    auto row_base = [&](const RowRef &rr) -> const char * {
        return (rr.j >= 0 ? P.target : P.draft) + rr.phys * P.stride_bytes;
    };
    auto item_bytes = [&](int64_t chunk) -> int64_t {
        return min((int64_t)kItemBytes, P.row_bytes - chunk * kItemBytes);
    };

    // Producer cursor, identical in every lane. The row descriptor of the
    // warp's next item is loaded one item ahead, so issuing a stage never
    // waits on a global load.
    int64_t p_item = gw;
    int p_st = 0, p_nst = 0;
    const char *p_src = nullptr;
    int64_t p_bytes = 0;
    RowRef p_next{};
    auto p_enter = [&](const RowRef &rr) {
        const int64_t chunk = p_item % cpr;
        p_src = row_base(rr) + chunk * kItemBytes;
        p_bytes = item_bytes(chunk);
        p_nst = (int)((p_bytes + kStageBytes - 1) / kStageBytes);
        p_st = 0;
        if (p_item + NW < n_items) p_next = P.rows[(p_item + NW) / cpr];
    };
    if (p_item < n_items) p_enter(P.rows[p_item / cpr]);
    uint32_t pcnt = 0;
    auto issue_next = [&]() {
        if (p_item >= n_items) return;
        const int64_t off = (int64_t)p_st * kStageBytes;
        const uint32_t tma = (uint32_t)min((int64_t)kStageBytes, p_bytes - off) & ~15u;
        if (lane == 0) {
            const int slot = pcnt % kStages;
            const uint32_t bar = bar0 + 8 * slot;
            if (tma > 0) {
                mbar_arrive_expect_tx(bar, tma);
                bulk_load(smem_u32(wbuf + slot * kStageBytes), p_src + off, tma, bar);
            } else {
                mbar_arrive(bar);
            }
        }
        ++pcnt;
        if (++p_st == p_nst) {
            p_item += NW;
            if (p_item < n_items) p_enter(p_next);
        }
    };
    for (int s = 0; s < kStages; ++s) issue_next();

    SampleAcc sa = sample_acc_init();
    GreedyAcc ga{-INFINITY, -1};
    uint32_t ccnt = 0;
    bool timed_out = false;
    for (int64_t item = gw; item < n_items; item += NW) {
        const int64_t lrow = item / cpr;
        const int64_t chunk = item - lrow * cpr;
        const int64_t ibytes = item_bytes(chunk);
        const int nst = (int)((ibytes + kStageBytes - 1) / kStageBytes);
        for (int st = 0; st < nst; ++st) {
            const int slot = ccnt % kStages;
            if (!mbar_wait_bounded(bar0 + 8 * slot, (ccnt / kStages) & 1u)) {
                timed_out = true;
                break;
            }
            const int64_t off = (int64_t)st * kStageBytes;
            const int64_t bytes = min((int64_t)kStageBytes, ibytes - off);
            const int nvec = (int)(bytes >> 4);
            const uint4 *vb = reinterpret_cast<const uint4 *>(wbuf + slot * kStageBytes);
            const int64_t elem0 = (chunk * kItemBytes + off) / ESZ;
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
                const int rem = (int)(bytes & 15) / ESZ;
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
            issue_next();
        }
        if (timed_out) break;
        // chunk partial
        float2 part;
        if (MODE == 0) {
            float s = sample_acc_sum(sa);
            // a sum overflowed: an element lay far above its lane's reference
            if (__any_sync(0xffffffffu, s == INFINITY)) {
                sample_chunk_exact<DT>(sa, row_base(P.rows[lrow]), chunk * kItemBytes / ESZ,
                                       (chunk * kItemBytes + ibytes) / ESZ, lane, P.c2);
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
            const int slot = ccnt % kStages;
            if (!mbar_wait_bounded(bar0 + 8 * slot, (ccnt / kStages) & 1u)) break;
            ++ccnt;
        }
    }
}

}  // namespace sv
