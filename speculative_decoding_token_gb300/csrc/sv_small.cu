// sv_small.cu -- the sampling verify step for small batches: one thread-block
// cluster of kSmallCtas CTAs per sequence, the whole step in one launch
// without a grid barrier, a queue or a cross-CTA wait of its own.
//
// The same step as the fused kernel ("DistillSpec" Sec. 3 and App. A.3
// Algorithm A.1; the Leviathan et al. explainer's rule for n; lenience per
// "DistillSpec" Sec. 4), laid out for a batch whose rows fit a few SMs' worth
// of loads: CTA c of a sequence's cluster owns columns [c per, (c + 1) per)
// of every row of that sequence.
//  1. Row statistics: each warp takes whole rows' column slices and keeps the
//     online (max, sum of 2^((l - max) log2(e)/T)); the CTA's partial of
//     every row goes to every CTA of the cluster (distributed shared memory),
//     and after a cluster barrier each CTA folds the kSmallCtas partials in
//     rank order, so all CTAs hold the same statistics.
//  2. The accept tests of every position (one lane each), as in the fused
//     kernel; every CTA computes the same n.
//  3. The draw on rows p_{n+1} (and q_{n+1}): float-float weights from the
//     table-driven exponential; the CTAs' compensated totals S_p, S_q are
//     exchanged, giving the exact rho = S_p / S_q; the residual weights
//     max(0, e_p - rho e_q) (or e_p for the bonus token) are summed per warp
//     and per CTA and exchanged again; u R is located CTA by CTA, warp by
//     warp, then token by token in index order.
// Every CTA of a cluster takes the same branches (its inputs and arithmetic
// are the same), so every CTA reaches every cluster barrier.
#include "sv_draw.cuh"
#include "sv_rows.cuh"
#include "sv_small.h"

namespace sv {

namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kSmallRows = 2 * kSmallMaxGamma + 1;

// float-float sum of the CTA: warp butterflies, then warp 0 over the warps'
// totals in warp order (s_w: kSmallWarps float2). Every thread of warp 0 ends
// with the total; the warps' totals stay in s_w.
__device__ __forceinline__ void cta_sum_ff(float &h, float &l, float2 *s_w, int lane, int warp) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float oh = __shfl_xor_sync(kAll, h, off), ol = __shfl_xor_sync(kAll, l, off);
        ff_add(h, l, oh, ol, h, l);
    }
    if (lane == 0) s_w[warp] = make_float2(h, l);
    __syncthreads();
    h = 0.0f;
    l = 0.0f;
    if (warp == 0)
        for (int w = 0; w < kSmallWarps; ++w) ff_add(h, l, s_w[w].x, s_w[w].y, h, l);
}

// FP64 is a narrow, slow pipe on this part: the kernel keeps its decisions in
// float (the accept test, the fused kernel's own) and float-float (the draw's
// sums, prefixes and comparisons, about 48 bits).

// (e_p, e_q) of one token as float-float pairs (eph, epl, eqh, eql); the
// out-of-line copy serves the rarely run passes
__device__ __forceinline__ float4 pair_weights_inl(float lp, float lq, const ExpRow &er,
                                                   const float2 *tab) {
    f32x2 eh, el;
    exp2_pair<true>(pack2(lp, lq), er, tab, eh, el);
    const float2 h = unpack2(eh), l = unpack2(el);
    return make_float4(h.x, l.x, h.y, l.y);
}

__device__ __noinline__ float4 pair_weights(float lp, float lq, ExpRow er, const float2 *tab) {
    return pair_weights_inl(lp, lq, er, tab);
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kSmallWarps * 32, 1) small_kernel(const __grid_constant__ Params P) {
    constexpr int PV = DT == SV_DT_FP32 ? 4 : 8;
    constexpr int ESZ = DT == SV_DT_FP32 ? 4 : 2;
    __shared__ float4 s_part[kSmallCtas][kSmallRows];  // (max, sum, bad, -) of each CTA's slice
    __shared__ float4 s_tot[kSmallCtas];               // each CTA's draw totals
    __shared__ float2 s_stat[kSmallRows];              // the rows' (max, sum)
    __shared__ int s_rowbad[kSmallRows];
    __shared__ float2 s_w[kSmallWarps];
    __shared__ float2 s_wr[kSmallWarps];               // the warps' weight totals
    __shared__ int s_n;
    __shared__ float2 s_u[kSmallMaxGamma + 1];  // the draw uniform for n = 0..gamma
    __shared__ __align__(8) uint64_t s_bar;
    extern __shared__ __align__(128) uint8_t smem[];   // the exp2 table, then the row slices
    float2 *s_tab = reinterpret_cast<float2 *>(smem);
    uint8_t *s_rows = smem + kExpTab * sizeof(float2);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.x / kSmallCtas;
    const int gm = P.gamma_max;
    const float c2 = P.c2;

    // validation (every CTA, the same answer)
    const int g = P.gamma[b];
    int bad_in = 0;
    int64_t po = 0, qo = 0;
    if (g < 0 || g > gm) {
        bad_in = SPECVERIFY_STATUS_BAD_GAMMA;
    } else {
        po = P.p_row_off[b];
        if (po < 0 || po + g + 1 > P.target_rows) bad_in |= SPECVERIFY_STATUS_BAD_ROW;
        if (g > 0) {
            qo = P.q_row_off[b];
            if (qo < 0 || qo + g > P.draft_rows) bad_in |= SPECVERIFY_STATUS_BAD_ROW;
        }
        for (int i = 0; i < g; ++i) {
            const int32_t x = __ldg(&P.tokens[(int64_t)b * gm + i]);
            if (x < 0 || (int64_t)x >= P.V) bad_in |= SPECVERIFY_STATUS_BAD_TOKEN;
        }
    }
    int32_t *tok = P.tok_out + (int64_t)b * (gm + 1);
    if (bad_in) {
        if (rank == 0) {
            for (int i = threadIdx.x; i <= gm; i += blockDim.x) tok[i] = -1;
            if (threadIdx.x == 0) {
                P.n_out[b] = -1;
                atomicOr(P.status, bad_in);
            }
        }
        return;  // every CTA of the cluster leaves here
    }
    const int rows = 2 * g + 1;
    // row j of the sequence: p_j for j <= g, q_{j - g - 1} after
    auto row_ptr = [&](int j) -> const char * {
        return j <= g ? P.target + (po + j) * P.stride_bytes
                      : P.draft + (qo + j - g - 1) * P.stride_bytes;
    };
    // this CTA's columns: a whole number of 16-byte vectors
    const int64_t per = ((P.V + kSmallCtas - 1) / kSmallCtas + PV - 1) / PV * PV;
    const int64_t c0 = min(P.V, (int64_t)rank * per), c1 = min(P.V, c0 + per);
    const int nvec = (int)((c1 - c0) / PV);  // full vectors; the row's ragged tail is
    const int rem = (int)((c1 - c0) - (int64_t)nvec * PV);  // in the last CTA

    // every row's slice (full vectors) and the exp2 table into shared memory:
    // one barrier, one bulk copy per row
    const uint32_t bar = smem_u32(&s_bar);
    const uint32_t slice_bytes = (uint32_t)nvec * 16u;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(bar, slice_bytes * (uint32_t)rows + kExpTab * 8u);
        bulk_load(smem_u32(s_tab), P.exp2_tab, kExpTab * 8u, bar);
        if (slice_bytes > 0)
            for (int j = 0; j < rows; ++j)
                bulk_load(smem_u32(s_rows + (size_t)j * slice_bytes), row_ptr(j) + c0 * ESZ,
                          slice_bytes, bar);
    }
    __syncthreads();
    // While the copies land: warp 0 gathers each position's logits of its draft
    // token and its accept uniform (lane i: position i + 1), and the draw
    // uniform of every possible n (lane n), all of which the decision needs.
    float t_lp = 0.0f, t_lq = 0.0f, t_r = 0.0f;
    if (warp == 0) {
        if (lane < g) {
            const int32_t x = __ldg(&P.tokens[(int64_t)b * gm + lane]);
            t_lp = load_logit<DT>(row_ptr(lane), x);
            t_lq = load_logit<DT>(row_ptr(g + 1 + lane), x);
            t_r = accept_uniform(P.seed, (uint32_t)b, (uint32_t)(lane + 1));
        }
        if (lane <= g) {
            float uh, ul;
            draw_uniform_ff(P.seed, (uint32_t)b, (uint32_t)(lane + 1), uh, ul);
            s_u[lane] = make_float2(uh, ul);
        }
    }
    // (a wait that gives up marks every row of the sequence: the cluster then
    // reports a timeout, all of its CTAs taking the same branches)
    const bool loaded = mbar_wait_bounded(bar, 0);
    if (!loaded) mbar_wait_bounded(bar, 0);  // let the copies in flight land (bounded)
    auto slice = [&](int j) -> const uint4 * {
        return reinterpret_cast<const uint4 *>(s_rows + (size_t)j * slice_bytes);
    };

    // ---- 1. row statistics of this CTA's slice of every row
    for (int j = warp; j < rows; j += kSmallWarps) {
        const char *row = row_ptr(j);
        const uint4 *vp = slice(j);
        SoftAcc a = soft_init();
        // two passes over the slice in shared memory: the maximum, then the
        // sum of 2^((l - max) c2) with that reference (no rescaling)
        float m = -INFINITY;
#pragma unroll 4
        for (int v = lane; v < nvec; v += 32) m = max_nan(m, vec_max<DT>(vp[v]));
        if (lane < rem) m = max_nan(m, load_logit<DT>(row, c0 + (int64_t)nvec * PV + lane));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = max_nan(m, __shfl_xor_sync(kAll, m, off));
        if (m != m || m == INFINITY) {
            a.bad = true;
        } else if (m != -INFINITY) {
            const float mc = m * c2;
            float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 2
            for (int v = lane; v < nvec; v += 32) {
                float f[PV];
                vec_floats<DT>(vp[v], f);
#pragma unroll
                for (int e = 0; e < PV; ++e)
                    s4[e & 3] += ex2_approx(fmaxf(fmaf(f[e], c2, -mc), kXMin));
            }
            if (lane < rem)
                s4[0] += ex2_approx(fmaxf(fmaf(load_logit<DT>(row, c0 + (int64_t)nvec * PV + lane),
                                              c2, -mc), kXMin));
            float ssum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ssum += __shfl_xor_sync(kAll, ssum, off);
            a.m = m;
            a.s = ssum;
        }
        const bool wok = __all_sync(kAll, loaded);
        if (lane < kSmallCtas) {
            const float4 part = make_float4(a.m, a.s, a.bad ? 1.0f : 0.0f, wok ? 0.0f : 1.0f);
            st_cluster_f4(cluster_addr(&s_part[rank][j], (uint32_t)lane), part);
        }
    }
    cluster_sync();

    // ---- 2. the rows' statistics (rank order), the accept tests
    if (threadIdx.x < rows) {
        const int j = threadIdx.x;
        SoftAcc a = soft_init();
        bool late = false;
        for (int c = 0; c < kSmallCtas; ++c) {
            const float4 pc = s_part[c][j];
            soft_merge<false>(a, SoftAcc{pc.x, pc.y, 0.0f, pc.z != 0.0f}, c2);
            late |= pc.w != 0.0f;
        }
        const bool bad = late || a.bad || a.m == -INFINITY || !(a.s > 0.0f);
        s_stat[j] = make_float2(a.m, a.s);
        s_rowbad[j] = late ? 2 : (bad ? 1 : 0);
        if (rank == 0) {
            float *lse_out = j <= g ? P.p_lse : P.q_lse;
            const int64_t phys = j <= g ? po + j : qo + j - g - 1;
            if (lse_out)
                lse_out[phys] = bad ? __int_as_float(0x7fffffff)
                                    : (float)((double)a.m * P.invT + log((double)a.s));
        }
    }
    __syncthreads();
    if (warp == 0) {
        // n: the first rejection; a bad row the result depends on (every row
        // when logsumexp outputs were asked for) makes the sequence bad (-2)
        int n = g;
        bool seq_bad = false;
        for (int i0 = 0; i0 < g; i0 += 32) {
            const int i = i0 + lane;
            bool rej = false, rbad = false;
            if (i < g) {
                rbad = s_rowbad[i] != 0 || s_rowbad[g + 1 + i] != 0;
                if (!rbad) {
                    // (gamma <= 16: lane i holds position i + 1's gathered inputs)
                    const float ratio = accept_ratio(P, t_lp, t_lq, s_stat[i], s_stat[g + 1 + i]);
                    rej = t_r > ratio;
                }
            }
            const uint32_t stop = __ballot_sync(kAll, rej || rbad);
            if (stop) {
                const int first = __ffs(stop) - 1;
                n = i0 + first;
                seq_bad = (__ballot_sync(kAll, rbad) >> first) & 1u;
                break;
            }
        }
        if (!seq_bad && n == g) seq_bad = s_rowbad[g] != 0;
        if (!P.skip) {
            bool any = false;
            for (int j = lane; j < rows; j += 32) any |= s_rowbad[j] != 0;
            seq_bad |= __any_sync(kAll, any);
        }
        bool late = false;
        for (int j = lane; j < rows; j += 32) late |= s_rowbad[j] == 2;
        late = __any_sync(kAll, late);
        if (lane == 0) s_n = late ? -2 : (seq_bad ? -1 : n);
    }
    __syncthreads();
    const int n = s_n;
    if (n < 0) {
        if (rank == 0) {
            for (int i = threadIdx.x; i <= gm; i += blockDim.x) tok[i] = -1;
            if (threadIdx.x == 0) {
                P.n_out[b] = -1;
                atomicOr(P.status, n == -2 ? SPECVERIFY_STATUS_TIMEOUT : SPECVERIFY_STATUS_BAD_LOGIT);
            }
        }
        return;  // every CTA of the cluster leaves here
    }

    // ---- 3. the draw: rows p_{n+1} and, after a rejection, q_{n+1}
    const bool residual = n < g;
    const char *prow = row_ptr(n);
    const char *qrow = residual ? row_ptr(g + 1 + n) : prow;
    const float2 sp = s_stat[n], sq = residual ? s_stat[g + 1 + n] : sp;
    ExpRow er;
    er.ch = splat2(P.c2h);
    er.cl = splat2(P.c2l);
    // (any integer near M c keeps the weights in range; float arithmetic, the
    // same in every CTA)
    er.shift = pack2(rintf(sp.x * P.c2h), rintf(sq.x * P.c2h));
    er.lmin = pack2(sp.x - P.lspan, sq.x - P.lspan);
    const float2 *tab = s_tab;
    const uint4 *pv = slice(n);
    const uint4 *qv = residual ? slice(g + 1 + n) : pv;
    // this warp's vectors of the slice: [wv0, wv1), lane-interleaved in rounds of 32;
    // the slice's ragged tail (last CTA) belongs to the last warp
    const int vpw = (nvec + kSmallWarps - 1) / kSmallWarps;
    const int wv0 = min(nvec, warp * vpw), wv1 = min(nvec, wv0 + vpw);
    const int ntail = warp == kSmallWarps - 1 ? rem : 0;
    const int64_t tail0 = c0 + (int64_t)nvec * PV;
    // (e_p, e_q) of logits (lp, lq)
    auto weights = [&](float lp, float lq, float &eph, float &epl, float &eqh, float &eql) {
        const float4 e = pair_weights(lp, lq, er, tab);
        eph = e.x;
        epl = e.y;
        eqh = e.z;
        eql = e.w;
    };
    float rh = 0.0f, rl = 0.0f;  // rho = S_p / S_q as a float-float (residual draws)
    // the draw weight: max(0, e_p - rho e_q) after a rejection, e_p for the bonus token
    auto draw_w = [&](float lp, float lq, float &wh, float &wl) {
        float eph, epl, eqh, eql;
        weights(lp, lq, eph, epl, eqh, eql);
        if (residual) {
            residual_weight(eph, epl, eqh, eql, rh, rl, wh, wl);
        } else {
            wh = eph;
            wl = epl;
        }
    };
    auto draw_w_of = [&](const float4 &e, float &wh, float &wl) {
        if (residual) {
            residual_weight(e.x, e.y, e.z, e.w, rh, rl, wh, wl);
        } else {
            wh = e.x;
            wl = e.y;
        }
    };
    // fn(column, lp, lq) for every element of the lane's share, vector by vector
    auto for_elems = [&](auto &&fn) {
#pragma unroll 2
        for (int v = wv0 + lane; v < wv1; v += 32) {
            const uint4 a = pv[v], c = qv[v];
            float fp[PV], fq[PV];
            vec_floats<DT>(a, fp);
            vec_floats<DT>(c, fq);
            const int64_t col = c0 + (int64_t)v * PV;
#pragma unroll
            for (int e = 0; e < PV; ++e) fn(col + e, fp[e], fq[e]);
        }
        if (lane < ntail)
            fn(tail0 + lane, load_logit<DT>(prow, tail0 + lane), load_logit<DT>(qrow, tail0 + lane));
    };
    // The weights of up to kCacheE elements a lane stay in registers from
    // pass A to pass B and the locate (lane j's k-th vector is wv0 + j + 32 k);
    // a lane with more elements (a large vocabulary) recomputes them.
    constexpr int kCacheV = 8 / PV;
    const bool cached = vpw <= 32 * kCacheV;
    float4 ce[kCacheV * PV];
    // pass A: the slice's S_p and S_q, compensated
    float sph = 0.0f, spl = 0.0f, sqh = 0.0f, sql = 0.0f;
    if (cached) {
#pragma unroll
        for (int k = 0; k < kCacheV; ++k) {
            const int v = wv0 + lane + 32 * k;
            float fp[PV], fq[PV];
            if (v < wv1) {
                vec_floats<DT>(pv[v], fp);
                vec_floats<DT>(qv[v], fq);
            }
#pragma unroll
            for (int e = 0; e < PV; ++e) {
                // (inline here: the lane's elements interleave)
                ce[k * PV + e] = v < wv1 ? pair_weights_inl(fp[e], fq[e], er, tab)
                                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                ff_add(sph, spl, ce[k * PV + e].x, ce[k * PV + e].y, sph, spl);
                ff_add(sqh, sql, ce[k * PV + e].z, ce[k * PV + e].w, sqh, sql);
            }
        }
        if (lane < ntail) {
            float eph, epl, eqh, eql;
            weights(load_logit<DT>(prow, tail0 + lane), load_logit<DT>(qrow, tail0 + lane), eph,
                    epl, eqh, eql);
            ff_add(sph, spl, eph, epl, sph, spl);
            ff_add(sqh, sql, eqh, eql, sqh, sql);
        }
    } else {
        for_elems([&](int64_t, float lp, float lq) {
            float eph, epl, eqh, eql;
            weights(lp, lq, eph, epl, eqh, eql);
            ff_add(sph, spl, eph, epl, sph, spl);
            ff_add(sqh, sql, eqh, eql, sqh, sql);
        });
    }
    cta_sum_ff(sph, spl, s_w, lane, warp);
    __syncthreads();
    cta_sum_ff(sqh, sql, s_w, lane, warp);
    if (threadIdx.x < kSmallCtas)
        st_cluster_f4(cluster_addr(&s_tot[rank], (uint32_t)threadIdx.x),
                      make_float4(sph, spl, sqh, sql));
    cluster_sync();
    // the rows' totals in rank order; rho; the CTAs' S_p
    float Sph = 0.0f, Spl = 0.0f, Sqh = 0.0f, Sql = 0.0f;
    float2 cta_sp[kSmallCtas];
#pragma unroll
    for (int c = 0; c < kSmallCtas; ++c) {
        const float4 tc = s_tot[c];
        ff_add(Sph, Spl, tc.x, tc.y, Sph, Spl);
        ff_add(Sqh, Sql, tc.z, tc.w, Sqh, Sql);
        cta_sp[c] = make_float2(tc.x, tc.y);
    }
    if (residual) ff_div(Sph, Spl, Sqh, Sql, rh, rl);
    // pass B: the draw weights of the lane, the warp, the CTA
    float rwh = 0.0f, rwl = 0.0f;
    if (cached) {
#pragma unroll
        for (int i = 0; i < kCacheV * PV; ++i) {
            float wh, wl;
            draw_w_of(ce[i], wh, wl);
            ff_add(rwh, rwl, wh, wl, rwh, rwl);
        }
        if (lane < ntail) {
            float wh, wl;
            draw_w(load_logit<DT>(prow, tail0 + lane), load_logit<DT>(qrow, tail0 + lane), wh, wl);
            ff_add(rwh, rwl, wh, wl, rwh, rwl);
        }
    } else {
        for_elems([&](int64_t, float lp, float lq) {
            float wh, wl;
            draw_w(lp, lq, wh, wl);
            ff_add(rwh, rwl, wh, wl, rwh, rwl);
        });
    }
    {
        float h = rwh, l = rwl;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oh = __shfl_xor_sync(kAll, h, off), ol = __shfl_xor_sync(kAll, l, off);
            ff_add(h, l, oh, ol, h, l);
        }
        if (lane == 0) s_wr[warp] = make_float2(h, l);
    }
    float2 cta_w[kSmallCtas];
    if (residual) {
        __syncthreads();  // every CTA has read s_tot (pass A) before it is overwritten
        float h = rwh, l = rwl;
        cta_sum_ff(h, l, s_w, lane, warp);
        cluster_sync();   // (all CTAs past their reads of s_tot)
        if (threadIdx.x < kSmallCtas)
            st_cluster_f4(cluster_addr(&s_tot[rank], (uint32_t)threadIdx.x),
                          make_float4(h, l, 0.0f, 0.0f));
        cluster_sync();
#pragma unroll
        for (int c = 0; c < kSmallCtas; ++c) cta_w[c] = make_float2(s_tot[c].x, s_tot[c].y);
    } else {
        __syncthreads();
#pragma unroll
        for (int c = 0; c < kSmallCtas; ++c) cta_w[c] = cta_sp[c];
    }
    float Rh = 0.0f, Rl = 0.0f;
#pragma unroll
    for (int c = 0; c < kSmallCtas; ++c) ff_add(Rh, Rl, cta_w[c].x, cta_w[c].y, Rh, Rl);
    float uh, ul;
    uh = s_u[n].x;
    ul = s_u[n].y;
    const bool zero_mass = !(Rh > 0.0f);
    float th, tl;
    ff_mul(uh, ul, Rh, Rl, th, tl);
    int cstar = -1;
    float bh = 0.0f, bl = 0.0f;  // the mass before CTA cstar
    {
        float runh = 0.0f, runl = 0.0f;
#pragma unroll
        for (int c = 0; c < kSmallCtas; ++c) {
            float nh, nl;
            ff_add(runh, runl, cta_w[c].x, cta_w[c].y, nh, nl);
            if (cstar < 0 && ff_gt(nh, nl, th, tl)) {
                cstar = c;
                bh = runh;
                bl = runl;
            }
            runh = nh;
            runl = nl;
        }
    }
    if (zero_mass || cstar < 0) {
        // Rare paths, one warp of the last CTA over the whole rows: no
        // residual mass after rounding (the token is drawn from p_{n+1} and a
        // status bit says so), or t at or past R through rounding (the last
        // token of positive weight).
        if (rank != kSmallCtas - 1 || warp != 0) return;
        float tzh = th, tzl = tl;
        if (zero_mass) ff_mul(uh, ul, Sph, Spl, tzh, tzl);
        float runh = 0.0f, runl = 0.0f;
        int32_t pick = -1, last = -1;
        for (int64_t base = 0; base < P.V; base += 32) {
            const int64_t col = base + lane;
            float wh = 0.0f, wl = 0.0f;
            if (col < P.V) {
                const float lp = load_logit<DT>(prow, col), lq = load_logit<DT>(qrow, col);
                if (zero_mass) {
                    float eqh, eql;
                    weights(lp, lq, wh, wl, eqh, eql);
                } else {
                    draw_w(lp, lq, wh, wl);
                }
            }
            float ch = wh, cl = wl;
            warp_incl_scan_ff(ch, cl, lane);
            float nh, nl;
            ff_add(runh, runl, ch, cl, nh, nl);
            const uint32_t pos = __ballot_sync(kAll, wh > 0.0f);
            if (pos) last = (int32_t)(base + 31 - __clz(pos));
            const uint32_t hit = __ballot_sync(kAll, wh > 0.0f && ff_gt(nh, nl, tzh, tzl));
            if (pick < 0 && hit) pick = (int32_t)(base + __ffs(hit) - 1);
            ff_add(runh, runl, __shfl_sync(kAll, ch, 31), __shfl_sync(kAll, cl, 31), runh, runl);
        }
        if (pick < 0) pick = last;
        for (int i = lane; i <= gm; i += 32)
            tok[i] = i < n ? __ldg(&P.tokens[(int64_t)b * gm + i]) : (i == n ? pick : -1);
        if (lane == 0) {
            P.n_out[b] = n;
            if (zero_mass) atomicOr(P.status, SPECVERIFY_STATUS_DRAW_ZERO_MASS);
        }
        return;
    }
    if ((int)rank != cstar) return;
    // the warp whose elements hold t (warp order)
    int wstar = -1;
    float wbh = 0.0f, wbl = 0.0f;
    {
        float runh = bh, runl = bl;
        for (int w = 0; w < kSmallWarps; ++w) {
            float nh, nl;
            ff_add(runh, runl, s_wr[w].x, s_wr[w].y, nh, nl);
            if (wstar < 0 && ff_gt(nh, nl, th, tl)) {
                wstar = w;
                wbh = runh;
                wbl = runl;
            }
            runh = nh;
            runl = nl;
        }
    }
    bool past = false;
    if (wstar < 0) {
        // t at or past the CTA's weight through rounding: its last warp with weight
        for (int w = kSmallWarps - 1; w >= 0 && wstar < 0; --w)
            if (s_wr[w].x > 0.0f) wstar = w;
        past = true;
    }
    if (warp != wstar) return;
    // the element: rounds of 32 vectors in index order (lane j: vector r0 + j), then the tail
    float runh = wbh, runl = wbl;
    int32_t token = -1, last = -1;
    for (int r0 = wv0; r0 < wv1 && token < 0; r0 += 32) {
        const int v = r0 + lane;
        float wvh[PV], wvl[PV];
        float sh = 0.0f, sl = 0.0f;
        const int64_t col0 = c0 + (int64_t)v * PV;
        if (v < wv1 && cached) {
            // round k = (r0 - wv0) / 32 is the lane's k-th cached vector
            const int k = (r0 - wv0) >> 5;
#pragma unroll
            for (int kk = 0; kk < kCacheV; ++kk)
                if (kk == k)
#pragma unroll
                    for (int e = 0; e < PV; ++e) {
                        draw_w_of(ce[kk * PV + e], wvh[e], wvl[e]);
                        ff_add(sh, sl, wvh[e], wvl[e], sh, sl);
                    }
        } else if (v < wv1) {
            float fp[PV], fq[PV];
            vec_floats<DT>(pv[v], fp);
            vec_floats<DT>(qv[v], fq);
#pragma unroll
            for (int e = 0; e < PV; ++e) {
                draw_w(fp[e], fq[e], wvh[e], wvl[e]);
                ff_add(sh, sl, wvh[e], wvl[e], sh, sl);
            }
        } else {
#pragma unroll
            for (int e = 0; e < PV; ++e) {
                wvh[e] = 0.0f;
                wvl[e] = 0.0f;
            }
        }
        int32_t lane_last = -1;
#pragma unroll
        for (int e = 0; e < PV; ++e)
            if (wvh[e] > 0.0f) lane_last = (int32_t)(col0 + e);
        for (int off = 16; off > 0; off >>= 1)
            lane_last = max(lane_last, __shfl_xor_sync(kAll, lane_last, off));
        if (lane_last >= 0) last = lane_last;
        float ch = sh, cl = sl;
        warp_incl_scan_ff(ch, cl, lane);
        float nh, nl;
        ff_add(runh, runl, ch, cl, nh, nl);
        const uint32_t hit = __ballot_sync(kAll, !past && v < wv1 && ff_gt(nh, nl, th, tl));
        if (hit) {
            const int j = __ffs(hit) - 1;
            int32_t tk = -1;
            if (lane == j) {
                // the mass before this lane's vector, then its elements in order
                float rh2, rl2;
                ff_add(nh, nl, -sh, -sl, rh2, rl2);
                for (int e = 0; e < PV; ++e) {
                    ff_add(rh2, rl2, wvh[e], wvl[e], rh2, rl2);
                    if (wvh[e] > 0.0f && ff_gt(rh2, rl2, th, tl)) {
                        tk = (int32_t)(col0 + e);
                        break;
                    }
                }
                if (tk < 0) tk = lane_last;
            }
            token = __shfl_sync(kAll, tk, j);
        }
        ff_add(runh, runl, __shfl_sync(kAll, ch, 31), __shfl_sync(kAll, cl, 31), runh, runl);
    }
    if (token < 0 && ntail > 0) {
        // the slice's ragged tail, in order
        int32_t tk = -1;
        if (lane == 0) {
            for (int e = 0; e < ntail && tk < 0; ++e) {
                const int64_t col = tail0 + e;
                float wh, wl;
                draw_w(load_logit<DT>(prow, col), load_logit<DT>(qrow, col), wh, wl);
                ff_add(runh, runl, wh, wl, runh, runl);
                if (wh > 0.0f) last = (int32_t)col;
                if (!past && wh > 0.0f && ff_gt(runh, runl, th, tl)) tk = (int32_t)col;
            }
        }
        token = __shfl_sync(kAll, tk, 0);
        last = __shfl_sync(kAll, last, 0);
    }
    if (token < 0) token = last;  // t past the warp's total through rounding
    for (int i = lane; i <= gm; i += 32)
        tok[i] = i < n ? __ldg(&P.tokens[(int64_t)b * gm + i]) : (i == n ? token : -1);
    if (lane == 0) P.n_out[b] = n;
}

cudaError_t prepare_small() {
    cudaError_t e = cudaFuncSetAttribute(small_kernel<SV_DT_FP32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(small_kernel<SV_DT_BF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmem);
    return e;
}

// The greedy step for a small batch (the Kadimisetty notes, "Greedy vs
// sampling": keep the longest prefix of drafts that equal argmax p_i, then
// append the target's argmax): one cluster of kSmallCtas CTAs per sequence,
// CTA c reading columns [c per, (c + 1) per) of the target rows
// p_1..p_{gamma+1} straight from global memory, one warp a row. Each lane
// keeps the first maximum of its logits in index order (a NaN is sticky: the
// row is bad); the warp's (maximum, index) goes to rank 0 of the cluster
// (distributed shared memory), which after a cluster barrier folds the
// slices in rank order (ties to the lower index) and runs the exact-match
// scan. The same results as the plan, row-statistics and accept kernels.
template <int DT>
__global__ void __launch_bounds__(kSmallWarps * 32, 1) small_greedy_kernel(const __grid_constant__ Params P) {
    __shared__ __align__(16) float4 s_arg[kSmallMaxGamma + 1][kSmallCtas];
    constexpr int PV = DT == SV_DT_FP32 ? 4 : 8;  // logits in a 16-byte vector
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.x / kSmallCtas;
    const int gm = P.gamma_max;
    int32_t *tok = P.tok_out + (int64_t)b * (gm + 1);

    // validation (every CTA, the same answer)
    const int g = P.gamma[b];
    int bad = 0;
    int64_t po = 0;
    if (g < 0 || g > gm) {
        bad = SPECVERIFY_STATUS_BAD_GAMMA;
    } else {
        po = P.p_row_off[b];
        if (po < 0 || po + g + 1 > P.target_rows) bad = SPECVERIFY_STATUS_BAD_ROW;
    }
    int tb = 0;
    if (bad == 0 && threadIdx.x < g) {
        const int32_t x = __ldg(&P.tokens[(int64_t)b * gm + threadIdx.x]);
        tb = (x < 0 || (int64_t)x >= P.V) ? 1 : 0;
    }
    if (__syncthreads_or(tb)) bad |= SPECVERIFY_STATUS_BAD_TOKEN;
    if (bad) {
        if (rank == 0) {
            for (int i = threadIdx.x; i <= gm; i += blockDim.x) tok[i] = -1;
            if (threadIdx.x == 0) {
                P.n_out[b] = -1;
                atomicOr(P.status, bad);
            }
        }
        return;  // every CTA of the cluster leaves here
    }

    // this CTA's columns: whole vectors, the last CTA's ending at V
    const int64_t V = P.V;
    const int64_t per = ((V + kSmallCtas - 1) / kSmallCtas + PV - 1) / PV * PV;
    const int64_t c0 = min(V, (int64_t)rank * per), c1 = min(V, c0 + per);
    const int64_t v0 = c0 / PV, v1 = c1 / PV;  // vectors inside [c0, c1)
    for (int j = warp; j <= g; j += kSmallWarps) {
        const char *row = P.target + (po + j) * P.stride_bytes;
        const uint4 *rv = reinterpret_cast<const uint4 *>(row);
        float best = -INFINITY;
        int32_t idx = -1;
        auto offer = [&](float m, const float *f, int n, int64_t e0) {
            if (best != best) return;  // NaN: sticky
            if (m != m) {
                best = m;
                return;
            }
            if (idx < 0 || m > best) {
                int e = 0;
                while (e < n - 1 && f[e] != m) ++e;
                best = m;
                idx = (int32_t)(e0 + e);
            }
        };
#pragma unroll 4
        for (int64_t vi = v0 + lane; vi < v1; vi += 32) {
            const uint4 w = __ldg(rv + vi);
            float f[PV];
            vec_floats<DT>(w, f);
            offer(vec_max<DT>(w), f, PV, vi * PV);
        }
        for (int64_t e = v1 * PV + lane; e < c1; e += 32) {  // the ragged end at V
            const float f1[1] = {load_logit<DT>(row, e)};
            offer(f1[0], f1, 1, e);
        }
        const float2 r = warp_combine_greedy(best, idx);
        if (lane == 0)
            st_cluster_f4(cluster_addr(&s_arg[j][rank], 0u), make_float4(r.x, r.y, 0.0f, 0.0f));
    }
    cluster_sync();
    if (rank != 0 || warp != 0) return;
    // fold the slices of row j (lane j) in rank order, then the exact-match scan
    float best = -INFINITY;
    int32_t idx = -1;
    if (lane <= g) {
        for (int c = 0; c < kSmallCtas; ++c) {
            const float4 v = s_arg[lane][c];
            const float ob = v.x;
            const int32_t oi = __float_as_int(v.y);
            const bool take = (ob != ob) ? true
                              : (best != best) ? false
                              : (oi >= 0 && (idx < 0 || ob > best || (ob == best && oi < idx)));
            if (take) {
                best = ob;
                idx = oi;
            }
        }
    }
    if (__any_sync(0xffffffffu, lane <= g && best != best)) {
        for (int i = lane; i <= gm; i += 32) tok[i] = -1;
        if (lane == 0) {
            P.n_out[b] = -1;
            atomicOr(P.status, SPECVERIFY_STATUS_BAD_LOGIT);
        }
        return;
    }
    const int32_t x = lane < g ? __ldg(&P.tokens[(int64_t)b * gm + lane]) : 0;
    const uint32_t mism = __ballot_sync(0xffffffffu, lane < g && x != idx);
    const int n = mism ? __ffs(mism) - 1 : g;
    const int32_t an = __shfl_sync(0xffffffffu, idx, n);
    for (int i = lane; i <= gm; i += 32) {
        const int32_t xi = i < n ? __ldg(&P.tokens[(int64_t)b * gm + i]) : -1;
        tok[i] = i < n ? xi : (i == n ? an : -1);
    }
    if (lane == 0) P.n_out[b] = n;
}

cudaError_t launch_small(const Params &p, int dtype, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * kSmallCtas));
    cfg.blockDim = dim3(kSmallWarps * 32);
    cfg.dynamicSmemBytes = small_smem_bytes(p);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSmallCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == SV_DT_FP32) return cudaLaunchKernelEx(&cfg, small_kernel<SV_DT_FP32>, p);
    return cudaLaunchKernelEx(&cfg, small_kernel<SV_DT_BF16>, p);
}

cudaError_t launch_small_greedy(const Params &p, int dtype, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * kSmallCtas));
    cfg.blockDim = dim3(kSmallWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSmallCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == SV_DT_FP32) return cudaLaunchKernelEx(&cfg, small_greedy_kernel<SV_DT_FP32>, p);
    return cudaLaunchKernelEx(&cfg, small_greedy_kernel<SV_DT_BF16>, p);
}

}  // namespace sv
