// sv_features.cu -- per-row diagnostics beside the verify step.
//
// Acceptance statistics ("DistillSpec" Sec. 3: the acceptance rate
// beta = sum_x min(p(x), q(x)); Sec. 4: the total variation distance
// TVD = 1/2 sum_x |p(x) - q(x)| = 1 - beta as its proxy): for every position
// i <= gamma_b of every sequence, the pair of rows (p_i, q_i) at one
// temperature. One CTA per pair at a time, two CTAs an SM: a first pass
// streams both rows for their softmax statistics (max, sum of
// 2^((l - max) log2(e)/T)), a second pass streams them again -- from L2: the
// CTA read them microseconds before -- and sums min(p, q) with p and q
// normalised (one exponential a token: min(2^a, 2^b) = 2^min(a, b)); TVD is
// then 1 - beta, equal to 1/2 sum |p - q| for normalised distributions.
//
// Draft features ("DISCO" Sec. 3 Eq. 2 and App. D.1: the classifier that
// sets the lookahead reads the top-k probabilities and the entropy of the
// draft distribution): for every given row, in one pass, the softmax
// statistics, the entropy -sum q ln q and the k largest probabilities with
// their token indices (ties to the lower index). The rows' stages are split
// into one contiguous range per warp; a warp keeps the statistics and the k
// best (logit, index) pairs of each row piece (a group of logits is looked at
// only when its maximum reaches the warp's k-th best, which after the first
// stage of a piece almost never happens), and a second kernel merges each
// row's pieces.
//
// The features kernel runs one persistent CTA of kFeatWarps warps per SM, the
// pair kernel two of kPairWarps; each warp streams 4 KiB stages (or 2 KiB of
// each of two rows) through its own ring of shared-memory slots filled by
// 1-D bulk asynchronous copies.
#include "sv_rows.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// draft features

// The row pass: the rows' 4 KiB stages are cut into equal contiguous ranges,
// one per warp (the restricted verify's split); a warp keeps per-lane softmax
// statistics with the entropy accumulator and the exact K best (logit,
// token) pairs of the current row piece, and stores both when the piece
// ends: pstat = (max, sum, entropy sum, flags), parts = the sorted list.
template <int DT, int K>
__global__ void __launch_bounds__(kFeatWarps * 32, 1) features_rows_kernel(const __grid_constant__ FeatParams F) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kFeatWarps][kFeatSlots];
    __shared__ __align__(16) TopK s_cand[kFeatWarps][64];
    constexpr int PV = DT == SV_DT_FP32 ? 4 : 8;
    constexpr int ESZ = DT == SV_DT_FP32 ? 4 : 2;
    constexpr int SB = kFeatSlotBytes;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar0 = smem_u32(&bars[warp][0]);
    uint8_t *wbuf = smem + warp * kFeatSlots * SB;
    if (lane == 0) {
        for (int s = 0; s < kFeatSlots; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();  // a warp uses only its own barriers and buffers

    const int64_t spr = (F.row_bytes + SB - 1) / SB;
    const int64_t S = F.nrows * spr;
    const int64_t nw = (int64_t)gridDim.x * kFeatWarps;
    const int64_t nv = nw * kRestrictRangesPerWarp;
    const int64_t range = (S + nv - 1) / nv;
    const int64_t w = (int64_t)blockIdx.x * kFeatWarps + warp;
    if (w * range >= S) return;
    const float c2 = F.c2;
    const int32_t V32 = (int32_t)F.V;
    SoftAcc acc = soft_init();
    WarpTopK<K> tk;
    tk.buf = s_cand[warp];
    tk.reset();
    split_stream<kRestrictRangesPerWarp>(
        w, nw, range, spr, S, F.row_bytes, wbuf, bar0, lane,
        [&](const SplitCur &c) { return F.rows + c.rr * F.stride_bytes; },
        [&](const SplitCur &c, const uint8_t *slot, int bytes) {
            const uint4 *vb = reinterpret_cast<const uint4 *>(slot);
            const int nvec = bytes >> 4;
            const int32_t e0 = c.st * (SB / ESZ);
            for (int j = 0; j < SB / 16 / 32; ++j) {
                const int vi = lane + 32 * j;
                if (__all_sync(0xffffffffu, vi >= nvec)) break;
                // past the stage's vectors: -inf logits (bf16 pair 0xff80ff80)
                const uint4 v = vi < nvec ? vb[vi]
                                          : (DT == SV_DT_FP32 ? make_uint4(0xff800000u, 0xff800000u,
                                                                           0xff800000u, 0xff800000u)
                                                              : make_uint4(0xff80ff80u, 0xff80ff80u,
                                                                           0xff80ff80u, 0xff80ff80u));
                float f[PV];
                if (DT == SV_DT_BF16) {
                    // the sums see logits below the stand-in (-inf among them)
                    // as the stand-in: weight 0 and a finite exponent, so the
                    // entropy needs no clamp a logit; the maximum (and NaN or
                    // +inf detection) comes from the raw logits
                    uint4 u;
                    asm("max.bf16x2 %0, %1, %2;" : "=r"(u.x) : "r"(v.x), "r"(F.ninf_sub));
                    asm("max.bf16x2 %0, %1, %2;" : "=r"(u.y) : "r"(v.y), "r"(F.ninf_sub));
                    asm("max.bf16x2 %0, %1, %2;" : "=r"(u.z) : "r"(v.z), "r"(F.ninf_sub));
                    asm("max.bf16x2 %0, %1, %2;" : "=r"(u.w) : "r"(v.w), "r"(F.ninf_sub));
                    vec_floats<DT>(u, f);
                    soft_add_vec<PV, false>(acc, f, vec_max<DT>(v), c2);
                } else {
                    vec_floats<DT>(v, f);
                    soft_add_vec<PV>(acc, f, vec_max<DT>(v), c2);
                }
            }
            tk.template offer_stage<DT, SB / 16 / 32>(vb, nvec, e0, V32, lane);
            const int rem = (bytes & 15) / ESZ;
            if (rem > 0) {
                const int32_t e = e0 + nvec * PV + lane;
                float f1[1] = {tail_logit<DT>(F.rows + c.rr * F.stride_bytes, e, lane < rem)};
                soft_add<true>(acc, f1, 1, f1[0], c2);
                tk.offer(f1, 1, f1[0], e, V32, lane);
            }
        },
        [&](const SplitCur &c, uint32_t extra) {
            const TopK t = tk.finish(lane);
            SoftAcc tot = acc;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) soft_merge<true>(tot, soft_shfl_xor<true>(tot, off), c2);
            uint32_t flags = extra | (tot.bad ? 1u : 0u);
            const int64_t pi = w * F.cap + c.k;  // one range per warp
            if (c.k < F.cap) {
                F.parts[pi * 32 + lane] = RTop{t.v, t.i};
                if (lane == 0) F.pstat[pi] = make_float4(tot.m, tot.s, tot.t, __uint_as_float(flags));
            }
            acc = soft_init();
            tk.reset();
        });
}

// One warp per row: merge the row's pieces (softmax statistics in a fixed
// order, sorted lists by bitonic merges) and write the features.
template <int K>
__global__ void __launch_bounds__(256) features_final_kernel(const __grid_constant__ FeatParams F) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= F.nrows) return;
    const int64_t spr = (F.row_bytes + kFeatSlotBytes - 1) / kFeatSlotBytes;
    const int64_t S = F.nrows * spr;
    const int64_t nv = (int64_t)F.row_grid * kFeatWarps * kRestrictRangesPerWarp;
    const int64_t range = (S + nv - 1) / nv;
    const float c2 = F.c2;
    const int64_t vf = r * spr / range, vl = ((r + 1) * spr - 1) / range;
    SoftAcc tot = soft_init();
    TopK list{-INFINITY, INT_MAX};
    uint32_t flags = 0;
    for (int64_t v = vf; v <= vl; ++v) {
        const int64_t k = r - v * range / spr;
        if (k >= F.cap) {
            flags |= 2u;
            continue;
        }
        const int64_t pi = v * F.cap + k;
        const float4 st = __ldcg(&F.pstat[pi]);
        const float2 e = __ldcg(reinterpret_cast<const float2 *>(F.parts + pi * 32 + lane));
        list = merge_lists(list, TopK{e.x, __float_as_int(e.y)}, lane);
        const uint32_t f = __float_as_uint(st.w);
        flags |= f;
        soft_merge<true>(tot, SoftAcc{st.x, st.y, st.z, (f & 1u) != 0}, c2);
    }
    const bool bad = flags != 0u || tot.bad || tot.m == -INFINITY || !(tot.s > 0.0f);
    const float nan = __int_as_float(0x7fffffff);
    if (lane == 0) {
        // H = ln S - ln 2 * t / S (t in log2 units)
        F.entropy[r] = bad ? nan
                           : (float)(log((double)tot.s) -
                                     0.6931471805599453 * (double)tot.t / (double)tot.s);
        if (bad && F.status)
            atomicOr(F.status, (flags & 2u) ? SPECVERIFY_STATUS_TIMEOUT : SPECVERIFY_STATUS_BAD_LOGIT);
    }
    if (lane < F.k) {
        const bool live = !bad && lane < K && list.i != INT_MAX;
        F.topk_prob[r * F.k + lane] =
            bad ? nan : live ? ex2_approx(fmaxf((list.v - tot.m) * c2, kXMin)) / tot.s : 0.0f;
        F.topk_idx[r * F.k + lane] = live ? list.i : -1;
    }
}

// ---------------------------------------------------------------------------
// acceptance statistics

// Two CTAs of kPairWarps warps share an SM, so that one CTA's DRAM-bound
// first pass overlaps the other's L2-bound, ALU-heavy second pass; both
// passes run on packed float pairs.
constexpr int kPairWarps = 8;
constexpr int kPairSmem = kPairWarps * kFeatSlots * kFeatSlotBytes;  // 96 KiB

// Per-lane softmax statistics of one row: sum 2^((l - m) c2) with m the
// lane's running maximum, raised a vector at a time.
struct PairAcc {
    float m, s;
    bool bad;
};

// Adds the PV logits f (maximum g) to a.
template <int PV>
__device__ __forceinline__ void pair_add(PairAcc &a, const float *f, float g, float c2) {
    if (g != g || g == INFINITY) {  // NaN or +inf logit: a bad row
        a.bad = true;
        return;
    }
    if (g == -INFINITY) return;
    if (g > a.m) {
        if (a.m != -INFINITY) a.s *= ex2_approx((a.m - g) * c2);
        a.m = g;
    }
    const float mc = a.m * c2;
    const f32x2 c2x2 = pack2(c2, c2), nmc = pack2(-mc, -mc);
    f32x2 acc = 0ull;
#pragma unroll
    for (int e = 0; e < PV; e += 2) {
        const float2 x = unpack2(fma2(pack2(f[e], f[e + 1]), c2x2, nmc));
        acc = add2(acc, pack2(ex2_approx(x.x), ex2_approx(x.y)));
    }
    const float2 t = unpack2(acc);
    a.s += t.x + t.y;
}

__device__ __forceinline__ void pair_merge(PairAcc &a, const PairAcc &b, float c2) {
    a.bad |= b.bad;
    if (b.m == -INFINITY) return;
    if (a.m == -INFINITY) {
        a.m = b.m;
        a.s = b.s;
        return;
    }
    const float M = fmaxf(a.m, b.m);
    a.s = a.s * ex2_approx((a.m - M) * c2) + b.s * ex2_approx((b.m - M) * c2);
    a.m = M;
}

// The CTA's statistics of two rows at once: warp butterflies, then every
// thread folds the warps' totals in warp order.
__device__ void pair_cta_reduce(PairAcc &ap, PairAcc &aq, float c2, PairAcc (*sm)[2], int lane,
                                int warp) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        PairAcc b;
        b.m = __shfl_xor_sync(0xffffffffu, ap.m, off);
        b.s = __shfl_xor_sync(0xffffffffu, ap.s, off);
        b.bad = __shfl_xor_sync(0xffffffffu, ap.bad ? 1 : 0, off) != 0;
        pair_merge(ap, b, c2);
        b.m = __shfl_xor_sync(0xffffffffu, aq.m, off);
        b.s = __shfl_xor_sync(0xffffffffu, aq.s, off);
        b.bad = __shfl_xor_sync(0xffffffffu, aq.bad ? 1 : 0, off) != 0;
        pair_merge(aq, b, c2);
    }
    if (lane == 0) {
        sm[warp][0] = ap;
        sm[warp][1] = aq;
    }
    __syncthreads();
    ap = sm[0][0];
    aq = sm[0][1];
    for (int w = 1; w < kPairWarps; ++w) {
        pair_merge(ap, sm[w][0], c2);
        pair_merge(aq, sm[w][1], c2);
    }
    __syncthreads();  // sm reusable
}

// One position (p_i, q_i) per CTA at a time: pass 1 streams both rows for
// their statistics, pass 2 streams them again (from L2: the CTA read them
// microseconds before) and sums min(p, q) and |p - q| of the normalised
// p = 2^(l c2 - o_p), q = 2^(l c2 - o_q), a token's (p, q) pair in one
// packed register.
template <int DT>
__global__ void __launch_bounds__(kPairWarps * 32, 2) pair_kernel(const __grid_constant__ FeatParams F) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kPairWarps][kFeatSlots];
    __shared__ PairAcc s_acc[kPairWarps][2];
    __shared__ float s_sum[kPairWarps];
    __shared__ int s_timeout;
    constexpr int PV = DT == SV_DT_FP32 ? 4 : 8;
    constexpr int ESZ = DT == SV_DT_FP32 ? 4 : 2;
    constexpr int SB = kFeatSlotBytes / 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar0 = smem_u32(&bars[warp][0]);
    uint8_t *wbuf = smem + warp * kFeatSlots * kFeatSlotBytes;
    if (lane == 0) {
        for (int s = 0; s < kFeatSlots; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    uint32_t parity = 0;
    const float c2 = F.c2;
    const int gm = F.gamma_max;
    const float nan = __int_as_float(0x7fffffff);
    const f32x2 c2x2 = pack2(c2, c2);
    // positions b * gamma_max + i, i < gamma_b, one per CTA at a time
    for (int64_t pi = blockIdx.x; pi < F.nrows * gm; pi += gridDim.x) {
        const int64_t b = pi / gm;
        const int i = (int)(pi - b * gm);
        const int g = F.gamma[b];
        if (g < 0 || g > gm) {
            if (threadIdx.x == 0) {
                F.beta[pi] = nan;
                F.tvd[pi] = nan;
                if (F.status && i == 0) atomicOr(F.status, SPECVERIFY_STATUS_BAD_GAMMA);
            }
            continue;
        }
        const int64_t po = F.p_row_off[b], qo = F.q_row_off[b];
        const bool rows_ok = g == 0 || (po >= 0 && po + g + 1 <= F.target_rows && qo >= 0 &&
                                        qo + g <= F.draft_rows);
        if (i >= g || !rows_ok) {
            if (threadIdx.x == 0) {
                F.beta[pi] = nan;
                F.tvd[pi] = nan;
                if (!rows_ok && i == 0 && F.status) atomicOr(F.status, SPECVERIFY_STATUS_BAD_ROW);
            }
            continue;
        }
        if (threadIdx.x == 0) s_timeout = 0;
        const char *rows2[2] = {F.rows + (po + i) * F.stride_bytes,
                                F.rows2 + (qo + i) * F.stride_bytes};
        // pass 1: statistics of both rows
        PairAcc ap{-INFINITY, 0.0f, false}, aq{-INFINITY, 0.0f, false};
        bool ok = ring_stream<2, SB>(
            rows2, F.row_bytes, warp, kPairWarps, wbuf, bar0, parity, lane,
            [&](const uint8_t *slot, int64_t s, int bytes) {
                const int nvec = bytes >> 4;
                const int64_t e0 = s * (SB / ESZ);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint4 *vb = reinterpret_cast<const uint4 *>(slot + r * SB);
                    PairAcc &a = r == 0 ? ap : aq;
                    for (int vi = lane; vi < nvec; vi += 32) {
                        const uint4 w = vb[vi];
                        float f[PV];
                        vec_floats<DT>(w, f);
                        pair_add<PV>(a, f, vec_max<DT>(w), c2);
                    }
                    const int rem = (bytes & 15) / ESZ;
                    if (lane < rem) {
                        const float v = load_logit<DT>(rows2[r], e0 + (int64_t)nvec * PV + lane);
                        float f2[2] = {v, -INFINITY};
                        pair_add<2>(a, f2, v, c2);
                    }
                }
            });
        __syncthreads();
        if (!ok && lane == 0) s_timeout = 1;
        pair_cta_reduce(ap, aq, c2, s_acc, lane, warp);
        const bool bad = ap.bad || aq.bad || ap.m == -INFINITY || aq.m == -INFINITY ||
                         !(ap.s > 0.0f) || !(aq.s > 0.0f);
        if (bad) {
            if (threadIdx.x == 0) {
                F.beta[pi] = nan;
                F.tvd[pi] = nan;
                if (F.status) atomicOr(F.status, SPECVERIFY_STATUS_BAD_LOGIT);
            }
            continue;
        }
        // pass 2: beta = sum min(p, q) = sum 2^min(l_p c2 - op, l_q c2 - oq) with
        // p and q normalised: one exponential a token; TVD = 1 - beta, which
        // equals 1/2 sum |p - q| for normalised distributions
        const f32x2 no = pack2(-(ap.m * c2 + __log2f(ap.s)), -(aq.m * c2 + __log2f(aq.s)));
        float mn = 0.0f;
        auto token = [&](float lp, float lq) {
            const float2 x = unpack2(fma2(pack2(lp, lq), c2x2, no));
            mn += ex2_approx(fminf(x.x, x.y));
        };
        // in reverse stage order: the stages this CTA read last are the ones
        // most likely still in L2
        const int64_t nst = (F.row_bytes + SB - 1) / SB;
        const int64_t last = warp < nst ? warp + (nst - 1 - warp) / kPairWarps * kPairWarps : -1;
        ok &= ring_stream<2, SB>(
            rows2, F.row_bytes, last, -kPairWarps, wbuf, bar0, parity, lane,
            [&](const uint8_t *slot, int64_t s, int bytes) {
                const int nvec = bytes >> 4;
                const int64_t e0 = s * (SB / ESZ);
                const uint4 *vp = reinterpret_cast<const uint4 *>(slot);
                const uint4 *vq = reinterpret_cast<const uint4 *>(slot + SB);
                for (int vi = lane; vi < nvec; vi += 32) {
                    float fp[PV], fq[PV];
                    vec_floats<DT>(vp[vi], fp);
                    vec_floats<DT>(vq[vi], fq);
#pragma unroll
                    for (int e = 0; e < PV; ++e) token(fp[e], fq[e]);
                }
                const int rem = (bytes & 15) / ESZ;
                if (lane < rem) {
                    const int64_t e = e0 + (int64_t)nvec * PV + lane;
                    token(load_logit<DT>(rows2[0], e), load_logit<DT>(rows2[1], e));
                }
            });
        if (!ok && lane == 0) s_timeout = 1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mn += __shfl_xor_sync(0xffffffffu, mn, off);
        if (lane == 0) s_sum[warp] = mn;
        __syncthreads();
        if (threadIdx.x == 0) {
            float sm = 0.0f;
            for (int w = 0; w < kPairWarps; ++w) sm += s_sum[w];
            F.beta[pi] = s_timeout ? nan : sm;
            F.tvd[pi] = s_timeout ? nan : fmaxf(0.0f, 1.0f - sm);
            if (s_timeout && F.status) atomicOr(F.status, SPECVERIFY_STATUS_TIMEOUT);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// launchers

cudaError_t launch_features(const FeatParams &p, int dtype, cudaStream_t s) {
    if (p.nrows <= 0) return cudaSuccess;
    const dim3 block(kFeatWarps * 32);
    const int fgrid = (int)((p.nrows + 7) / 8);
#define SV_FEAT_LAUNCH(DTV, KV)                                                   \
    do {                                                                          \
        features_rows_kernel<DTV, KV><<<p.row_grid, block, kFeatSmem, s>>>(p);    \
        features_final_kernel<KV><<<fgrid, 256, 0, s>>>(p);                       \
    } while (0)
    if (dtype == SV_DT_FP32) {
        if (p.k <= 8) SV_FEAT_LAUNCH(SV_DT_FP32, 8);
        else if (p.k <= 16) SV_FEAT_LAUNCH(SV_DT_FP32, 16);
        else SV_FEAT_LAUNCH(SV_DT_FP32, 32);
    } else {
        if (p.k <= 8) SV_FEAT_LAUNCH(SV_DT_BF16, 8);
        else if (p.k <= 16) SV_FEAT_LAUNCH(SV_DT_BF16, 16);
        else SV_FEAT_LAUNCH(SV_DT_BF16, 32);
    }
#undef SV_FEAT_LAUNCH
    return cudaGetLastError();
}

cudaError_t launch_pairs(const FeatParams &p, int dtype, int num_sms, cudaStream_t s) {
    const int64_t units = p.nrows * p.gamma_max;
    const int64_t ctas = 2 * (int64_t)num_sms;  // two CTAs an SM
    const int grid = (int)(units < ctas ? units : ctas);
    if (grid <= 0) return cudaSuccess;
    if (dtype == SV_DT_FP32)
        pair_kernel<SV_DT_FP32><<<grid, kPairWarps * 32, kPairSmem, s>>>(p);
    else
        pair_kernel<SV_DT_BF16><<<grid, kPairWarps * 32, kPairSmem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t prepare_features() {
    const void *fns[] = {(const void *)features_rows_kernel<SV_DT_FP32, 8>,
                         (const void *)features_rows_kernel<SV_DT_FP32, 16>,
                         (const void *)features_rows_kernel<SV_DT_FP32, 32>,
                         (const void *)features_rows_kernel<SV_DT_BF16, 8>,
                         (const void *)features_rows_kernel<SV_DT_BF16, 16>,
                         (const void *)features_rows_kernel<SV_DT_BF16, 32>,
                         (const void *)pair_kernel<SV_DT_FP32>,
                         (const void *)pair_kernel<SV_DT_BF16>};
    for (const void *f : fns) {
        const int bytes = (f == (const void *)pair_kernel<SV_DT_FP32> ||
                           f == (const void *)pair_kernel<SV_DT_BF16>)
                              ? kPairSmem
                              : kFeatSmem;
        const cudaError_t e =
            cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace sv
