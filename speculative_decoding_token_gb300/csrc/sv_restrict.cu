// sv_restrict.cu -- restricted speculative sampling ("Speculative Decoding
// and Distillation" (Kadimisetty notes), "Greedy vs sampling": temperature,
// top-k and top-p restrict the target and the draft distributions alike, and
// the accept / residual rule of speculative sampling ("DistillSpec" Sec. 3,
// App. A.3 Algorithm A.1) then runs on the restricted distributions).
//
// Per sequence b a temperature T_b, a top-k k_b <= 32 and a top-p p_b. A row
// keeps its k_b largest logits (ties: the lower token index first); on their
// softmax(l / T_b), renormalised, it keeps the shortest prefix in that order
// whose probability reaches p_b, and renormalises again. The selection by
// logit does not depend on T_b (x -> x / T is increasing), so the pass over
// the rows only keeps each row's 32 best (logit, token) pairs; everything
// after it works on those lists.
//
// Two launches:
//  - restrict_plan_kernel (one CTA): validates every sequence, writes the
//    outputs of the bad ones, and lays the rows of the good ones out one
//    after another (p_0..p_gamma then q_0..q_{gamma-1} per sequence).
//  - restrict_kernel (one persistent CTA of 16 warps per SM): the rows' 4 KiB
//    stages are cut into equal contiguous ranges, one per warp, so every warp
//    streams the same number of bytes through its own ring of bulk copies. A
//    warp keeps the 32 best pairs of the current row piece spread over its
//    lanes and stores the list when it leaves the row; when it leaves a
//    sequence it counts itself in, and the warp that completes the count
//    finalises that sequence: it merges the lists of the rows it needs
//    (bitonic merges of sorted lists), builds the restricted distributions in
//    double precision, runs the accept scan and draws the final token in
//    token-index order. That warp also resets the sequence's counter and
//    flags, so the next call finds them zero.
#include "sv_rows.cuh"

namespace sv {

namespace {

constexpr int kRK = kMaxRestrictK;
static_assert(kRK == 32, "one list entry per lane");
constexpr unsigned kAll = 0xffffffffu;

struct SortEnt {
    int32_t i;
    int32_t pad;
    double w;
};

__device__ __forceinline__ TopK shfl_topk(const TopK &t, int src) {
    return TopK{__shfl_sync(kAll, t.v, src), __shfl_sync(kAll, t.i, src)};
}

// The 32 best of two sorted lists (lane j holds the j-th best of each): the
// better of a_j and b_{31-j} forms a bitonic sequence holding the 32 best,
// which five compare-exchange stages sort.
__device__ __forceinline__ TopK merge_lists(TopK a, TopK b, int lane) {
    const TopK br = shfl_topk(b, 31 - lane);
    TopK c = topk_better(a.v, a.i, br.v, br.i) ? a : br;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const TopK o = TopK{__shfl_xor_sync(kAll, c.v, off), __shfl_xor_sync(kAll, c.i, off)};
        const bool low = (lane & off) == 0;
        if (low == topk_better(o.v, o.i, c.v, c.i)) c = o;
    }
    return c;
}

__device__ __forceinline__ TopK load_part(const RTop *p) {
    const float2 e = __ldcg(reinterpret_cast<const float2 *>(p));
    return TopK{e.x, __float_as_int(e.y)};
}

// A restricted distribution from a row's sorted list (lane j: the j-th best).
struct RDist {
    TopK e;      // the lane's entry
    int m;       // kept entries (lanes 0..m-1)
    double pr;   // the lane's probability (0 past m)
};

__device__ __forceinline__ RDist restrict_dist(const TopK &e, double T, int k, double top_p,
                                               int lane) {
    const bool valid = lane < k && e.i != INT_MAX;
    const double l0 = (double)__shfl_sync(kAll, e.v, 0);
    // w_j = exp(l_j / T - l_0 / T); -inf logits weigh 0
    const double w = valid ? exp((double)e.v / T - l0 / T) : 0.0;
    double c = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(kAll, c, off);
        if (lane >= off) c += y;
    }
    const int nvalid = __popc(__ballot_sync(kAll, valid));  // valid lanes are a prefix
    const double total = __shfl_sync(kAll, c, nvalid - 1);
    // the shortest prefix whose probability reaches top_p (the last valid lane always does)
    const uint32_t reach = __ballot_sync(kAll, valid && c / total >= top_p);
    const int m = __ffs(reach);
    const double z = __shfl_sync(kAll, c, m - 1);
    return RDist{e, m, lane < m ? w / z : 0.0};
}

__device__ __forceinline__ double prob_of(const RDist &d, int32_t x, int lane) {
    const uint32_t hit = __ballot_sync(kAll, lane < d.m && d.e.i == x);
    const double p = __shfl_sync(kAll, d.pr, hit ? __ffs(hit) - 1 : 0);
    return hit ? p : 0.0;
}

}  // namespace

// ---------------------------------------------------------------------------
// plan: validation and the row layout

__global__ void __launch_bounds__(1024) restrict_plan_kernel(RestrictParams R) {
    __shared__ int32_t s_wsum[32];
    __shared__ int32_t s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gm = R.gamma_max;
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (int32_t c0 = 0; c0 < R.B; c0 += 1024) {
        const int32_t b = c0 + tid;
        int32_t cnt = 0, g = 0, bad = 0;
        int64_t po = 0, qo = 0;
        if (b < R.B) {
            g = R.gamma[b];
            if (g < 0 || g > gm) {
                bad = SPECVERIFY_STATUS_BAD_GAMMA;
            } else {
                po = R.p_row_off[b];
                if (po < 0 || po + g + 1 > R.target_rows) bad |= SPECVERIFY_STATUS_BAD_ROW;
                if (g > 0) {
                    qo = R.q_row_off[b];
                    if (qo < 0 || qo + g > R.draft_rows) bad |= SPECVERIFY_STATUS_BAD_ROW;
                }
                for (int i = 0; i < g; ++i) {
                    const int32_t x = R.tokens[(int64_t)b * gm + i];
                    if (x < 0 || (int64_t)x >= R.V) bad |= SPECVERIFY_STATUS_BAD_TOKEN;
                }
                const float T = R.temperature[b];
                const int32_t k = R.top_k[b];
                const float tp = R.top_p ? R.top_p[b] : 1.0f;
                if (!(T > 0.0f && T < INFINITY) || k < 1 || k > kRK || !(tp > 0.0f && tp <= 1.0f))
                    bad |= SPECVERIFY_STATUS_BAD_PARAM;
            }
            cnt = bad ? 0 : 2 * g + 1;
        }
        // exclusive scan of the row counts over the CTA
        int32_t x = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(kAll, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t v = s_wsum[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t y = __shfl_up_sync(kAll, v, off);
                if (lane >= off) v += y;
            }
            s_wsum[lane] = v;
        }
        __syncthreads();
        const int32_t base = s_carry + (warp > 0 ? s_wsum[warp - 1] : 0) + x - cnt;
        if (b < R.B) {
            if (bad) {
                atomicOr(R.status, bad);
                R.n_out[b] = -1;
                for (int i = 0; i <= gm; ++i) R.tok_out[(int64_t)b * (gm + 1) + i] = -1;
            } else {
                const char *p0 = R.target + po * R.stride_bytes;
                for (int j = 0; j <= g; ++j)
                    R.rows[base + j] =
                        RRow{p0 + (int64_t)j * R.stride_bytes, b, (uint16_t)j, (uint16_t)cnt};
                const char *q0 = R.draft + qo * R.stride_bytes;
                for (int i = 0; i < g; ++i)
                    R.rows[base + g + 1 + i] = RRow{q0 + (int64_t)i * R.stride_bytes, b,
                                                    (uint16_t)(g + 1 + i), (uint16_t)cnt};
            }
        }
        __syncthreads();
        if (tid == 0) s_carry += s_wsum[31];
        __syncthreads();
    }
    if (tid == 0) *R.total_rows = s_carry;
}

// ---------------------------------------------------------------------------
// rows and finalisation

namespace {

// Geometry of the stage split: stage s of the call is stage s % spr of row
// s / spr; warp w streams stages [w range, (w + 1) range).
struct Split {
    int64_t spr, range;
    __device__ int64_t warp_of(int64_t s) const { return s / range; }
    __device__ int64_t first_row(int64_t w) const { return w * range / spr; }
};

// The sorted list of row rr: the merge of the pieces of every warp that
// streamed part of it.
__device__ __forceinline__ TopK row_list(const RestrictParams &R, const Split &sp, int64_t rr,
                                         int lane) {
    const int64_t wf = sp.warp_of(rr * sp.spr), wl = sp.warp_of((rr + 1) * sp.spr - 1);
    TopK acc{-INFINITY, INT_MAX};
    for (int64_t w0 = wf; w0 <= wl; w0 += 4) {
        TopK l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t w = w0 + u;
            const int64_t k = rr - sp.first_row(w);
            l[u] = w <= wl && k < R.cap ? load_part(R.parts + (w * R.cap + k) * kRK + lane)
                                        : TopK{-INFINITY, INT_MAX};
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (w0 + u <= wl) acc = (w0 + u == wf) ? l[u] : merge_lists(acc, l[u], lane);
    }
    return acc;
}

// Sequence b is complete: rows base..base+cnt-1 have all been streamed.
__device__ __forceinline__ void finalize(const RestrictParams &R, const Split &sp, int32_t b,
                                         int64_t base, int cnt, SortEnt *scratch, int lane) {
    __threadfence();
    const int gm = R.gamma_max;
    const int g = (cnt - 1) / 2;
    const uint32_t flag = __ldcg(&R.seq_flag[b]);
    bool fin = true;
    for (int c = lane; c < cnt; c += 32) fin &= __ldcg(&R.row_fin[base + c]) != 0u;
    fin = __all_sync(kAll, fin);
    // leave the counters and flags zero for the next call
    for (int c = lane; c < cnt; c += 32) R.row_fin[base + c] = 0u;
    if (lane == 0) {
        R.seq_flag[b] = 0u;
        R.seq_ctr[b] = 0u;
    }
    int32_t *tok = R.tok_out + (int64_t)b * (gm + 1);
    if (flag != 0u || !fin) {
        for (int i = lane; i <= gm; i += 32) tok[i] = -1;
        if (lane == 0) {
            R.n_out[b] = -1;
            atomicOr(R.status, (flag & 2u) ? SPECVERIFY_STATUS_TIMEOUT : SPECVERIFY_STATUS_BAD_LOGIT);
        }
        return;
    }
    const double T = (double)R.temperature[b];
    const int k = (int)min((int64_t)R.top_k[b], R.V);
    const double top_p = R.top_p ? (double)R.top_p[b] : 1.0;
    const int32_t *x = R.tokens + (int64_t)b * gm;

    // the accept scan on the restricted distributions
    int n = g;
    RDist dp{}, dq{};
    for (int i = 0; i < g; ++i) {
        const TopK lp = row_list(R, sp, base + i, lane);
        const TopK lq = row_list(R, sp, base + g + 1 + i, lane);
        dp = restrict_dist(lp, T, k, top_p, lane);
        dq = restrict_dist(lq, T, k, top_p, lane);
        const int32_t xi = x[i];
        const double px = prob_of(dp, xi, lane), qx = prob_of(dq, xi, lane);
        const double ratio = qx > 0.0 ? px / qx : (px > 0.0 ? INFINITY : 0.0);
        if (accept_uniform(R.seed, (uint32_t)b, (uint32_t)(i + 1)) > ratio) {
            n = i;
            break;
        }
    }

    // the final token: from norm(max(0, p' - q')) after a rejection, else from p'
    double d;
    bool zero_mass = false;
    if (n < g) {
        double qv = 0.0;
        for (int t = 0; t < 32; ++t) {
            const int32_t qi = __shfl_sync(kAll, dq.e.i, t);
            const double qp = __shfl_sync(kAll, dq.pr, t);
            if (t < dq.m && qi == dp.e.i) qv = qp;
        }
        d = lane < dp.m ? fmax(0.0, dp.pr - qv) : 0.0;
        if (!__any_sync(kAll, d > 0.0)) {
            d = dp.pr;
            zero_mass = true;
        }
    } else {
        dp = restrict_dist(row_list(R, sp, base + g, lane), T, k, top_p, lane);
        d = dp.pr;
    }
    // order the kept tokens by index
    int rank = 0;
    for (int t = 0; t < 32; ++t) {
        const int32_t oi = __shfl_sync(kAll, dp.e.i, t);
        rank += (t < dp.m && oi < dp.e.i) ? 1 : 0;
    }
    if (lane < dp.m) scratch[rank] = SortEnt{dp.e.i, 0, d};
    __syncwarp();
    const SortEnt e = lane < dp.m ? scratch[lane] : SortEnt{INT_MAX, 0, 0.0};
    __syncwarp();
    double c = e.w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(kAll, c, off);
        if (lane >= off) c += y;
    }
    const double total = __shfl_sync(kAll, c, dp.m - 1);
    const double t_u = draw_uniform(R.seed, (uint32_t)b, (uint32_t)(n + 1)) * total;
    const uint32_t hit = __ballot_sync(kAll, lane < dp.m && c > t_u);
    // (t_u below the total always hits but for rounding: then the last token of positive weight)
    const int sel = hit ? __ffs(hit) - 1
                        : 31 - __clz(__ballot_sync(kAll, lane < dp.m && e.w > 0.0));
    const int32_t token = __shfl_sync(kAll, e.i, sel);
    for (int i = lane; i <= gm; i += 32) tok[i] = i < n ? x[i] : (i == n ? token : -1);
    if (lane == 0) {
        R.n_out[b] = n;
        if (zero_mass) atomicOr(R.status, SPECVERIFY_STATUS_DRAW_ZERO_MASS);
    }
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kRestrictWarps * 32, 1) restrict_kernel(RestrictParams R) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kRestrictWarps][kFeatSlots];
    __shared__ __align__(16) SortEnt s_sort[kRestrictWarps][32];
    static_assert(kRestrictWarps * kFeatSlots * kFeatSlotBytes == kFeatSmem, "ring size");
    constexpr int PV = DT == SV_DT_FP32 ? 4 : 8;
    constexpr int ESZ = DT == SV_DT_FP32 ? 4 : 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bar0 = smem_u32(&bars[warp][0]);
    uint8_t *wbuf = smem + warp * kFeatSlots * kFeatSlotBytes;
    if (lane == 0) {
        for (int s = 0; s < kFeatSlots; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();  // a warp uses only its own barriers and scratch

    const int64_t total = *R.total_rows;
    Split sp;
    sp.spr = (R.row_bytes + kFeatSlotBytes - 1) / kFeatSlotBytes;
    const int64_t nwarps = (int64_t)gridDim.x * kRestrictWarps;
    sp.range = (total * sp.spr + nwarps - 1) / nwarps;
    const int64_t w = (int64_t)blockIdx.x * kRestrictWarps + warp;
    const int64_t s0 = w * sp.range;
    const int64_t s1 = min(total * sp.spr, s0 + sp.range);
    if (s0 >= s1) return;
    const int64_t r_first = s0 / sp.spr, r_last = (s1 - 1) / sp.spr;

    // the warp's rows, one per lane (rows past the first 32 are loaded when needed)
    RRow mine{nullptr, 0, 0, 0};
    if (r_first + lane <= r_last) mine = R.rows[r_first + lane];
    auto row_at = [&](int64_t rr) -> RRow {
        const int d = (int)min(rr - r_first, (int64_t)32);
        const unsigned long long a =
            __shfl_sync(kAll, reinterpret_cast<unsigned long long>(mine.addr), d & 31);
        const int32_t bb = __shfl_sync(kAll, mine.b, d & 31);
        const uint32_t jc =
            __shfl_sync(kAll, ((uint32_t)mine.cnt << 16) | (uint32_t)mine.j, d & 31);
        if (d < 32)
            return RRow{reinterpret_cast<const char *>(a), bb, (uint16_t)(jc & 0xffffu),
                        (uint16_t)(jc >> 16)};
        return R.rows[rr];
    };

    TopK t{-INFINITY, INT_MAX};
    float kth = -INFINITY;
    bool bad = false;
    int64_t cur = r_first;

    // store the list of row rr; count in when the warp leaves rr's sequence
    auto close_row = [&](int64_t rr, uint32_t extra) {
        const RRow row = row_at(rr);
        uint32_t flag = extra | (__any_sync(kAll, bad) ? 1u : 0u);
        const int64_t k = rr - r_first;
        if (k < R.cap)
            R.parts[(w * R.cap + k) * kRK + lane] = RTop{t.v, t.i};
        else
            flag |= 2u;  // not reachable: cap bounds the rows of any warp
        const float top = __shfl_sync(kAll, t.v, 0);
        if (lane == 0) {
            if (flag) atomicOr(&R.seq_flag[row.b], flag);
            if (top > -INFINITY) R.row_fin[rr] = 1u;
        }
        if (rr == r_last || (int)row.j + 1 == (int)row.cnt) {
            __threadfence();
            __syncwarp();
            const int64_t base = rr - row.j;
            const int64_t wf = sp.warp_of(base * sp.spr);
            const int64_t wl = sp.warp_of((base + row.cnt) * sp.spr - 1);
            uint32_t old = 0;
            if (lane == 0) old = atomicAdd(&R.seq_ctr[row.b], 1u);
            old = __shfl_sync(kAll, old, 0);
            if ((int64_t)old + 1 == wl - wf + 1)
                finalize(R, sp, row.b, base, row.cnt, s_sort[warp], lane);
        }
        t = TopK{-INFINITY, INT_MAX};
        kth = -INFINITY;
        bad = false;
    };

    auto src = [&](int64_t kk, const char *&ptr, int &bytes) {
        const int64_t s = s0 + kk;
        const int64_t rr = s / sp.spr;
        const int64_t off = (s - rr * sp.spr) * kFeatSlotBytes;
        ptr = row_at(rr).addr + off;
        bytes = (int)min((int64_t)kFeatSlotBytes, R.row_bytes - off);
    };

    auto body = [&](const uint8_t *slot, int64_t kk, const char *ptr, int bytes) {
        const int64_t s = s0 + kk;
        const int64_t rr = s / sp.spr;
        while (cur < rr) close_row(cur++, 0u);
        const int64_t e0 = (s - rr * sp.spr) * (kFeatSlotBytes / ESZ);
        const uint4 *vb = reinterpret_cast<const uint4 *>(slot);
        const int nvec = bytes >> 4;
        for (int j = 0; j < kFeatSlotBytes / 16 / 32; ++j) {
            const int vi = lane + 32 * j;
            if (__all_sync(kAll, vi >= nvec)) break;
            float f[PV];
            if (vi < nvec) {
                vec_floats<DT>(vb[vi], f);
            } else {
#pragma unroll
                for (int e = 0; e < PV; ++e) f[e] = -INFINITY;
            }
            float g = f[0];
#pragma unroll
            for (int e = 1; e < PV; ++e) g = max_nan(g, f[e]);
            bad |= !(g < INFINITY);  // a NaN or +inf logit
            topk_offer<kRK>(t, kth, f, PV, vi < nvec ? g : __int_as_float(0x7fffffff),
                            e0 + (int64_t)vi * PV, R.V, lane);
        }
        const int rem = (bytes & 15) / ESZ;
        if (rem > 0) {
            const int64_t e = e0 + (int64_t)nvec * PV + lane;
            float f1[1] = {tail_logit<DT>(ptr - e0 * ESZ, e, lane < rem)};
            bad |= !(f1[0] < INFINITY);
            topk_offer<kRK>(t, kth, f1, 1, f1[0], e, R.V, lane);
        }
    };

    uint32_t parity = 0;
    const bool ok = ring_stream_list(s1 - s0, wbuf, bar0, parity, lane, src, body);
    // the last row, or (after a wait gave up) every row not closed yet
    while (cur <= r_last) close_row(cur++, ok ? 0u : 2u);
}

// ---------------------------------------------------------------------------
// launchers

cudaError_t prepare_restricted() {
    cudaError_t e = cudaFuncSetAttribute(restrict_kernel<SV_DT_FP32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kFeatSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(restrict_kernel<SV_DT_BF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kFeatSmem);
    return e;
}

cudaError_t launch_restrict_plan(const RestrictParams &p, cudaStream_t s) {
    restrict_plan_kernel<<<1, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_restrict(const RestrictParams &p, int dtype, int num_ctas, cudaStream_t s) {
    if (dtype == SV_DT_FP32)
        restrict_kernel<SV_DT_FP32><<<num_ctas, kRestrictWarps * 32, kFeatSmem, s>>>(p);
    else
        restrict_kernel<SV_DT_BF16><<<num_ctas, kRestrictWarps * 32, kFeatSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sv
