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
// Three launches:
//  - restrict_plan_kernel (one CTA): validates every sequence, writes the
//    outputs of the bad ones, and lays the rows of the good ones out one
//    after another (p_0..p_gamma then q_0..q_{gamma-1} per sequence).
//  - restrict_rows_kernel (one persistent CTA of 16 warps per SM): the rows'
//    4 KiB stages are cut into equal contiguous ranges, kRangesPerWarp per
//    warp, so every warp streams the same number of bytes through its own
//    ring of bulk copies. A warp keeps the 32 best pairs of the current row
//    piece (the part of a row inside one range) spread over its lanes and
//    stores the list when the piece ends. Nothing waits on another warp.
//  - restrict_final_kernel (one CTA per sequence): merges the pieces of each
//    row (bitonic merges of sorted lists) and builds its restricted
//    distribution (float-float weights and sums; one warp per row), runs every
//    position's accept test (one warp per position), and draws the final
//    token in token-index order from the residual or the bonus distribution.
//    It also resets the sequence's flags, so the next call finds them zero.
#include "sv_draw.cuh"
#include "sv_rows.cuh"

namespace sv {

namespace {

constexpr int kRK = kMaxRestrictK;
constexpr int kRangesPerWarp = kRestrictRangesPerWarp;
static_assert(kRK == 32, "one list entry per lane");
constexpr unsigned kAll = 0xffffffffu;

struct SortEnt {
    int32_t i;
    int32_t pad;
    float wh, wl;  // a weight as a float-float
};

__device__ __forceinline__ TopK load_part(const RTop *p) {
    const float2 e = __ldcg(reinterpret_cast<const float2 *>(p));
    return TopK{e.x, __float_as_int(e.y)};
}

// A restricted distribution from a row's sorted list (lane j: the j-th best).
struct RDist {
    TopK e;      // the lane's entry
    int m;       // kept entries (lanes 0..m-1)
    float ph, pl;  // the lane's probability as a float-float (0 past m)
};

// The weights w_j = 2^((l_j - l_0) log2(e) / T), scaled by the constant
// 2^(l_0 c - I) (c = log2(e)/T, I = floor(l_0 c)), come from the
// table-driven float-float exponential of the draw (relative error about
// 1e-13); their prefix sums, the prefix test and the probabilities are
// float-float too (about 48 bits), all on the FP32 pipe: FP64 is a narrow
// pipe on this part. The constant scale cancels in every normalised quantity.
__device__ __forceinline__ RDist restrict_dist(const TopK &e, const ExpRow &er0, float c,
                                               int k, float top_p, const float2 *tab, int lane) {
    const bool valid = lane < k && e.i != INT_MAX;
    const float l0 = __shfl_sync(kAll, e.v, 0);
    ExpRow er = er0;
    {
        float yh, yl;  // l0 c, exactly enough for its floor
        ff_mul(l0, 0.0f, unpack2(er0.ch).x, unpack2(er0.cl).x, yh, yl);
        float fl = floorf(yh);
        if (fl == yh && yl < 0.0f) fl -= 1.0f;
        er.shift = splat2(fl);
    }
    er.lmin = splat2(l0 - 1000.0f / c);
    f32x2 eh, el;
    exp2_pair<true>(pack2(e.v, e.v), er, tab, eh, el);
    // the weight as a normalised float-float (a tail within half an ulp of
    // its head), so that equal sums compare equal below
    float wh = 0.0f, wl = 0.0f;
    if (valid) two_sum(unpack2(eh).x, unpack2(el).x, wh, wl);
    float ch = wh, cl = wl;
    warp_incl_scan_ff(ch, cl, lane);
    const int nvalid = __popc(__ballot_sync(kAll, valid));  // valid lanes are a prefix
    const float zh = __shfl_sync(kAll, ch, nvalid - 1), zl = __shfl_sync(kAll, cl, nvalid - 1);
    // the shortest prefix whose probability reaches top_p, C_j >= top_p Z (the
    // last valid lane always does: there C_j = Z)
    float pzh, pzl;
    ff_mul(zh, zl, top_p, 0.0f, pzh, pzl);
    const uint32_t reach = __ballot_sync(kAll, valid && !ff_gt(pzh, pzl, ch, cl));
    const int m = reach ? __ffs(reach) : nvalid;
    const float mh = __shfl_sync(kAll, ch, m - 1), ml = __shfl_sync(kAll, cl, m - 1);
    RDist d{e, m, 0.0f, 0.0f};
    if (lane < m) ff_div(wh, wl, mh, ml, d.ph, d.pl);
    return d;
}

// a restricted distribution kept in shared memory (lane j's entry at [j])
struct DistCache {
    int32_t idx[32];
    float2 pr[32];
    int m;
};

__device__ __forceinline__ void dist_store(DistCache &c, const RDist &d, int lane) {
    c.idx[lane] = d.e.i;
    c.pr[lane] = make_float2(d.ph, d.pl);
    if (lane == 0) c.m = d.m;
}

__device__ __forceinline__ RDist dist_load(const DistCache &c, int lane) {
    const float2 p = c.pr[lane];
    return RDist{TopK{0.0f, c.idx[lane]}, c.m, p.x, p.y};
}

// the probability of token x (0 outside the kept entries), as a float-float
__device__ __forceinline__ float2 prob_of(const RDist &d, int32_t x, int lane) {
    const uint32_t hit = __ballot_sync(kAll, lane < d.m && d.e.i == x);
    const int src = hit ? __ffs(hit) - 1 : 0;
    const float h = __shfl_sync(kAll, d.ph, src), l = __shfl_sync(kAll, d.pl, src);
    return hit ? make_float2(h, l) : make_float2(0.0f, 0.0f);
}

}  // namespace

// ---------------------------------------------------------------------------
// plan: validation and the row layout

__global__ void __launch_bounds__(1024) restrict_plan_kernel(const __grid_constant__ RestrictParams R) {
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
            R.seq_rows[b] = make_int2(base, cnt);
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
// s / spr; range v of the split covers stages [v range, (v + 1) range).
struct Split {
    int64_t spr, range;
    __device__ int64_t range_of(int64_t s) const { return s / range; }
    __device__ int64_t first_row(int64_t v) const { return v * range / spr; }
};

// The sorted list of row rr: the merge of the pieces of every warp that
// streamed part of it.
__device__ __forceinline__ TopK row_list(const RestrictParams &R, const Split &sp, int64_t rr,
                                         int lane) {
    const int64_t wf = sp.range_of(rr * sp.spr), wl = sp.range_of((rr + 1) * sp.spr - 1);
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

// The final token of sequence b (warp-wide): drawn in token-index order from
// the weights (dh, dl) (lane j: the float-float weight of the lane's entry
// dp.e, 0 past dp.m); prefix sums and t = u * total in float-float.
__device__ __forceinline__ int32_t draw_token(const RDist &dp, float dh, float dl, uint64_t seed,
                                              uint32_t b, uint32_t pos, SortEnt *scratch,
                                              int lane) {
    // order the kept tokens by index
    int rank = 0;
    for (int t = 0; t < 32; ++t) {
        const int32_t oi = __shfl_sync(kAll, dp.e.i, t);
        rank += (t < dp.m && oi < dp.e.i) ? 1 : 0;
    }
    if (lane < dp.m) scratch[rank] = SortEnt{dp.e.i, 0, dh, dl};
    __syncwarp();
    const SortEnt e = lane < dp.m ? scratch[lane] : SortEnt{INT_MAX, 0, 0.0f, 0.0f};
    __syncwarp();
    float ch = e.wh, cl = e.wl;
    warp_incl_scan_ff(ch, cl, lane);
    const float th0 = __shfl_sync(kAll, ch, dp.m - 1), tl0 = __shfl_sync(kAll, cl, dp.m - 1);
    float uh, ul, th, tl;
    draw_uniform_ff(seed, b, pos, uh, ul);
    ff_mul(uh, ul, th0, tl0, th, tl);
    const uint32_t hit = __ballot_sync(kAll, lane < dp.m && ff_gt(ch, cl, th, tl));
    // (t below the total always hits but for rounding: then the last token of positive weight)
    const int sel = hit ? __ffs(hit) - 1
                        : 31 - __clz(__ballot_sync(kAll, lane < dp.m && e.wh > 0.0f));
    return __shfl_sync(kAll, e.i, sel);
}

// the geometry of the row pass's stage split, from the call's row count
__device__ __forceinline__ Split make_split(const RestrictParams &R, int64_t total, int grid) {
    Split sp;
    sp.spr = (R.row_bytes + kFeatSlotBytes - 1) / kFeatSlotBytes;
    const int64_t nv = (int64_t)grid * kRestrictWarps * kRangesPerWarp;
    sp.range = (total * sp.spr + nv - 1) / nv;
    return sp;
}

}  // namespace

// ---------------------------------------------------------------------------
// the row pass

// Each warp streams its ranges of the stage split through its ring and keeps
// the 32 best (logit, token) pairs of each row piece (the part of a row inside
// one range); a piece's list goes to parts[range][row - first row of the
// range]. A NaN or +inf logit marks the sequence (seq_flag bit 0), a finite
// logit marks the row (row_fin); a wait that gave up marks the sequences of
// every piece not finished (bit 1).
template <int DT>
__global__ void __launch_bounds__(kRestrictWarps * 32, 1) restrict_rows_kernel(const __grid_constant__ RestrictParams R) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kRestrictWarps][kFeatSlots];
    __shared__ __align__(16) TopK s_cand[kRestrictWarps][64];
    static_assert(kRestrictWarps * kFeatSlots * kFeatSlotBytes == kFeatSmem, "ring size");
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

    const int64_t total = *R.total_rows;
    const Split sp = make_split(R, total, gridDim.x);
    const int64_t S = total * sp.spr;
    const int64_t nw = (int64_t)gridDim.x * kRestrictWarps;
    const int64_t w = (int64_t)blockIdx.x * kRestrictWarps + warp;
    if (w * sp.range >= S) return;
    const int cap = R.cap;
    // the warp's ranges q = 0..kRangesPerWarp-1 are ranges w + q nw of the split
    auto vr_of = [&](int q) -> int64_t { return w + (int64_t)q * nw; };

    // the warp's rows, lane q cap + k holding row k of range q (others loaded when needed)
    RRow mine{nullptr, 0, 0, 0};
    {
        const int q = lane / cap, k = lane - q * cap;
        if (q < kRangesPerWarp) {
            const int64_t s0 = vr_of(q) * sp.range;
            if (s0 < S) {
                const int64_t rr = s0 / sp.spr + k;
                if (rr <= (min(S, s0 + sp.range) - 1) / sp.spr) mine = R.rows[rr];
            }
        }
    }

    auto row_of = [&](const SplitCur &c) -> RRow {
        const int li = c.q * cap + c.k;
        const int src = li < 32 ? li : 0;
        const unsigned long long a =
            __shfl_sync(kAll, reinterpret_cast<unsigned long long>(mine.addr), src);
        const int32_t bb = __shfl_sync(kAll, mine.b, src);
        if (li < 32) return RRow{reinterpret_cast<const char *>(a), bb, 0, 0};
        return R.rows[c.rr];
    };

    WarpTopK<kRK> tk;
    tk.buf = s_cand[warp];
    tk.reset();
    bool bad = false;
    const int32_t V32 = (int32_t)R.V;
    split_stream<kRangesPerWarp>(
        w, nw, sp.range, sp.spr, S, R.row_bytes, wbuf, bar0, lane,
        [&](const SplitCur &c) { return row_of(c).addr; },
        [&](const SplitCur &c, const uint8_t *slot, int bytes) {
            const int32_t e0 = c.st * (SB / ESZ);
            const uint4 *vb = reinterpret_cast<const uint4 *>(slot);
            const int nvec = bytes >> 4;
            bad |= tk.template offer_stage<DT, SB / 16 / 32>(vb, nvec, e0, V32, lane);
            const int rem = (bytes & 15) / ESZ;
            if (rem > 0) {
                const int32_t e = e0 + nvec * PV + lane;
                float f1[1] = {tail_logit<DT>(row_of(c).addr, e, lane < rem)};
                bad |= !(f1[0] < INFINITY);
                tk.offer(f1, 1, f1[0], e, V32, lane);
            }
        },
        // store the list of the piece under cursor c
        [&](const SplitCur &c, uint32_t extra) {
            const TopK t = tk.finish(lane);
            uint32_t flag = extra | (__any_sync(kAll, bad) ? 1u : 0u);
            if (c.k < cap)
                R.parts[(vr_of(c.q) * cap + c.k) * kRK + lane] = RTop{t.v, t.i};
            else
                flag |= 2u;  // not reachable: cap bounds the rows of any range
            const float top = __shfl_sync(kAll, t.v, 0);
            const int32_t b = row_of(c).b;
            if (lane == 0) {
                if (flag) atomicOr(&R.seq_flag[b], flag);
                if (top > -INFINITY) R.row_fin[c.rr] = 1u;
            }
            tk.reset();
            bad = false;
        });
}

// ---------------------------------------------------------------------------
// finalisation: one CTA per sequence

constexpr int kFinalWarps = 16;
constexpr int kFinalRows = 33;  // rows whose distributions stay in shared memory (gamma <= 16)

__global__ void __launch_bounds__(kFinalWarps * 32) restrict_final_kernel(const __grid_constant__ RestrictParams R) {
    __shared__ uint32_t s_rej[(kMaxGamma + 31) / 32];
    __shared__ uint32_t s_flag;
    __shared__ __align__(16) SortEnt s_sort[32];
    __shared__ DistCache s_dist[kFinalRows];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t b = blockIdx.x;
    const int2 sr = R.seq_rows[b];
    if (sr.y == 0) return;  // a bad sequence: the plan wrote its outputs
    const int64_t base = sr.x;
    const int cnt = sr.y, g = (cnt - 1) / 2, gm = R.gamma_max;
    const Split sp = make_split(R, *R.total_rows, R.row_grid);
    if (threadIdx.x == 0) s_flag = 0u;
    for (int i = threadIdx.x; i < (g + 31) / 32; i += blockDim.x) s_rej[i] = 0u;
    // every row must hold a finite logit; the flags are left zero for the next call
    bool fin = true;
    for (int c = threadIdx.x; c < cnt; c += blockDim.x) {
        fin &= R.row_fin[base + c] != 0u;
        R.row_fin[base + c] = 0u;
    }
    // log2(e) / T as a float-float: the log2(e) pair divided by T
    float c2h, c2l;
    ff_div(1.44269502162933349609375f, 1.925963033500011079e-08f, R.temperature[b], 0.0f, c2h,
           c2l);
    ExpRow er;
    er.ch = splat2(c2h);
    er.cl = splat2(c2l);
    const int k = (int)min((int64_t)R.top_k[b], R.V);
    const float top_p = R.top_p ? R.top_p[b] : 1.0f;
    const int32_t *x = R.tokens + (int64_t)b * gm;
    // row j of the sequence: p_j for j <= g, q_{j-g-1} after
    auto row_dist = [&](int j) -> RDist {
        return restrict_dist(row_list(R, sp, base + j, lane), er, c2h, k, top_p, R.exp2_tab, lane);
    };
    auto cached = [&](int j) -> RDist {
        return j < kFinalRows ? dist_load(s_dist[j], lane) : row_dist(j);
    };

    // the restricted distribution of every row, one warp per row (the work
    // of a sequence with bad rows is discarded)
    for (int j = warp; j < min(cnt, kFinalRows); j += kFinalWarps)
        dist_store(s_dist[j], row_dist(j), lane);
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t f = R.seq_flag[b];
        R.seq_flag[b] = 0u;
        if (f) atomicOr(&s_flag, f);
    }
    if (!fin) atomicOr(&s_flag, 1u);
    // the accept test of every position, one warp per position
    for (int i = warp; i < g; i += kFinalWarps) {
        const RDist dp = cached(i), dq = cached(g + 1 + i);
        const int32_t xi = x[i];
        // p'(x) / q'(x) in float (about 1e-7 relative: far inside the accept
        // test's flag band); +inf when q'(x) = 0 < p'(x), 0 when both are 0
        const float px = prob_of(dp, xi, lane).x, qx = prob_of(dq, xi, lane).x;
        const float ratio = qx > 0.0f ? px / qx : (px > 0.0f ? INFINITY : 0.0f);
        if (lane == 0 && accept_uniform(R.seed, (uint32_t)b, (uint32_t)(i + 1)) > ratio)
            atomicOr(&s_rej[i >> 5], 1u << (i & 31));
    }
    __syncthreads();
    if (warp != 0) return;
    const uint32_t flag = s_flag;
    int32_t *tok = R.tok_out + (int64_t)b * (gm + 1);
    if (flag != 0u) {
        for (int i = lane; i <= gm; i += 32) tok[i] = -1;
        if (lane == 0) {
            R.n_out[b] = -1;
            atomicOr(R.status, (flag & 2u) ? SPECVERIFY_STATUS_TIMEOUT : SPECVERIFY_STATUS_BAD_LOGIT);
        }
        return;
    }
    // n: the first rejection (the tests after it do not count)
    int n = g;
    for (int c = 0; c < (g + 31) / 32; ++c) {
        const uint32_t m = s_rej[c];
        if (m) {
            n = c * 32 + __ffs(m) - 1;
            break;
        }
    }
    // the final token: from norm(max(0, p' - q')) after a rejection, else from p'
    const RDist dp = cached(n);
    float dh = dp.ph, dl = dp.pl;
    bool zero_mass = false;
    if (n < g) {
        const RDist dq = cached(g + 1 + n);
        float qh = 0.0f, ql = 0.0f;
        for (int t = 0; t < 32; ++t) {
            const int32_t qi = __shfl_sync(kAll, dq.e.i, t);
            const float h = __shfl_sync(kAll, dq.ph, t), l = __shfl_sync(kAll, dq.pl, t);
            if (t < dq.m && qi == dp.e.i) {
                qh = h;
                ql = l;
            }
        }
        // max(0, p' - q') as a float-float
        ff_add(dp.ph, dp.pl, -qh, -ql, dh, dl);
        if (lane >= dp.m || !(dh > 0.0f || (dh == 0.0f && dl > 0.0f))) dh = dl = 0.0f;
        if (!__any_sync(kAll, dh > 0.0f)) {
            dh = dp.ph;
            dl = dp.pl;
            zero_mass = true;
        }
    }
    const int32_t token =
        draw_token(dp, dh, dl, R.seed, (uint32_t)b, (uint32_t)(n + 1), s_sort, lane);
    for (int i = lane; i <= gm; i += 32) tok[i] = i < n ? x[i] : (i == n ? token : -1);
    if (lane == 0) {
        R.n_out[b] = n;
        if (zero_mass) atomicOr(R.status, SPECVERIFY_STATUS_DRAW_ZERO_MASS);
    }
}

// ---------------------------------------------------------------------------
// launchers

cudaError_t prepare_restricted() {
    cudaError_t e = cudaFuncSetAttribute(restrict_rows_kernel<SV_DT_FP32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kFeatSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(restrict_rows_kernel<SV_DT_BF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kFeatSmem);
    return e;
}

cudaError_t launch_restrict_plan(const RestrictParams &p, cudaStream_t s) {
    restrict_plan_kernel<<<1, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_restrict_rows(const RestrictParams &p, int dtype, cudaStream_t s) {
    if (dtype == SV_DT_FP32)
        restrict_rows_kernel<SV_DT_FP32><<<p.row_grid, kRestrictWarps * 32, kFeatSmem, s>>>(p);
    else
        restrict_rows_kernel<SV_DT_BF16><<<p.row_grid, kRestrictWarps * 32, kFeatSmem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_restrict_final(const RestrictParams &p, cudaStream_t s) {
    restrict_final_kernel<<<p.B, kFinalWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sv
