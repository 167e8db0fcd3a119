// sv_rows.cuh -- building blocks of the kernels that read whole rows beside
// the verify step (row diagnostics, restricted sampling): warp rings of
// shared-memory slots filled by 1-D bulk asynchronous copies, over the
// stages of a CTA's row or over a warp's range of a split of every row's
// stages; per-lane softmax statistics (with an optional entropy
// accumulator); the warp's exact K best (logit, token) pairs, sorted lists
// and their bitonic merges.
#pragma once

#include <climits>

#include "sv_stream.cuh"
#include "sv_rows_params.h"

namespace sv {

namespace rows {

constexpr int kFeatWarps = 16;
constexpr int kFeatSlots = 3;
constexpr int kFeatSlotBytes = 4096;
constexpr int kFeatSmem = kFeatWarps * kFeatSlots * kFeatSlotBytes;  // 192 KiB
constexpr float kXMin = -1000.0f;  // exponents below this weigh 0 (and keep 0 * x finite)

}  // namespace rows

using rows::kFeatWarps;
using rows::kFeatSlots;
using rows::kFeatSlotBytes;
using rows::kFeatSmem;
using rows::kXMin;

// ---------------------------------------------------------------------------
// thread-block clusters: rank, barrier and distributed shared memory

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// the address of the same shared-memory variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// the warp's ring

// Streams stages s_begin, s_begin + s_step, ... (while 0 <= s < the stage
// count; s_step may be negative) of NR rows (stage s covers bytes
// [s SB, (s + 1) SB) of each row, the last one ragged) through the warp's
// kFeatSlots slots of NR * SB bytes; every lane then calls
// body(slot, s, bytes). parity: one bit per slot, kept across calls (a slot's
// barrier completes once per use). Returns false when a wait gave up (after
// draining the copies it issued, with bounded waits).
template <int NR, int SB, class Body>
__device__ bool ring_stream(const char *const *rows, int64_t nbytes, int64_t s_begin,
                            int64_t s_step, uint8_t *wbuf, uint32_t bar0, uint32_t &parity,
                            int lane, Body &&body) {
    static_assert(NR * SB == kFeatSlotBytes, "a slot holds one stage of every row");
    const int64_t nst = (nbytes + SB - 1) / SB;
    int64_t p_s = s_begin;
    auto issue = [&](int slot) -> bool {
        if (p_s < 0 || p_s >= nst) return false;
        const int64_t off = p_s * SB;
        const uint32_t tma = (uint32_t)min((int64_t)SB, nbytes - off) & ~15u;
        if (lane == 0) {
            const uint32_t bar = bar0 + 8 * slot;
            if (tma > 0) {
                mbar_arrive_expect_tx(bar, tma * NR);
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    bulk_load(smem_u32(wbuf + slot * kFeatSlotBytes + r * SB), rows[r] + off, tma,
                              bar);
            } else {
                mbar_arrive(bar);
            }
        }
        p_s += s_step;
        return true;
    };
    int inflight = 0;
    for (int k = 0; k < kFeatSlots; ++k) inflight += issue(k) ? 1 : 0;
    int c_slot = 0;
    int64_t c_s = s_begin;
    bool ok = true;
    while (inflight > 0) {
        if (!mbar_wait_bounded(bar0 + 8 * c_slot, (parity >> c_slot) & 1u)) {
            ok = false;
            break;
        }
        parity ^= 1u << c_slot;
        --inflight;
        const int bytes = (int)min((int64_t)SB, nbytes - c_s * SB);
        body(wbuf + c_slot * kFeatSlotBytes, c_s, bytes);
        __syncwarp();
        inflight += issue(c_slot) ? 1 : 0;
        c_s += s_step;
        if (++c_slot == kFeatSlots) c_slot = 0;
    }
    if (!ok) {
        // drain what is in flight (bounded), so that no copy outlives the kernel
        while (inflight > 0) {
            if (!mbar_wait_bounded(bar0 + 8 * c_slot, (parity >> c_slot) & 1u)) break;
            parity ^= 1u << c_slot;
            --inflight;
            if (++c_slot == kFeatSlots) c_slot = 0;
        }
    }
    return ok;
}

// ---------------------------------------------------------------------------
// a warp's share of a row-stage split

// The rows' stages (kFeatSlotBytes each, the last of a row ragged) are
// numbered s = row * spr + st; the split cuts them into ranges of `range`
// stages, NQ ranges per warp: warp w streams ranges w, w + nw, w + 2 nw, ...
// A row piece is the part of one row inside one range.
struct SplitCur {
    int q, st, k;          // range of the warp, stage of the row, row of the range
    int64_t s, s_end, rr;  // stage of the split, end of the range, row
    bool live;
};

// Streams warp w's ranges through its ring: stage(c, slot, bytes) for every
// stage (every lane, the stage's bytes in shared memory at slot), then
// close(c, extra) after the last stage of each piece, with extra = 0; after
// a wait gave up, every piece not finished is closed with extra = 2 and the
// copies in flight are drained (bounded). row_addr(c) is the address of row
// c.rr (every lane calls it with the same c).
template <int NQ, class RowAddr, class Stage, class Close>
__device__ void split_stream(int64_t w, int64_t nw, int64_t range, int64_t spr, int64_t S,
                             int64_t row_bytes, uint8_t *wbuf, uint32_t bar0, int lane,
                             RowAddr &&row_addr, Stage &&stage, Close &&close) {
    constexpr int SB = kFeatSlotBytes;
    auto enter = [&](SplitCur &c, int q) {
        c.q = q;
        c.s = q < NQ ? (w + (int64_t)q * nw) * range : S;
        c.live = c.s < S;
        if (!c.live) return;
        c.s_end = min(S, c.s + range);
        c.rr = c.s / spr;
        c.st = (int)(c.s - c.rr * spr);
        c.k = 0;
    };
    auto next_stage = [&](SplitCur &c) {
        if (++c.s == c.s_end) {
            enter(c, c.q + 1);
        } else if (++c.st == spr) {
            c.st = 0;
            ++c.rr;
            ++c.k;
        }
    };
    auto stage_bytes = [&](const SplitCur &c) -> int {
        return (int)min((int64_t)SB, row_bytes - (int64_t)c.st * SB);
    };
    SplitCur p, c;
    enter(p, 0);
    enter(c, 0);
    auto issue = [&](int slot) -> bool {
        if (!p.live) return false;
        const int bytes = stage_bytes(p);
        const char *src = row_addr(p) + (int64_t)p.st * SB;
        const uint32_t tma = (uint32_t)bytes & ~15u;
        if (lane == 0) {
            const uint32_t bar = bar0 + 8 * slot;
            if (tma > 0) {
                mbar_arrive_expect_tx(bar, tma);
                bulk_load(smem_u32(wbuf + slot * SB), src, tma, bar);
            } else {
                mbar_arrive(bar);
            }
        }
        next_stage(p);
        return true;
    };
    uint32_t parity = 0;
    int inflight = 0;
    for (int k = 0; k < kFeatSlots; ++k) inflight += issue(k) ? 1 : 0;
    int c_slot = 0;
    bool ok = true;
    while (inflight > 0) {
        if (!mbar_wait_bounded(bar0 + 8 * c_slot, (parity >> c_slot) & 1u)) {
            ok = false;
            break;
        }
        parity ^= 1u << c_slot;
        --inflight;
        stage(c, wbuf + c_slot * SB, stage_bytes(c));
        __syncwarp();
        inflight += issue(c_slot) ? 1 : 0;
        if (++c_slot == kFeatSlots) c_slot = 0;
        // the piece ends with its row or its range
        if (c.st + 1 == spr || c.s + 1 == c.s_end) close(c, 0u);
        next_stage(c);
    }
    if (!ok) {
        while (c.live) {
            close(c, 2u);
            // to the next piece: the next row of the range, or the next range
            const int64_t row_end = (c.rr + 1) * spr;
            if (row_end >= c.s_end) {
                enter(c, c.q + 1);
            } else {
                c.s = row_end;
                c.st = 0;
                ++c.rr;
                ++c.k;
            }
        }
        while (inflight > 0) {
            if (!mbar_wait_bounded(bar0 + 8 * c_slot, (parity >> c_slot) & 1u)) break;
            parity ^= 1u << c_slot;
            --inflight;
            if (++c_slot == kFeatSlots) c_slot = 0;
        }
    }
}

// the logits of one 16-byte vector (PV of them)
template <int DT>
__device__ __forceinline__ void vec_floats(const uint4 &w, float *f) {
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

// NaN-propagating maximum of the logits of one 16-byte vector
template <int DT>
__device__ __forceinline__ float vec_max(const uint4 &w) {
    if (DT == SV_DT_FP32) {
        return max_nan(max_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                       max_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
    } else {
        uint32_t a, b, m;
        asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(w.x), "r"(w.y));
        asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(w.z), "r"(w.w));
        asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
        return max_nan(bf16_lo(m), bf16_hi(m));
    }
}

// ---------------------------------------------------------------------------
// per-lane softmax statistics with an entropy accumulator

// m: reference (the lane's running maximum logit), s = sum 2^x, t = sum 2^x x
// with x = (l - m) log2(e)/T; bad: a NaN or +inf logit was seen.
struct SoftAcc {
    float m, s, t;
    bool bad;
};

__device__ __forceinline__ SoftAcc soft_init() { return SoftAcc{-INFINITY, 0.0f, 0.0f, false}; }

// Adds n logits whose maximum is g. ENT: also accumulate t.
template <bool ENT>
__device__ __forceinline__ void soft_add(SoftAcc &a, const float *f, int n, float g, float c2) {
    if (g != g || g == INFINITY) {
        a.bad = true;
        return;
    }
    if (g == -INFINITY) return;  // nothing but -inf: weight 0
    if (g > a.m) {
        if (a.m != -INFINITY) {
            const float d = fmaxf((a.m - g) * c2, kXMin);
            const float sc = ex2_approx(d);
            if (ENT) a.t = sc * fmaf(d, a.s, a.t);
            a.s *= sc;
        }
        a.m = g;
    }
    const float mc = a.m * c2;
    // two independent chains (even and odd logits), folded in at the end
    float s0 = 0.0f, s1 = 0.0f, t0 = 0.0f, t1 = 0.0f;
    int e = 0;
    for (; e + 1 < n; e += 2) {
        const float x0 = fmaxf(fmaf(f[e], c2, -mc), kXMin);
        const float x1 = fmaxf(fmaf(f[e + 1], c2, -mc), kXMin);
        const float w0 = ex2_approx(x0), w1 = ex2_approx(x1);
        s0 += w0;
        s1 += w1;
        if (ENT) {
            t0 = fmaf(w0, x0, t0);
            t1 = fmaf(w1, x1, t1);
        }
    }
    if (e < n) {
        const float x0 = fmaxf(fmaf(f[e], c2, -mc), kXMin);
        const float w0 = ex2_approx(x0);
        s0 += w0;
        if (ENT) t0 = fmaf(w0, x0, t0);
    }
    a.s += s0 + s1;
    if (ENT) a.t += t0 + t1;
}

// soft_add with the entropy accumulator for the PV logits of one 16-byte
// vector (g their maximum): the exponent arguments, the sums and the
// entropy products on packed float pairs, two independent chains.
// kClamp: clamp the exponents at kXMin, which keeps a -inf logit (weight 0)
// out of the entropy product as 0 * -inf; without it every logit must be
// finite (bf16 rows have theirs replaced by a finite stand-in first).
template <int PV, bool kClamp = true>
__device__ __forceinline__ void soft_add_vec(SoftAcc &a, const float *f, float g, float c2) {
    if (g != g || g == INFINITY) {
        a.bad = true;
        return;
    }
    if (g == -INFINITY) return;  // nothing but -inf: weight 0
    if (g > a.m) {
        if (a.m != -INFINITY) {
            const float d = fmaxf((a.m - g) * c2, kXMin);
            const float sc = ex2_approx(d);
            a.t = sc * fmaf(d, a.s, a.t);
            a.s *= sc;
        }
        a.m = g;
    }
    const float mc = a.m * c2;
    const f32x2 c2x2 = pack2(c2, c2), nmc = pack2(-mc, -mc);
    f32x2 s = 0ull, t = 0ull;
#pragma unroll
    for (int e = 0; e < PV; e += 2) {
        float2 x = unpack2(fma2(pack2(f[e], f[e + 1]), c2x2, nmc));
        if (kClamp) {
            x.x = fmaxf(x.x, kXMin);
            x.y = fmaxf(x.y, kXMin);
        }
        const f32x2 w = pack2(ex2_approx(x.x), ex2_approx(x.y));
        s = add2(s, w);
        t = fma2(w, pack2(x.x, x.y), t);
    }
    const float2 s2 = unpack2(s), t2 = unpack2(t);
    a.s += s2.x + s2.y;
    a.t += t2.x + t2.y;
}

// Folds b into a (same rules as adding b's logits one by one).
template <bool ENT>
__device__ __forceinline__ void soft_merge(SoftAcc &a, const SoftAcc &b, float c2) {
    a.bad |= b.bad;
    if (b.m == -INFINITY) return;
    if (a.m == -INFINITY) {
        a.m = b.m;
        a.s = b.s;
        a.t = b.t;
        return;
    }
    const float M = fmaxf(a.m, b.m);
    const float da = fmaxf((a.m - M) * c2, kXMin), db = fmaxf((b.m - M) * c2, kXMin);
    const float sa = ex2_approx(da), sb = ex2_approx(db);
    if (ENT) a.t = sa * fmaf(da, a.s, a.t) + sb * fmaf(db, b.s, b.t);
    a.s = sa * a.s + sb * b.s;
    a.m = M;
}

template <bool ENT>
__device__ __forceinline__ SoftAcc soft_shfl_xor(const SoftAcc &a, int off) {
    SoftAcc b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, off);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, off);
    b.t = ENT ? __shfl_xor_sync(0xffffffffu, a.t, off) : 0.0f;
    b.bad = __shfl_xor_sync(0xffffffffu, a.bad ? 1 : 0, off) != 0;
    return b;
}

// The CTA's statistics: warp butterflies, then warp 0 over the warps' totals
// (smem: kFeatWarps entries). Every thread returns the total.
template <bool ENT>
__device__ SoftAcc soft_cta_reduce(SoftAcc a, float c2, SoftAcc *smem, int lane, int warp) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) soft_merge<ENT>(a, soft_shfl_xor<ENT>(a, off), c2);
    if (lane == 0) smem[warp] = a;
    __syncthreads();
    SoftAcc tot = smem[0];
    for (int w = 1; w < kFeatWarps; ++w) soft_merge<ENT>(tot, smem[w], c2);
    __syncthreads();  // smem reusable
    return tot;
}

// Ragged row tail (fewer than 16 bytes after the last whole vector): the
// lanes below `rem` load one logit each.
template <int DT>
__device__ __forceinline__ float tail_logit(const char *row, int64_t e, bool live) {
    return live ? load_logit<DT>(row, e) : -INFINITY;
}

// ---------------------------------------------------------------------------
// warp top-k

// Lane j < K holds the warp's j-th best (value, index): descending values,
// ties by ascending index; empty slots hold (-inf, INT_MAX).
struct TopK {
    float v;
    int32_t i;
};

__device__ __forceinline__ bool topk_better(float av, int32_t ai, float bv, int32_t bi) {
    return av > bv || (av == bv && ai < bi);
}

__device__ __forceinline__ TopK shfl_topk(const TopK &t, int src) {
    return TopK{__shfl_sync(0xffffffffu, t.v, src), __shfl_sync(0xffffffffu, t.i, src)};
}

__device__ __forceinline__ TopK better_of(const TopK &a, const TopK &b) {
    return topk_better(a.v, a.i, b.v, b.i) ? a : b;
}

// Sorts one entry per lane, best first (a bitonic sorting network).
__device__ __forceinline__ TopK sort32(TopK x, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const TopK o{__shfl_xor_sync(0xffffffffu, x.v, j), __shfl_xor_sync(0xffffffffu, x.i, j)};
            const bool keep_better = ((lane & k) == 0) == ((lane & j) == 0);
            const bool ob = topk_better(o.v, o.i, x.v, x.i);
            if (ob == keep_better) x = o;
        }
    }
    return x;
}

// The 32 best of two sorted lists (lane j holds the j-th best of each): the
// better of a_j and b_{31-j} forms a bitonic sequence holding the 32 best,
// which five compare-exchange stages sort.
__device__ __forceinline__ TopK merge_lists(TopK a, TopK b, int lane) {
    TopK c = better_of(a, shfl_topk(b, 31 - lane));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const TopK o{__shfl_xor_sync(0xffffffffu, c.v, off), __shfl_xor_sync(0xffffffffu, c.i, off)};
        const bool low = (lane & off) == 0;
        if (low == topk_better(o.v, o.i, c.v, c.i)) c = o;
    }
    return c;
}

// Exact K best (K <= 32) of the logits a warp streams. The warp keeps a
// sorted list of its 32 best so far (lane j: the j-th), a threshold kth that
// bounds its K-th best from below, and up to 64 candidates in shared memory
// that passed the threshold when they were seen. Each group of logits (one
// lane's 16-byte vector) is tested by its maximum alone; only groups that
// pass test their logits, and every 32 buffered candidates are sorted and
// merged into the list, which raises the threshold. A logit equal to the
// threshold value passes only with a lower index: with low-precision logits
// many tokens tie there. Before the list has K entries the threshold is the
// smallest group maximum of the warp's first full set of groups (32 distinct
// tokens at least that large exist, so the K-th best is no smaller).
template <int K>
struct WarpTopK {
    TopK list;
    TopK kth;
    int cnt;
    TopK *buf;  // 64 entries of shared memory, the warp's own

    __device__ void reset() {
        list = TopK{-INFINITY, INT_MAX};
        kth = TopK{-INFINITY, INT_MAX};
        cnt = 0;
    }

    __device__ __forceinline__ bool passes(float v, int32_t i) const {
        return v > kth.v || (v == kth.v && i < kth.i);
    }

    // merge buffered entries [0, n) (n <= 32) into the list
    __device__ void merge_buffer(int n, int lane) {
        __syncwarp();
        const TopK x = lane < n ? buf[lane] : TopK{-INFINITY, INT_MAX};
        list = merge_lists(list, sort32(x, lane), lane);
        kth = better_of(shfl_topk(list, K - 1), kth);
        const int rest = cnt - n;
        const TopK y = lane < rest ? buf[32 + lane] : TopK{};
        __syncwarp();
        if (lane < rest) buf[lane] = y;
        __syncwarp();
        cnt = rest;
    }

    // One group per lane: n logits f[0..n) of tokens i0.. (none past i_end),
    // g their maximum (NaN never passes).
    __device__ __forceinline__ void offer(const float *f, int n, float g, int32_t i0,
                                          int32_t i_end, int lane) {
        if (kth.v == -INFINITY) {
            // no bound yet: the smallest group maximum of a full set of groups
            float m = g == g ? g : -INFINITY;  // a lane without a group (NaN) gives no bound
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fminf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (m > -INFINITY && m < INFINITY) kth = TopK{m, INT_MAX};
        }
        const bool cand = passes(g, i0);
        if (!__any_sync(0xffffffffu, cand)) return;
        for (int e = 0; e < n; ++e) {
            const int32_t i = i0 + e;
            const bool q = cand && i < i_end && passes(f[e], i);
            const uint32_t mask = __ballot_sync(0xffffffffu, q);
            if (q) buf[cnt + __popc(mask & ((1u << lane) - 1u))] = TopK{f[e], i};
            cnt += __popc(mask);
            if (cnt >= 32) merge_buffer(32, lane);
        }
    }

    // Pushes the logits f[e] with bit e of qm set (tokens i0 + e), all lanes
    // at once: a warp scan of the counts gives every lane its place. A round
    // with more than 32 pushes takes the element-by-element path instead.
    template <int PV>
    __device__ __forceinline__ void push_mask(const float *f, uint32_t qm, int32_t i0,
                                              int32_t i_end, int lane) {
        const int c = __popc(qm);
        int incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (total == 0) return;
        if (total > 32) {
            offer(f, PV, qm ? INFINITY : __int_as_float(0x7fffffff), i0, i_end, lane);
            return;
        }
        int at = cnt + incl - c;  // cnt < 32, so cnt + total < 64
#pragma unroll
        for (int e = 0; e < PV; ++e)
            if (qm & (1u << e)) buf[at++] = TopK{f[e], i0 + e};
        cnt += total;
        if (cnt >= 32) merge_buffer(32, lane);
    }

    // One stage of the row in shared memory: vectors vb[lane + 32 j] (j < NJ;
    // those at or past nvec absent) hold the logits of tokens
    // e0 + (lane + 32 j) PV + e. The vectors are first tested by their maxima
    // alone; only the lanes whose vectors pass expand them, one vector per lane
    // per round. While there is no bound yet, a full stage gives one: each
    // lane's maximum is a distinct token, so the K-th best is at least the
    // smallest of them. Returns whether a NaN or +inf logit was seen.
    template <int DT, int NJ>
    __device__ __forceinline__ bool offer_stage(const uint4 *vb, int nvec, int32_t e0,
                                                int32_t i_end, int lane) {
        constexpr int PV = DT == SV_DT_FP32 ? 4 : 8;
        float g[NJ];
        bool bad = false;
        float lmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int vi = lane + 32 * j;
            g[j] = vi < nvec ? vec_max<DT>(vb[vi]) : __int_as_float(0x7fffffff);
            bad |= vi < nvec && !(g[j] < INFINITY);
            lmax = fmaxf(lmax, g[j]);  // (fmaxf skips NaN)
        }
        if (kth.v == -INFINITY && nvec == NJ * 32) {
            float m = lmax;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                m = fminf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (m > -INFINITY && m < INFINITY) kth = TopK{m, INT_MAX};
        }
        uint32_t mask = 0;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            if (passes(g[j], e0 + (lane + 32 * j) * PV)) mask |= 1u << j;
        while (__any_sync(0xffffffffu, mask != 0u)) {
            float f[PV];
            int32_t i0 = 0;
            uint32_t qm = 0;
            if (mask) {
                const int j = __ffs(mask) - 1;
                mask &= mask - 1;
                vec_floats<DT>(vb[lane + 32 * j], f);
                i0 = e0 + (lane + 32 * j) * PV;
#pragma unroll
                for (int e = 0; e < PV; ++e)
                    if (i0 + e < i_end && passes(f[e], i0 + e)) qm |= 1u << e;
            } else {
#pragma unroll
                for (int e = 0; e < PV; ++e) f[e] = -INFINITY;
            }
            push_mask<PV>(f, qm, i0, i_end, lane);
        }
        return bad;
    }

    // the final list (lane j: the j-th best)
    __device__ TopK finish(int lane) {
        if (cnt > 0) merge_buffer(cnt, lane);
        return list;
    }
};

}  // namespace sv
