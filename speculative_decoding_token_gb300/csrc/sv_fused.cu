// sv_fused.cu -- the sampling verify step as one persistent kernel.
//
// One cooperative CTA per SM. Its first kFusedStreamWarps warps stream the
// rows in position-major order (p_1 and q_1 of every sequence, then p_2 and
// q_2, ...; sv_stream.cuh), storing one partial per chunk. The warp that
// stores the last partial of a position queues that position for its test.
// One more warp serves position tests only; every streaming warp, once its
// stream is done (and any warp beyond the tester from the start), runs from
// two queues:
//   position tests: combine the two rows, the accept test of that position
//     ("DistillSpec" Algorithm A.1); the first rejection decides the
//     sequence (n = k - 1), as does the bonus row after gamma acceptances;
//     the warp that decides it writes the draw descriptor and queues the
//     sequence's pass tasks;
//   draw tasks: a pass over a span of chunks of the draw rows; the warp that
//     finishes a sequence's last pass runs its finalize, which draws the
//     token (sv_draw.cuh).
// When no logsumexp output is requested, rows after a sequence's first known
// rejection are skipped: they cannot change n or any token. The first warps
// to finish their stream start on the ALU-heavy draw of the sequences
// decided so far while the others still stream, so the HBM-bound stream and
// the issue-bound draw share every SM.
//
// Progress: a queue slot is claimed only once published; a position test
// waits only for partials already stored; no warp waits for a pass (the
// last one to finish runs the finalize); streaming warps wait on nothing
// but their own copies. Every wait is still bounded by about two seconds of
// wall time, after which it sets SPECVERIFY_STATUS_TIMEOUT and marks the call
// aborted, and every other wait of the call returns at once.
#include <climits>

#include "sv_draw.cuh"

namespace sv {

constexpr int kUndecided = -1, kBadSeq = -2;

// Is sequence b decided by the position results so far? Returns n, or
// kUndecided, or kBadSeq (the whole warp; lane L reads positions L + 1,
// L + 33, ...). Streaming only the needed rows, the first position that is
// not accepted decides (a rejection at k gives n = k - 1; a bad row makes the
// sequence bad); with every row streamed, every position must be tested
// first and a bad row anywhere makes the sequence bad.
__device__ int decide_scan(const Params &P, int b, int g, int lane) {
    const uint32_t *res = P.pos_res + (int64_t)b * P.G;
    int first_open = INT_MAX, first_rej = INT_MAX, first_bad = INT_MAX;
    for (int k0 = 1; k0 <= g + 1; k0 += 32) {
        const int k = k0 + lane;
        const uint32_t r = k <= g + 1 ? ld_volatile_u32(&res[k - 1]) : 1u;
        const uint32_t open = __ballot_sync(0xffffffffu, r == 0u);
        const uint32_t rej = __ballot_sync(0xffffffffu, r == 2u);
        const uint32_t bad = __ballot_sync(0xffffffffu, r == 3u);
        if (open && first_open == INT_MAX) first_open = k0 + __ffs(open) - 1;
        if (rej && first_rej == INT_MAX) first_rej = k0 + __ffs(rej) - 1;
        if (bad && first_bad == INT_MAX) first_bad = k0 + __ffs(bad) - 1;
    }
    if (P.skip) {
        const int first = min(first_open, min(first_rej, first_bad));
        if (first == INT_MAX) return g;  // every position accepted, bonus row ready
        if (first == first_open) return kUndecided;
        if (first == first_bad) return kBadSeq;
        return first - 1;
    }
    if (first_open != INT_MAX) return kUndecided;
    if (first_bad != INT_MAX) return kBadSeq;
    return first_rej == INT_MAX ? g : first_rej - 1;
}

// The (max, sum) statistics of logical row lrow, folded from its chunk
// partials in chunk order -- the same fold, so the same values, as the test
// of the row's position. Lane i waits (bounded) until chunks i, i + 32, ...
// are stored: a stored partial is recognised by its value, so this needs no
// ordering against the warp that tested the position. Returns false if the
// wait gave up (the call is then aborted).
__device__ bool row_stats_from_partials(const Params &P, int lrow, int lane, float2 &out) {
    const int cpr = P.cpr;
    const float2 *pp = P.partials + (int64_t)lrow * cpr;
    uint32_t ok = 1;
    const uint64_t t0 = global_ns();
    for (int i = lane; i < cpr && ok; i += 32) {
        while (ld_relaxed_f2(&pp[i]).y == kPartialPending) {
            __nanosleep(64);
            if (call_aborted(P) || global_ns() - t0 > P.wait_ns) {
                ok = 0;
                break;
            }
        }
    }
    if (!__all_sync(0xffffffffu, ok)) return false;
    float2 st = make_float2(0.0f, 0.0f);
    if (lane == 0) {
        float m = -INFINITY, ssum = 0.0f;
        bool nan = false;
        for (int c = 0; c < cpr; ++c) combine_step(ld_relaxed_f2(&pp[c]), P.c2, m, ssum, nan);
        const bool bad = nan || !(m > -INFINITY && m < INFINITY) || !(ssum > 0.0f) ||
                         ssum == INFINITY;
        st = bad ? make_float2(__int_as_float(0x7fffffff), __int_as_float(0x7fffffff))
                 : make_float2(m, ssum);
    }
    out = make_float2(__shfl_sync(0xffffffffu, st.x, 0), __shfl_sync(0xffffffffu, st.y, 0));
    return true;
}

// Sets up the draw of decided sequence b (n accepted drafts) and queues its
// draw tasks: the accepted tokens, the draw descriptor (rows p_{n+1} and, for
// a residual draw, q_{n+1} with their row statistics), then its pass tasks.
// sp, sq: the statistics of those rows when the caller has them
// (have_stats, the caller tested position n + 1), else they are folded again
// from the rows' chunk partials.
template <int DT>
__device__ void start_draw(const Params &P, int b, int g, int base, int n, bool have_stats,
                           float2 sp, float2 sq, int lane) {
    const int gm = P.gamma_max;
    if (!have_stats) {
        bool ok = row_stats_from_partials(P, base + n, lane, sp);
        if (ok && n < g) ok = row_stats_from_partials(P, base + g + 1 + n, lane, sq);
        if (!ok) {
            if (lane == 0) abort_call(P);
            return;
        }
    }
    for (int i = lane; i < n; i += 32)
        P.tok_out[(int64_t)b * (gm + 1) + i] = __ldg(&P.tokens[(int64_t)b * gm + i]);
    if (lane == 0) {
        DrawDesc d;
        d.n = n;
        d.residual = n < g ? 1 : 0;
        d.p_phys = P.p_row_off[b] + n;
        d.Mp = sp.x;
        d.Sp = sp.y;
        if (d.residual) {
            d.q_phys = P.q_row_off[b] + n;
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
        __threadfence();
    }
    uint32_t slot0 = 0;
    const int per = P.ntask;
    if (lane == 0) slot0 = atomicAdd(&P.ctr[kCtrDqTail * kCtrStride], (uint32_t)per);
    slot0 = __shfl_sync(0xffffffffu, slot0, 0);
    __syncwarp();
    for (int c = lane; c < per; c += 32)
        st_release_u64(&P.dq_slot[slot0 + c], ((unsigned long long)P.epoch << 32) | (uint32_t)(b * per + c));
}

// The decision encoded by a sequence's state word (G <= 32): bit k - 1 set
// for an accepted position k (or a ready bonus row), bit 31 + k for a
// rejected one, both for a bad row. Same rules as decide_scan.
__device__ __forceinline__ int decide_bits(unsigned long long w, int g, bool skip) {
    const uint32_t lo = (uint32_t)w, hi = (uint32_t)(w >> 32);
    const uint32_t valid = g + 1 >= 32 ? 0xFFFFFFFFu : (1u << (g + 1)) - 1u;
    const uint32_t acc = lo & ~hi & valid, rej = hi & ~lo & valid, bad = lo & hi & valid;
    const uint32_t open = ~(lo | hi) & valid;
    if (skip) {
        const uint32_t notacc = valid & ~acc;
        if (notacc == 0u) return g;
        const int f = __ffs(notacc) - 1;  // position f + 1
        if (open & (1u << f)) return kUndecided;
        if (bad & (1u << f)) return kBadSeq;
        return f;
    }
    if (open) return kUndecided;
    if (bad) return kBadSeq;
    return rej ? __ffs(rej) - 1 : g;
}

// The test of position k of sequence b ("DistillSpec" Algorithm A.1: accept
// x_k when r_k <= p_k(x_k) / q_k(x_k)), once every chunk partial of its rows
// is stored; position gamma_b + 1 (the bonus row p_{gamma+1}) only needs its
// statistics. Then the decision of b, and, by the one warp that makes it, the
// start of b's draw. Independent loads are issued before the waits, and the
// rows are combined from the partial values the wait itself read.
template <int DT>
__device__ void test_position(const Params &P, uint32_t pi, int lane) {
    const int b = (int)(pi / (uint32_t)P.G);
    const int k = (int)(pi - (uint32_t)b * (uint32_t)P.G) + 1;
    if (P.skip && ld_volatile_u32(&P.decided[b]) != 0u) return;  // nothing left to decide
    const int g = P.gamma[b];
    const int base = P.seq_base[b];
    const bool two = k <= g;
    const int lp = base + k - 1;
    const int lq = base + g + k;
    const int cpr = P.cpr;
    // the logits of x_k (lane 0), loaded while the partials are awaited
    float lpv = 0.0f, lqv = 0.0f;
    if (lane == 0 && two) {
        const int32_t x = __ldg(&P.tokens[(int64_t)b * P.gamma_max + (k - 1)]);
        lpv = load_logit<DT>(P.target + (P.p_row_off[b] + k - 1) * P.stride_bytes, x);
        lqv = load_logit<DT>(P.draft + (P.q_row_off[b] + k - 1) * P.stride_bytes, x);
    }
    // every partial of the position's rows is stored; wait until visible.
    // Lane i watches chunk i (and i + 32, ...) of both rows.
    float2 mp_ = make_float2(-INFINITY, 0.0f), mq_ = make_float2(-INFINITY, 0.0f);
    {
        uint32_t ok = 1;
        const uint64_t t0 = global_ns();
        for (int i = lane; i < cpr && ok; i += 32) {
            const float2 *fp = &P.partials[(int64_t)lp * cpr + i];
            const float2 *fq = &P.partials[(int64_t)lq * cpr + i];
            for (;;) {
                mp_ = ld_relaxed_f2(fp);
                if (two) mq_ = ld_relaxed_f2(fq);
                if (mp_.y != kPartialPending && (!two || mq_.y != kPartialPending)) break;
                __nanosleep(64);
                if (call_aborted(P) || global_ns() - t0 > P.wait_ns) {
                    ok = 0;
                    break;
                }
            }
        }
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) abort_call(P);
            return;
        }
    }
    // row statistics in chunk order: lane 0 row p_k, lane 1 row q_k
    float m = -INFINITY, ssum = 0.0f;
    bool nan = false;
    if (cpr <= 32) {
        for (int c = 0; c < cpr; ++c) {
            const float2 vp = make_float2(__shfl_sync(0xffffffffu, mp_.x, c),
                                          __shfl_sync(0xffffffffu, mp_.y, c));
            const float2 vq = make_float2(__shfl_sync(0xffffffffu, mq_.x, c),
                                          __shfl_sync(0xffffffffu, mq_.y, c));
            combine_step(lane == 0 ? vp : vq, P.c2, m, ssum, nan);
        }
    }
    float2 st = make_float2(0.0f, 0.0f);
    if (lane == 0) st = cpr <= 32 ? finish_row(P, lp, m, ssum, nan) : combine_one_row(P, lp);
    if (lane == 1 && two) st = cpr <= 32 ? finish_row(P, lq, m, ssum, nan) : combine_one_row(P, lq);
    const float2 sp = make_float2(__shfl_sync(0xffffffffu, st.x, 0), __shfl_sync(0xffffffffu, st.y, 0));
    const float2 sq = make_float2(__shfl_sync(0xffffffffu, st.x, 1), __shfl_sync(0xffffffffu, st.y, 1));
    int n = kUndecided;
    if (lane == 0) {
        const bool bad = sp.y != sp.y || (two && sq.y != sq.y);
        uint32_t res = bad ? 3u : 1u;
        if (!bad && two) {
            const float ratio = accept_ratio(P, lpv, lqv, sp, sq);
            if (accept_uniform(P.seed, (uint32_t)b, (uint32_t)k) > ratio) {
                res = 2u;
                if (P.skip) atomicMin(&P.first_rej[b], k);
            }
        }
        if (P.G <= 32) {
            // one atomic update of the sequence's state word: the warp that
            // moves it from undecided to decided starts the draw
            const unsigned long long mine =
                ((res & 2u) ? 1ull << (31 + k) : 0ull) | ((res & 1u) ? 1ull << (k - 1) : 0ull);
            const unsigned long long old = atomicOr(&P.seq_state[b], mine);
            const int n_old = decide_bits(old, g, P.skip != 0);
            const int n_new = decide_bits(old | mine, g, P.skip != 0);
            n = n_old == kUndecided ? n_new : kUndecided;
        } else {
            P.pos_res[pi] = res;
            // a concurrent test of the same sequence sees this result, or
            // this warp sees that one's
            __threadfence();
        }
    }
    if (P.G > 32) {
        __syncwarp();
        n = decide_scan(P, b, g, lane);
        if (lane == 0 && n != kUndecided && atomicCAS(&P.decided[b], 0u, 1u) != 0u) n = kUndecided;
    }
    n = __shfl_sync(0xffffffffu, n, 0);
    if (n != kUndecided && lane == 0) P.decided[b] = 1u;
    if (n == kBadSeq) {
        if (lane == 0) {
            atomicOr(P.status, SPECVERIFY_STATUS_BAD_LOGIT);
            atomicAdd(&P.ctr[kCtrDone * kCtrStride], 1u);
        }
    } else if (n >= 0) {
        start_draw<DT>(P, b, g, base, n, n + 1 == k, sp, sq, lane);
    }
}

// The warp's tickets on the two queues.
struct WarpQueues {
    Ticket rq, dq;
};

// Runs a queued position test if the warp's ticket on that queue is served.
template <int DT>
__device__ __forceinline__ bool try_position(const Params &P, WarpQueues &q, int lane) {
    ticket_take(P, kCtrRqHead, kCtrRqTail, (uint32_t)P.B * (uint32_t)P.G, q.rq, lane);
    const uint32_t pi = ticket_item(P, P.rq_slot, q.rq, lane);
    if (pi == kNoItem) return false;
    test_position<DT>(P, pi, lane);
    return true;
}

// Runs a queued draw task if the warp's ticket on that queue is served: a
// pass over chunks of sequence b; the warp that finishes b's last pass then
// runs b's finalize, which completes the sequence.
template <int DT>
__device__ bool try_draw(const Params &P, WarpQueues &q, const float2 *tab, const float2 *ct,
                         uint8_t *ring, int lane) {
    const uint32_t per = (uint32_t)P.ntask;
    // a ticket taken ahead: a draw task published later is taken after one
    // poll of its slot instead of a look at the tail and a claim
    ticket_take_ahead(P, kCtrDqHead, (uint32_t)P.B * per, q.dq, lane);
    const uint32_t v = ticket_item(P, P.dq_slot, q.dq, lane);
    if (v == kNoItem) return false;
    const int b = (int)(v / per);
    const int c = (int)(v - (uint32_t)b * per);
    const DrawDesc d = load_desc(&P.draw[b]);
    pass_task<DT>(P, b, c, d, tab, ct, ring, lane);
    // the chunk totals and listed tokens of every lane, then the count
    __threadfence();
    __syncwarp();
    uint32_t last = 0;
    if (lane == 0) {
        last = atomicSub(&P.pass_left[b], 1u) == 1u ? 1u : 0u;
        if (last) __threadfence();  // the other passes' results, before they are read
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return true;
    finalize_task<DT>(P, b, d, tab, ct, ring, lane);
    if (lane == 0) {
        __threadfence();
        atomicAdd(&P.ctr[kCtrDone * kCtrStride], 1u);
    }
    return true;
}

// The task loop: position tests first, then draw tasks, until every
// sequence is done (or the call is aborted, or nothing happened for about
// two seconds).
template <int DT>
__device__ void run_tasks(const Params &P, const float2 *tab, const float2 *ct, uint8_t *ring,
                          int lane) {
    WarpQueues q{{0u, false, false}, {0u, false, false}};
    uint64_t idle_since = global_ns();
    uint32_t backoff = 64;  // idle polling backs off up to 256 ns (measured faster than 2 us)
    for (;;) {
        if (try_position<DT>(P, q, lane) || try_draw<DT>(P, q, tab, ct, ring, lane)) {
            idle_since = global_ns();
            backoff = 64;
            continue;
        }
        uint32_t stop = 0;
        if (lane == 0) {
            if (ld_volatile_u32(&P.ctr[kCtrDone * kCtrStride]) >= (uint32_t)P.B || call_aborted(P)) {
                stop = 1;
            } else if (global_ns() - idle_since > P.wait_ns) {
                abort_call(P);
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return;
        __nanosleep(backoff);
        if (backoff < 256) backoff *= 2;
    }
}

// The tester warp of a CTA: position tests only, always holding a ticket
// taken ahead, so a queued position waits about one poll for its test.
template <int DT>
__device__ void run_tester(const Params &P, int lane) {
    Ticket t{0u, false, false};
    const uint32_t cap = (uint32_t)P.B * (uint32_t)P.G;
    uint64_t idle_since = global_ns();
    for (;;) {
        ticket_take_ahead(P, kCtrRqHead, cap, t, lane);
        const uint32_t pi = ticket_item(P, P.rq_slot, t, lane);
        if (pi != kNoItem) {
            test_position<DT>(P, pi, lane);
            idle_since = global_ns();
            continue;
        }
        uint32_t stop = 0;
        if (lane == 0) {
            if (t.dead || ld_volatile_u32(&P.ctr[kCtrDone * kCtrStride]) >= (uint32_t)P.B ||
                call_aborted(P)) {
                stop = 1;
            } else if (global_ns() - idle_since > P.wait_ns) {
                abort_call(P);
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return;
        __nanosleep(64);
    }
}

// ---------------------------------------------------------------------------
// prologue: the call's plan, spread over every CTA

// Grid-wide barrier of the cooperative launch on counter `bar`: every CTA
// adds one and waits (bounded) until `target` CTAs have arrived. The call
// uses one of two counters (by the parity of its epoch) and clears the other
// one for the next call, so no counter is ever cleared while in use.
__device__ bool grid_sync(const Params &P, unsigned long long *bar, uint64_t target) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        atomicAdd(bar, 1ull);
        int ok = 1;
        const uint64_t t0 = global_ns();
        while (ld_acquire_u64(bar) < target) {
            if (call_aborted(P) || global_ns() - t0 > P.wait_ns) {
                abort_call(P);
                ok = 0;
                break;
            }
            __nanosleep(32);
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// The per-call state a sampling call needs before it streams, built by every
// CTA of the fused kernel (a separate plan launch used to do it). Phase A,
// grid-strided: validate gamma, row offsets and draft tokens of every
// sequence ("Dynamic Speculation Lookahead ..." Sec. 3: gamma varies per
// sequence), reset its state and outputs, mark every chunk partial pending,
// clear the position counters and build the bf16 weight table. Phase B,
// after a grid barrier: every CTA tallies the valid sequences by gamma (in
// shared memory) and writes, for its own slice of sequences, their logical
// rows (p_1..p_{gamma+1}, q_1..q_gamma, numbered sequence-major) and their
// slots in the dense position-major stream order (the rows of position k
// before those of k + 1; within a position the pairs (p_k, q_k) of the
// sequences with gamma >= k by descending gamma, then the lone bonus rows p_k
// of those with gamma = k - 1). A second barrier, and the stream starts.
// Returns false if a barrier gave up (the call is then aborted).
__device__ bool fused_prologue(const Params &P, uint8_t *scratch) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * nt + tid, gnt = (int64_t)gridDim.x * nt;
    const int gm = P.gamma_max, G = P.G;
    unsigned long long *bar = P.grid_bar + (P.epoch & 1u) * kCtrStride;
    unsigned long long *bar_next = P.grid_bar + ((P.epoch + 1u) & 1u) * kCtrStride;

    // ---- phase A
    if (gtid == 0) *bar_next = 0ull;
    if (gtid < kNumCtr) P.ctr[gtid * kCtrStride] = 0u;
    for (int64_t b = gtid; b < P.B; b += gnt) {
        const int32_t g = P.gamma[b];
        int32_t bad = 0;
        if (g < 0 || g > gm) {
            bad = SPECVERIFY_STATUS_BAD_GAMMA;
        } else {
            const int64_t po = P.p_row_off[b];
            if (po < 0 || po + g + 1 > P.target_rows) bad = SPECVERIFY_STATUS_BAD_ROW;
            if (g > 0) {
                const int64_t qo = P.q_row_off[b];
                if (qo < 0 || qo + g > P.draft_rows) bad |= SPECVERIFY_STATUS_BAD_ROW;
            }
            for (int i = 0; i < g; ++i) {
                const int32_t x = __ldg(&P.tokens[b * gm + i]);
                if (x < 0 || (int64_t)x >= P.V) bad |= SPECVERIFY_STATUS_BAD_TOKEN;
            }
        }
        if (bad) atomicOr(P.status, bad);
        P.seq_info[b] = bad ? -1 : g;
        P.n_out[b] = -1;
        P.zone_cnt[b] = 0;
        P.draw[b].n = -1;
        P.first_rej[b] = G + 1;
        P.decided[b] = bad ? 1u : 0u;
        P.seq_state[b] = 0ull;
        P.pass_left[b] = (uint32_t)P.ntask;
    }
    {
        const int64_t nout = (int64_t)P.B * (gm + 1);
        for (int64_t i = gtid; i < nout; i += gnt) P.tok_out[i] = -1;
        const int64_t npos = (int64_t)P.B * G;
        for (int64_t i = gtid; i < npos; i += gnt) {
            P.pos_cnt[i] = 0u;
            P.pos_res[i] = 0u;
        }
        const int64_t npart = (int64_t)P.B * (2 * gm + 1) * P.cpr;
        for (int64_t i = gtid; i < npart; i += gnt) P.partials[i] = make_float2(0.0f, kPartialPending);
        if (P.code_tab) build_code_table(P.code_tab, P.exp2_tab, P.c2h, P.c2l, (int)gtid, (int)gnt);
    }
    if (!grid_sync(P, bar, gridDim.x)) return false;

    // ---- phase B: tallies in shared memory (scratch)
    int32_t *s_hist = reinterpret_cast<int32_t *>(scratch);   // [G + 1] valid sequences by gamma
    int32_t *s_phist = s_hist + (G + 1);                       // the same before this CTA's slice
    int32_t *s_ge = s_phist + (G + 1);                         // [G + 2] valid with gamma >= v
    int32_t *s_off = s_ge + (G + 2);                           // [G + 2] first slot of position k
    int32_t *s_misc = s_off + (G + 2);                         // rows before the slice, bad count
    const int64_t per = ((int64_t)P.B + gridDim.x - 1) / gridDim.x;
    const int64_t lo = min((int64_t)P.B, (int64_t)blockIdx.x * per);
    const int64_t hi = min((int64_t)P.B, lo + per);
    for (int i = tid; i < 2 * (G + 1); i += nt) s_hist[i] = 0;
    if (tid < 2) s_misc[tid] = 0;
    __syncthreads();
    for (int64_t b = tid; b < P.B; b += nt) {
        const int32_t info = __ldcg(&P.seq_info[b]);
        if (info >= 0) {
            atomicAdd(&s_hist[info], 1);
            if (b < lo) {
                atomicAdd(&s_phist[info], 1);
                atomicAdd(&s_misc[0], 2 * info + 1);
            }
        } else {
            atomicAdd(&s_misc[1], 1);
        }
    }
    __syncthreads();
    if (tid == 0) {
        int32_t ge = 0;
        s_ge[gm + 1] = 0;
        for (int v = gm; v >= 0; --v) {
            ge += s_hist[v];
            s_ge[v] = ge;
        }
        int32_t off = 0;
        for (int k = 1; k <= gm + 1; ++k) {
            s_off[k] = off;
            off += s_ge[k - 1] + s_ge[k];
        }
        if (blockIdx.x == 0) {
            *P.total_rows = off;
            if (s_misc[1] > 0) atomicAdd(&P.ctr[kCtrDone * kCtrStride], (uint32_t)s_misc[1]);
        }
    }
    __syncthreads();
    for (int64_t b = lo + tid; b < hi; b += nt) {
        const int32_t g = __ldcg(&P.seq_info[b]);
        // logical rows of the sequences before b, and the sequences with the
        // same gamma before b (for b's rank in descending-gamma order)
        int32_t base = s_misc[0], same = 0;
        for (int64_t c = lo; c < b; ++c) {
            const int32_t gc = __ldcg(&P.seq_info[c]);
            if (gc >= 0) base += 2 * gc + 1;
            same += (g >= 0 && gc == g) ? 1 : 0;
        }
        const int32_t rows = g < 0 ? 0 : 2 * g + 1;
        P.seq_base[b] = base;
        P.seq_rows[b] = rows;
        if (g < 0) continue;
        const int64_t po = P.p_row_off[b];
        const int64_t qo = g > 0 ? P.q_row_off[b] : 0;
        for (int i = 0; i < rows; ++i) {
            RowRef r;
            r.phys = i <= g ? po + i : qo + (i - g - 1);
            r.b = (int32_t)b;
            r.j = i <= g ? i : -(i - g);
            P.rows[base + i] = r;
        }
        const int32_t c = s_phist[g] + same;  // place among the sequences with this gamma
        const int32_t rank = s_ge[g + 1] + c;  // rank in descending-gamma order
        for (int k = 1; k <= g + 1; ++k) {
            const bool both = k <= g;
            const int64_t at = both ? s_off[k] + 2 * (int64_t)rank
                                    : s_off[k] + 2 * (int64_t)s_ge[k] + c;
            OrderRef o;
            o.b = (int32_t)b;
            o.pos = k;
            o.need = (both ? 2 : 1) * P.cpr;
            o.pad = 0;
            o.phys = po + k - 1;
            o.j = k - 1;
            o.lrow = base + k - 1;
            P.order[at] = o;
            if (both) {
                o.phys = qo + k - 1;
                o.j = -k;
                o.lrow = base + g + k;
                P.order[at + 1] = o;
            }
        }
    }
    return grid_sync(P, bar, 2ull * gridDim.x);
}

template <int DT>
__global__ void __launch_bounds__(kFusedWarps * 32, 1) fused_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kFusedStreamWarps][kFusedStages];
    __shared__ __align__(8) uint64_t tab_bar;
    __shared__ StageMeta meta[kFusedStreamWarps][kFusedStages];
    // One 32 KiB table lives in shared memory: the bf16 weight table when
    // the call has one (the exponential table is then read from global
    // memory on its rare path), else the exponential table. It arrives by
    // one bulk copy; only its users wait for it, after their stream.
    float2 *stab = reinterpret_cast<float2 *>(smem + kFusedTabOff);
    const float2 *src = P.code_tab ? P.code_tab : P.exp2_tab;
    const float2 *tab = P.code_tab ? P.exp2_tab : stab;
    const float2 *ct = P.code_tab ? stab : nullptr;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t tbar = smem_u32(&tab_bar);
    if (threadIdx.x == 0) {
        mbar_init(tbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp < kFusedStreamWarps && lane == 0) {
        const uint32_t bar0 = smem_u32(&bars[warp][0]);
        for (int s = 0; s < kFusedStages; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the call's plan (the stream rings serve as its scratch), then the
    // table, which phase A may have built, by one bulk copy
    if (!fused_prologue(P, smem)) return;
    if (threadIdx.x == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_expect_tx(tbar, kSmemTab * 8);
        bulk_load(smem_u32(stab), src, kSmemTab * 8, tbar);
    }
    __syncthreads();
    if (warp < kFusedStreamWarps)
        stream_needed<DT, kFusedStages, kFusedStageBytes>(
            P, smem + warp * (kFusedStages * kFusedStageBytes), &meta[warp][0],
            smem_u32(&bars[warp][0]), (int64_t)gridDim.x * kFusedStreamWarps, lane);
    if (warp == kTesterWarp) {
        run_tester<DT>(P, lane);  // position tests use no table
    } else {
        // the draw ring: a streaming warp's stream ring (its bulk copies have
        // all completed), else the task warp's own
        uint8_t *ring = warp < kFusedStreamWarps
                            ? smem + warp * (kFusedStages * kFusedStageBytes)
                            : smem + kFusedDrawRingOff + (warp - kTesterWarp - 1) * kPassRingBytes;
        if (warp < kFusedStreamWarps) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!mbar_wait_bounded(tbar, 0)) {
            if (lane == 0) abort_call(P);
            return;
        }
        run_tasks<DT>(P, tab, ct, ring, lane);
    }
}

cudaError_t launch_fused(const Params &p, int dtype, int num_ctas, cudaStream_t s) {
    Params copy = p;
    void *args[] = {&copy};
    const void *fn = dtype == SV_DT_FP32 ? (const void *)fused_kernel<SV_DT_FP32>
                                         : (const void *)fused_kernel<SV_DT_BF16>;
    return cudaLaunchCooperativeKernel(fn, dim3(num_ctas), dim3(kFusedWarps * 32), args,
                                       kFusedSmem, s);
}

cudaError_t prepare_fused() {
    cudaError_t e = cudaFuncSetAttribute(fused_kernel<SV_DT_FP32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fused_kernel<SV_DT_BF16>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem);
}

}  // namespace sv
