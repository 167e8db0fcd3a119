// sv_rowstats.cu -- plan kernel and row-statistics kernel of the verify step.
//
// Plan (one CTA): validates gamma, row offsets and draft tokens per sequence
// ("Dynamic Speculation Lookahead ...", Sec. 3: the lookahead varies per
// iteration, so gamma is ragged), numbers the logical rows sequence-major
// (p_1..p_{gamma+1}, then q_1..q_gamma when sampling), resets the draw counters
// and writes -1 into every output slot. Before the fused kernel it also marks
// every chunk partial pending and resets the task counter; for bf16 sampling
// it builds the call's bf16 weight table.
//
// Row statistics (persistent, one CTA per SM): streams every logical row
// exactly once, in 32 KiB chunks, each warp through its own ring of
// shared-memory stages filled by 1-D bulk asynchronous copies. Sampling mode
// keeps an online (max, sum of 2^((l - max) log2(e)/T)) per lane -- the
// temperature softmax normaliser of "Speculative Decoding and Distillation"
// (Kadimisetty notes, Part 2), applied to target and draft alike
// ("DistillSpec" App. B.3); greedy mode keeps the first argmax of the raw
// logits. Each warp stores one partial per chunk and synchronises with no
// other warp, so the stream never waits on a memory fence.
//
// Accept (one CTA per sequence, after the row statistics on the same
// stream): its warps combine the chunk partials of the sequence's rows in a
// fixed order, then one warp runs the accept scan ("DistillSpec" Algorithm
// A.1: rejection thresholds p/q, uniforms, n; the rule
// n = min({i-1 : r_i > p_i(x)/q_i(x)} U {gamma}) of the Leviathan et al.
// explainer), or, greedy, the exact-match scan (Kadimisetty notes, "Greedy vs
// sampling").
#include "sv_draw.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// plan

__global__ void __launch_bounds__(1024) plan_kernel(Params P) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry_s = 0;
        if (P.fused) P.ctr[kCtrDone * kCtrStride] = 0u;  // counts bad sequences below
    }
    if (P.code_tab) build_code_table(P.code_tab, P.exp2_tab, P.c2h, P.c2l, tid, blockDim.x);
    __syncthreads();
    const int gm = P.gamma_max;
    for (int base = 0; base < P.B; base += blockDim.x) {
        const int b = base + tid;
        int32_t rows = 0;
        int32_t g = 0;
        int32_t bad = 0;
        if (b < P.B) {
            g = P.gamma[b];
            if (g < 0 || g > gm) {
                bad = SPECVERIFY_STATUS_BAD_GAMMA;
            } else {
                const int64_t po = P.p_row_off[b];
                if (po < 0 || po + g + 1 > P.target_rows) bad = SPECVERIFY_STATUS_BAD_ROW;
                if (P.sampling && g > 0) {
                    const int64_t qo = P.q_row_off[b];
                    if (qo < 0 || qo + g > P.draft_rows) bad |= SPECVERIFY_STATUS_BAD_ROW;
                }
                // eight loads in flight at a time
                const int32_t *tk = P.tokens + (int64_t)b * gm;
                for (int i0 = 0; i0 < g; i0 += 8) {
                    int32_t x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) x[u] = i0 + u < g ? __ldg(&tk[i0 + u]) : 0;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (x[u] < 0 || (int64_t)x[u] >= P.V) bad |= SPECVERIFY_STATUS_BAD_TOKEN;
                }
            }
            if (bad) atomicOr(P.status, bad);
            rows = bad ? 0 : (g + 1 + (P.sampling ? g : 0));
            P.n_out[b] = -1;
            for (int i = 0; i <= gm; ++i) P.tok_out[(int64_t)b * (gm + 1) + i] = -1;
            P.zone_cnt[b] = 0;
            P.draw[b].n = -1;
            if (P.fused) {
                P.first_rej[b] = P.G + 1;
                P.decided[b] = rows == 0 ? 1u : 0u;  // a bad sequence is done at once
                P.seq_state[b] = 0ull;
                if (rows == 0) atomicAdd(&P.ctr[kCtrDone * kCtrStride], 1u);
                for (int k = 0; k < P.G; ++k) {
                    P.pos_cnt[(int64_t)b * P.G + k] = 0u;
                    P.pos_res[(int64_t)b * P.G + k] = 0u;
                }
            }
        }
        // block-wide exclusive scan of rows
        int32_t incl = rows;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int32_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int32_t carry = carry_s;
        const int32_t excl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + incl - rows;
        if (b < P.B) {
            P.seq_base[b] = excl;
            P.seq_rows[b] = rows;
            if (rows > 0) {
                const int64_t po = P.p_row_off[b];
                for (int i = 0; i <= g; ++i) {
                    RowRef r;
                    r.phys = po + i;
                    r.b = b;
                    r.j = i;
                    P.rows[excl + i] = r;
                }
                if (P.sampling) {
                    const int64_t qo = g > 0 ? P.q_row_off[b] : 0;
                    for (int i = 0; i < g; ++i) {
                        RowRef r;
                        r.phys = qo + i;
                        r.b = b;
                        r.j = -(i + 1);
                        P.rows[excl + g + 1 + i] = r;
                    }
                }
            }
        }
        __syncthreads();
        if (tid == 0) carry_s = carry + warp_sums[(blockDim.x >> 5) - 1];
        __syncthreads();
    }
    if (tid == 0) *P.total_rows = carry_s;
    const int32_t total_rows = carry_s;
    __syncthreads();
    if (P.fused) {
        if (tid < kNumCtr && tid != kCtrDone) P.ctr[tid * kCtrStride] = 0u;
        // the fused kernel's position tests poll the partials of their rows
        const int64_t n = (int64_t)total_rows * P.cpr;
        for (int64_t i = tid; i < n; i += blockDim.x) P.partials[i] = make_float2(0.0f, kPartialPending);
        // the stream order: position-major with fixed slots -- slot
        // (k - 1) * 2B + 2b holds p_k of sequence b, the next slot q_k --
        // so the test of position k of every sequence comes before its
        // later rows are streamed. Slots without a row (past gamma_b + 1,
        // or a bad sequence) have lrow = -1 and are skipped by the stream.
        for (int b = tid; b < P.B; b += blockDim.x) {
            const int32_t g = P.seq_rows[b] > 0 ? P.gamma[b] : -1;
            const int32_t sb = P.seq_base[b];
            const int64_t po = g >= 0 ? P.p_row_off[b] : 0;
            const int64_t qo = g > 0 ? P.q_row_off[b] : 0;
            for (int k = 1; k <= P.G; ++k) {
                const int32_t cnt = g < 0 ? 0 : (k <= g + 1 ? 1 : 0) + (k <= g ? 1 : 0);
                OrderRef o;
                o.b = b;
                o.pos = k;
                o.need = cnt * P.cpr;
                o.pad = 0;
                o.phys = po + (k - 1);
                o.j = k - 1;
                o.lrow = cnt >= 1 ? sb + k - 1 : -1;
                const int64_t slot = (int64_t)(k - 1) * 2 * P.B + 2 * b;
                P.order[slot] = o;
                o.phys = qo + (k - 1);
                o.j = -k;
                o.lrow = cnt == 2 ? sb + g + k : -1;
                P.order[slot + 1] = o;
            }
        }
    }
}

// One CTA per sequence, after the row-statistics kernel on the same stream.
// Sampling: warp 0 combines the rows (one lane per row) and runs the accept
// scan. Greedy: the warps combine the rows, then warp 0 runs the exact-match
// scan.
template <int DT, int MODE>
__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(Params P) {
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rows = P.seq_rows[b];
    if (rows == 0) return;  // bad input: outputs stay -1 from the plan kernel
    const int base = P.seq_base[b];
    if (MODE == 0) {
        // one warp, lanes over rows: the same combine as the fused kernel's
        if (warp == 0) {
            combine_rows_sample(P, base, rows, lane);
            __syncwarp();
            accept_scan_sampling<DT>(P, b, lane);
        }
        return;
    }
    for (int r = warp; r < rows; r += kAcceptThreads / 32) combine_row<MODE>(P, base + r, lane);
    __syncthreads();
    if (warp == 0) accept_scan_greedy(P, b, lane);
}

// ---------------------------------------------------------------------------
// the persistent row-statistics kernel

template <int DT, int MODE>
__global__ void __launch_bounds__(kWarps * 32, 1) rowstats_kernel(Params P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kWarps][kStages];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t bar0 = smem_u32(&bars[warp][0]);
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    stream_items<DT, MODE, kStages, kStageBytes>(P, smem + warp * (kStages * kStageBytes), bar0,
                           (int64_t)blockIdx.x * kWarps + warp, (int64_t)gridDim.x * kWarps, lane);
}

// ---------------------------------------------------------------------------
// launchers

cudaError_t launch_plan(const Params &p, cudaStream_t s) {
    plan_kernel<<<1, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_rowstats(const Params &p, int dtype, int num_ctas, cudaStream_t s) {
    const dim3 grid(num_ctas), block(kWarps * 32);
    if (dtype == SV_DT_FP32) {
        if (p.sampling)
            rowstats_kernel<SV_DT_FP32, 0><<<grid, block, kRowStatsSmem, s>>>(p);
        else
            rowstats_kernel<SV_DT_FP32, 1><<<grid, block, kRowStatsSmem, s>>>(p);
    } else {
        if (p.sampling)
            rowstats_kernel<SV_DT_BF16, 0><<<grid, block, kRowStatsSmem, s>>>(p);
        else
            rowstats_kernel<SV_DT_BF16, 1><<<grid, block, kRowStatsSmem, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_accept(const Params &p, int dtype, cudaStream_t s) {
    const dim3 grid(p.B), block(kAcceptThreads);
    if (dtype == SV_DT_FP32) {
        if (p.sampling)
            accept_kernel<SV_DT_FP32, 0><<<grid, block, 0, s>>>(p);
        else
            accept_kernel<SV_DT_FP32, 1><<<grid, block, 0, s>>>(p);
    } else {
        if (p.sampling)
            accept_kernel<SV_DT_BF16, 0><<<grid, block, 0, s>>>(p);
        else
            accept_kernel<SV_DT_BF16, 1><<<grid, block, 0, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t prepare_rowstats() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(rowstats_kernel<SV_DT_FP32, 0>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kRowStatsSmem)))
        return e;
    if ((e = cudaFuncSetAttribute(rowstats_kernel<SV_DT_FP32, 1>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kRowStatsSmem)))
        return e;
    if ((e = cudaFuncSetAttribute(rowstats_kernel<SV_DT_BF16, 0>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kRowStatsSmem)))
        return e;
    return cudaFuncSetAttribute(rowstats_kernel<SV_DT_BF16, 1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kRowStatsSmem);
}

}  // namespace sv
