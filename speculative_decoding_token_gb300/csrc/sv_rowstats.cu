// sv_rowstats.cu -- plan kernel and row-statistics kernel of the verify step.
//
// Plan (greedy calls and the no-allocation entry point; a sampling call of
// specverify_verify plans inside its fused kernel): CTA 0 validates gamma,
// row offsets and draft tokens per sequence ("Dynamic Speculation Lookahead
// ...", Sec. 3: the lookahead varies per iteration, so gamma is ragged),
// numbers the logical rows sequence-major (p_1..p_{gamma+1}, then
// q_1..q_gamma when sampling) and resets the draw counters. The other CTAs
// write -1 into every output slot and build the call's bf16 weight table
// (bf16 sampling). Every loop is flat and coalesced.
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
#include <algorithm>

#include "sv_draw.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// plan

// Work of the fill CTAs (1 .. gridDim.x - 1), none of which depends on the
// validation: the bf16 weight table and the -1 of every token output slot.
// Flat, coalesced loops.
__device__ void plan_fill(const Params &P, int64_t t, int64_t nt) {
    if (P.code_tab) build_code_table(P.code_tab, P.exp2_tab, P.c2h, P.c2l, (int)t, (int)nt);
    const int64_t nout = (int64_t)P.B * (P.gamma_max + 1);
    for (int64_t i = t; i < nout; i += nt) P.tok_out[i] = -1;
}

// Sequences handled per pass of the plan CTA.
constexpr int kPlanTile = 1024;

__global__ void __launch_bounds__(kPlanTile) plan_kernel(const __grid_constant__ Params P) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry_s;
    __shared__ int32_t s_g[kPlanTile], s_bad[kPlanTile], s_rows[kPlanTile], s_base[kPlanTile];
    __shared__ int64_t s_po[kPlanTile], s_qo[kPlanTile];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x > 0) {
        plan_fill(P, (int64_t)(blockIdx.x - 1) * blockDim.x + tid, (int64_t)(gridDim.x - 1) * blockDim.x);
        return;
    }
    if (tid == 0) carry_s = 0;
    __syncthreads();
    const int gm = P.gamma_max;
    for (int base = 0; base < P.B; base += kPlanTile) {
        const int tile = min(kPlanTile, P.B - base);
        // gamma and the row offsets of sequence base + tid
        if (tid < tile) {
            const int b = base + tid;
            const int32_t g = P.gamma[b];
            const int64_t po = P.p_row_off[b];
            const int64_t qo = P.sampling ? P.q_row_off[b] : 0;
            int32_t bad = 0;
            if (g < 0 || g > gm) {
                bad = SPECVERIFY_STATUS_BAD_GAMMA;
            } else {
                if (po < 0 || po + g + 1 > P.target_rows) bad = SPECVERIFY_STATUS_BAD_ROW;
                if (P.sampling && g > 0 && (qo < 0 || qo + g > P.draft_rows)) bad |= SPECVERIFY_STATUS_BAD_ROW;
            }
            s_g[tid] = bad & SPECVERIFY_STATUS_BAD_GAMMA ? -1 : g;
            s_bad[tid] = bad;
            s_po[tid] = po;
            s_qo[tid] = qo;
        }
        __syncthreads();
        // the draft tokens of the tile, flat over [tile, gamma_max]
        {
            const int64_t nt = (int64_t)tile * gm;
            const int32_t *tk = P.tokens + (int64_t)base * gm;
#pragma unroll 4
            for (int64_t i = tid; i < nt; i += kPlanTile) {
                const int32_t x = __ldg(&tk[i]);
                const int bl = (int)(i / gm);
                const int t = (int)(i - (int64_t)bl * gm);
                if (t < s_g[bl] && (x < 0 || (int64_t)x >= P.V)) atomicOr(&s_bad[bl], SPECVERIFY_STATUS_BAD_TOKEN);
            }
        }
        __syncthreads();
        int32_t rows = 0;
        if (tid < tile) {
            const int b = base + tid;
            const int32_t bad = s_bad[tid];
            const int32_t g = s_g[tid];
            if (bad) atomicOr(P.status, bad);
            rows = bad ? 0 : (g + 1 + (P.sampling ? g : 0));
            P.n_out[b] = -1;
            P.zone_cnt[b] = 0;
            P.draw[b].n = -1;
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
        if (tid < tile) {
            P.seq_base[base + tid] = excl;
            P.seq_rows[base + tid] = rows;
            s_rows[tid] = rows;
            s_base[tid] = excl;
        }
        __syncthreads();
        if (tid == 0) carry_s = carry + warp_sums[(blockDim.x >> 5) - 1];
        // the logical rows, one warp per sequence: p_1..p_{gamma+1}, then
        // q_1..q_gamma when sampling
        for (int bl = warp; bl < tile; bl += kPlanTile / 32) {
            const int32_t nr = s_rows[bl];
            const int32_t g = s_g[bl];
            for (int i = lane; i < nr; i += 32) {
                RowRef r;
                r.phys = i <= g ? s_po[bl] + i : s_qo[bl] + (i - g - 1);
                r.b = base + bl;
                r.j = i <= g ? i : -(i - g);
                P.rows[s_base[bl] + i] = r;
            }
        }
        __syncthreads();
    }
    if (tid == 0) *P.total_rows = carry_s;
}

// One CTA per sequence, after the row-statistics kernel on the same stream.
// Sampling: warp 0 combines the rows (one lane per row) and runs the accept
// scan. Greedy: the warps combine the rows, then warp 0 runs the exact-match
// scan.
template <int DT, int MODE>
__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(const __grid_constant__ Params P) {
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
__global__ void __launch_bounds__(kWarps * 32, 1) rowstats_kernel(const __grid_constant__ Params P) {
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
    // CTA 0 validates and numbers the rows; the others fill, about 8192
    // elements each
    const int64_t fill = (int64_t)p.B * (p.gamma_max + 1) + (p.code_tab ? kCodeTab : 0);
    const int nfill = (int)std::min<int64_t>(std::max<int64_t>((fill + 8191) / 8192, 1), 256);
    plan_kernel<<<1 + nfill, kPlanTile, 0, s>>>(p);
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
