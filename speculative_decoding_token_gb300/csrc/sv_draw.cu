// sv_draw.cu -- the final-token draw kernels (sv_draw.cuh holds the tasks).
//
// draw_task_kernel follows the stream kernel of a sampling call: its warps
// claim the pass tasks (sequence b, span of chunks t) in order, and the warp
// that finishes a sequence's last pass runs that sequence's finalize. The
// allocation-free entry point runs the same tasks as two kernels instead: the
// pass kernel (every pass task) and the finalize kernel (one per sequence).
#include "sv_draw.cuh"

namespace sv {

// Both tables into dynamic shared memory by bulk copies (one mbarrier);
// returns the weight table or null.
__device__ const float2 *load_tables(const Params &P, float2 *tab) {
    __shared__ __align__(8) uint64_t tab_bar;
    float2 *ct = tab + kExpTab;
    const uint32_t bar = smem_u32(&tab_bar);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(bar, kExpTab * 8 + (P.code_tab ? kCodeTab * 8 : 0));
        bulk_load(smem_u32(tab), P.exp2_tab, kExpTab * 8, bar);
        if (P.code_tab) bulk_load(smem_u32(ct), P.code_tab, kCodeTab * 8, bar);
    }
    __syncthreads();
    if (!mbar_wait_bounded(bar, 0) && threadIdx.x == 0)
        atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
    return P.code_tab ? ct : nullptr;
}

template <int DT>
__global__ void __launch_bounds__(kDrawWarps * 32) draw_pass_kernel(Params P) {
    extern __shared__ float2 tab[];
    const float2 *ct = load_tables(P, tab);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *ring = reinterpret_cast<uint8_t *>(tab) + kDrawRingOff + warp * kPassRingBytes;
    const int64_t items = (int64_t)P.B * P.ntask;
    for (int64_t it = (int64_t)blockIdx.x * kDrawWarps + warp; it < items;
         it += (int64_t)gridDim.x * kDrawWarps) {
        const int b = (int)(it / P.ntask);
        const int c = (int)(it - (int64_t)b * P.ntask);
        const DrawDesc d = P.draw[b];
        if (d.n < 0) continue;
        pass_task<DT>(P, b, c, d, tab, ct, ring, lane);
    }
}

template <int DT>
__global__ void __launch_bounds__(kDrawWarps * 32) draw_finalize_kernel(Params P) {
    extern __shared__ float2 tab[];
    const float2 *ct = load_tables(P, tab);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *ring = reinterpret_cast<uint8_t *>(tab) + kDrawRingOff + warp * kPassRingBytes;
    const int b = blockIdx.x * kDrawWarps + warp;
    if (b >= P.B) return;
    const DrawDesc d = P.draw[b];
    if (d.n < 0) return;
    finalize_task<DT>(P, b, d, tab, ct, ring, lane);
}

// Two CTAs per SM, kDrawTaskWarps warps each. A warp claims a pass task only
// when it is free to run it: a task claimed ahead would wait behind the
// claimer's current task, which stretches the end of the kernel.
template <int DT>
__global__ void __launch_bounds__(kDrawTaskWarps * 32, 2) draw_task_kernel(Params P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t tab_bar;
    // one 32 KiB table in shared memory: the bf16 weight table when the call
    // has one (the exponential table is then read from global memory on its
    // rare path), else the exponential table
    float2 *stab = reinterpret_cast<float2 *>(smem);
    const float2 *src = P.code_tab ? P.code_tab : P.exp2_tab;
    const float2 *tab = P.code_tab ? P.exp2_tab : stab;
    const float2 *ct = P.code_tab ? stab : nullptr;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t tbar = smem_u32(&tab_bar);
    if (threadIdx.x == 0) {
        mbar_init(tbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(tbar, kSmemTab * 8);
        bulk_load(smem_u32(stab), src, kSmemTab * 8, tbar);
    }
    __syncthreads();
    if (!mbar_wait_bounded(tbar, 0)) {
        if (threadIdx.x == 0) atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
        return;
    }
    uint8_t *ring = smem + kDrawTaskRingOff + warp * kPassRingBytes;
    const uint32_t per = (uint32_t)P.ntask;
    const uint32_t items = (uint32_t)P.B * per;
    for (;;) {
        uint32_t v = 0;
        if (lane == 0) v = atomicAdd(&P.ctr[kCtrDqHead * kCtrStride], 1u);
        v = __shfl_sync(0xffffffffu, v, 0);
        if (v >= items) break;
        const int b = (int)(v / per);
        const int c = (int)(v - (uint32_t)b * per);
        const DrawDesc d = load_desc(&P.draw[b]);
        if (d.n < 0) continue;  // a bad sequence (or one an aborted stream left undecided)
        pass_task<DT>(P, b, c, d, tab, ct, ring, lane);
        // the chunk totals and listed tokens of every lane, then the count
        __threadfence();
        __syncwarp();
        uint32_t last = 0;
        if (lane == 0) {
            last = atomicSub(&P.pass_left[b], 1u) == 1u ? 1u : 0u;
            if (last) __threadfence();  // the other passes' results, before they are read
        }
        if (__shfl_sync(0xffffffffu, last, 0)) finalize_task<DT>(P, b, d, tab, ct, ring, lane);
    }
}

cudaError_t launch_draw_tasks(const Params &p, int dtype, int num_sms, cudaStream_t s) {
    const int grid = 2 * num_sms;
    if (dtype == SV_DT_FP32)
        draw_task_kernel<SV_DT_FP32><<<grid, kDrawTaskWarps * 32, kDrawTaskSmem, s>>>(p);
    else
        draw_task_kernel<SV_DT_BF16><<<grid, kDrawTaskWarps * 32, kDrawTaskSmem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_draw(const Params &p, int dtype, int num_sms, cudaStream_t s) {
    const int64_t items = (int64_t)p.B * p.ntask;
    const int64_t want = (items + kDrawWarps - 1) / kDrawWarps;
    const int grid1 = (int)(want < (int64_t)num_sms * 8 ? want : (int64_t)num_sms * 8);
    const int grid2 = (p.B + kDrawWarps - 1) / kDrawWarps;
    if (dtype == SV_DT_FP32) {
        draw_pass_kernel<SV_DT_FP32><<<grid1, kDrawWarps * 32, kDrawSmem, s>>>(p);
        draw_finalize_kernel<SV_DT_FP32><<<grid2, kDrawWarps * 32, kDrawSmem, s>>>(p);
    } else {
        draw_pass_kernel<SV_DT_BF16><<<grid1, kDrawWarps * 32, kDrawSmem, s>>>(p);
        draw_finalize_kernel<SV_DT_BF16><<<grid2, kDrawWarps * 32, kDrawSmem, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t prepare_draw() {
    const void *fns[] = {(const void *)draw_pass_kernel<SV_DT_FP32>,
                         (const void *)draw_pass_kernel<SV_DT_BF16>,
                         (const void *)draw_finalize_kernel<SV_DT_FP32>,
                         (const void *)draw_finalize_kernel<SV_DT_BF16>};
    for (const void *f : fns) {
        const cudaError_t e =
            cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kDrawSmem);
        if (e != cudaSuccess) return e;
    }
    const void *tfns[] = {(const void *)draw_task_kernel<SV_DT_FP32>,
                          (const void *)draw_task_kernel<SV_DT_BF16>};
    for (const void *f : tfns) {
        const cudaError_t e =
            cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kDrawTaskSmem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace sv
