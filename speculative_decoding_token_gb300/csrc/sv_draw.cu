// sv_draw.cu -- the final-token draw as two standalone kernels.
//
// The pass kernel runs every pass task (sequence b, span of chunks t) and the
// finalize kernel one finalize task per sequence, after the accept kernel on
// the same stream (sv_draw.cuh holds the tasks). The allocation-free entry
// point uses these; the regular sampling entry point runs the same tasks
// inside the fused kernel.
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
__global__ void __launch_bounds__(kDrawWarps * 32) draw_pass_kernel(const __grid_constant__ Params P) {
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
__global__ void __launch_bounds__(kDrawWarps * 32) draw_finalize_kernel(const __grid_constant__ Params P) {
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
    return cudaSuccess;
}

}  // namespace sv
