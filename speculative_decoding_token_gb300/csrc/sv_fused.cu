// sv_fused.cu -- the sampling verify step as one persistent kernel.
//
// One cooperative CTA per SM. Its first kFusedStreamWarps warps stream every
// logical row once (sv_stream.cuh: per-warp rings of bulk copies, fence-free
// chunk partials); the warp that stores the last chunk partial of a
// sequence runs that sequence's accept step ("DistillSpec" Algorithm A.1:
// combine the rows, accept scan, draw descriptor) and publishes it. The
// other warps -- and every streaming warp once its stream is done -- take
// the draw tasks from one global counter, sequence by sequence:
//   pass(b, c):   wait for b's accept, run the draw pass over chunk c
//                 (sv_draw.cuh); publish that chunk;
//   finalize(b):  wait for b's chunks and draw the final token.
// So the ALU-heavy draw of early sequences runs while later rows stream.
//
// Progress: a task waits only on tasks taken earlier from the counter (whose
// warps are running, as the launch is cooperative) or on an accept step run
// by a streaming warp (which waits only on partials of other streaming
// warps), so every wait ends; each one is still bounded by about two seconds
// of wall time, after which it sets SPECVERIFY_STATUS_TIMEOUT and marks the
// call aborted, and every other wait of the call returns at once.
#include "sv_draw.cuh"

namespace sv {

__device__ __forceinline__ DrawDesc load_desc(const DrawDesc *p) {
    static_assert(sizeof(DrawDesc) % 16 == 0, "DrawDesc is loaded as 16-byte words");
    DrawDesc d;
    const int4 *src = reinterpret_cast<const int4 *>(p);
    int4 *dst = reinterpret_cast<int4 *>(&d);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(DrawDesc) / 16); ++i) dst[i] = __ldcg(src + i);
    return d;
}

// Draw tasks in counter order: for each sequence b, the pass tasks of its
// chunks, then its finalize task.
template <int DT>
__device__ void run_tasks(const Params &P, const float2 *tab, const float2 *ct, int lane) {
    const int64_t per = (int64_t)P.nch3 + 1;
    const int64_t total = (int64_t)P.B * per;
    for (;;) {
        while (try_accept<DT>(P, lane)) {
        }
        unsigned long long t = 0;
        if (lane == 0) t = atomicAdd(P.task_ctr, 1ull);
        t = __shfl_sync(0xffffffffu, t, 0);
        if ((int64_t)t >= total) {
            // the accept steps not claimed yet (each run once, in order)
            while ((int64_t)*reinterpret_cast<const volatile uint32_t *>(P.acc_next) < P.B) {
                if (!try_accept<DT>(P, lane)) {
                    __nanosleep(200);
                    if (call_aborted(P)) break;
                }
            }
            return;
        }
        const int b = (int)((int64_t)t / per);
        const int r = (int)((int64_t)t - (int64_t)b * per);
        if (!wait_flag_helping<DT>(P, &P.seq_flag[b], lane)) continue;
        const DrawDesc d = load_desc(&P.draw[b]);
        if (r < P.nch3) {
            if (d.n >= 0) pass_task<DT>(P, b, r, d, tab, ct, lane);
            publish(&P.pass_flag[(int64_t)b * P.nch3 + r], P.epoch, lane);
        } else if (d.n >= 0) {
            bool ok = true;
            for (int c = 0; c < P.nch3 && ok; ++c)
                ok = wait_flag_helping<DT>(P, &P.pass_flag[(int64_t)b * P.nch3 + c], lane);
            if (!ok) continue;
            finalize_task<DT>(P, b, d, tab, ct, lane);
        }
    }
}

template <int DT>
__global__ void __launch_bounds__(kFusedWarps * 32, 1) fused_kernel(Params P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kFusedStreamWarps][kFusedStages];
    // One 32 KiB table lives in shared memory: the bf16 weight table when
    // the call has one (the exponential table is then read from global
    // memory on its rare path), else the exponential table.
    float2 *stab = reinterpret_cast<float2 *>(smem + kFusedRingBytes);
    const float2 *src = P.code_tab ? P.code_tab : P.exp2_tab;
    for (int i = threadIdx.x; i < kSmemTab; i += blockDim.x) stab[i] = __ldcg(&src[i]);
    const float2 *tab = P.code_tab ? P.exp2_tab : stab;
    const float2 *ct = P.code_tab ? stab : nullptr;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (warp < kFusedStreamWarps && lane == 0) {
        const uint32_t bar0 = smem_u32(&bars[warp][0]);
        for (int s = 0; s < kFusedStages; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp < kFusedStreamWarps)
        stream_items<DT, 0, kFusedStages, kFusedStageBytes, true>(
            P, smem + warp * (kFusedStages * kFusedStageBytes), smem_u32(&bars[warp][0]),
            (int64_t)blockIdx.x * kFusedStreamWarps + warp, (int64_t)gridDim.x * kFusedStreamWarps,
            lane);
    run_tasks<DT>(P, tab, ct, lane);
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
