// sv_fused.cu -- the sampling verify step as one persistent kernel.
//
// One cooperative CTA per SM. Its first kFusedStreamWarps warps stream every
// logical row once (sv_stream.cuh: per-warp rings of bulk copies, fence-free
// chunk partials). The other warps -- and every streaming warp once its
// stream is done -- run the per-sequence tasks of the verify step from one
// global counter, in order:
//   accept(b):      wait until all chunk partials of b's rows are stored,
//                   combine them and run the accept scan ("DistillSpec"
//                   Algorithm A.1); publish the draw descriptor of b;
//   pass(b, c):     wait for b's descriptor, run the draw pass over chunk c
//                   (sv_draw.cuh); publish that chunk;
//   finalize(b):    wait for b's chunks and draw the final token.
// So the ALU-heavy draw of early sequences runs while later rows stream.
//
// Progress: a task only waits on tasks taken earlier from the counter (whose
// warps are running, as the launch is cooperative) or on streamed partials
// (whose warps never wait on anything), so every wait ends; each one is still
// bounded by about two seconds of wall time, after which it sets
// SPECVERIFY_STATUS_TIMEOUT and gives up its task.
#include "sv_draw.cuh"

namespace sv {

constexpr uint64_t kWaitNs = 2000000000ull;

// lane 0 polls an epoch flag with acquire loads; the warp then proceeds
__device__ __forceinline__ bool wait_flag(const uint32_t *f, uint32_t epoch, int lane) {
    uint32_t ok = 1;
    if (lane == 0 && ld_acquire_u32(f) != epoch) {
        const uint64_t t0 = global_ns();
        while (ld_acquire_u32(f) != epoch) {
            __nanosleep(200);
            if (global_ns() - t0 > kWaitNs) {
                ok = 0;
                break;
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// every lane polls its share of the chunk partials [begin, begin + count)
__device__ bool wait_partials(const Params &P, int64_t begin, int64_t count, int lane) {
    uint32_t ok = 1;
    const uint64_t t0 = global_ns();
    for (int64_t i = lane; i < count && ok; i += 32) {
        while (ld_relaxed_f2(&P.partials[begin + i]).y == kPartialPending) {
            __nanosleep(200);
            if (global_ns() - t0 > kWaitNs) {
                ok = 0;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok) != 0;
}

__device__ __forceinline__ DrawDesc load_desc(const DrawDesc *p) {
    DrawDesc d;
    d.n = __ldcg(&p->n);
    d.residual = __ldcg(&p->residual);
    d.p_phys = (int64_t)__ldcg(reinterpret_cast<const long long *>(&p->p_phys));
    d.q_phys = (int64_t)__ldcg(reinterpret_cast<const long long *>(&p->q_phys));
    d.Mp = __ldcg(&p->Mp);
    d.Sp = __ldcg(&p->Sp);
    d.Mq = __ldcg(&p->Mq);
    d.Sq = __ldcg(&p->Sq);
    return d;
}

__device__ __forceinline__ void publish(uint32_t *flag, uint32_t epoch, int lane) {
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        st_release_u32(flag, epoch);
    }
}

template <int DT>
__device__ void accept_task(const Params &P, int b, int lane) {
    const int rows = P.seq_rows[b];
    if (rows > 0) {
        const int base = P.seq_base[b];
        if (wait_partials(P, (int64_t)base * P.cpr, (int64_t)rows * P.cpr, lane)) {
            __threadfence();  // the polled partials are re-read below
            for (int r = 0; r < rows; ++r) combine_row<0>(P, base + r, lane);
            __syncwarp();
            accept_scan_sampling<DT>(P, b, lane);
        } else if (lane == 0) {
            atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
        }
    }
    publish(&P.seq_flag[b], P.epoch, lane);
}

template <int DT>
__device__ void run_tasks(const Params &P, const float2 *tab, const float2 *ct, int lane) {
    const int64_t per = (int64_t)P.nch3 + 2;
    const int64_t total = (int64_t)P.B * per;
    for (;;) {
        unsigned long long t = 0;
        if (lane == 0) t = atomicAdd(P.task_ctr, 1ull);
        t = __shfl_sync(0xffffffffu, t, 0);
        if ((int64_t)t >= total) return;
        const int b = (int)((int64_t)t / per);
        const int r = (int)((int64_t)t - (int64_t)b * per);
        if (r == 0) {
            accept_task<DT>(P, b, lane);
        } else if (r <= P.nch3) {
            const int c = r - 1;
            if (wait_flag(&P.seq_flag[b], P.epoch, lane)) {
                const DrawDesc d = load_desc(&P.draw[b]);
                if (d.n >= 0) pass_task<DT>(P, b, c, d, tab, ct, lane);
            } else if (lane == 0) {
                atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
            }
            publish(&P.pass_flag[(int64_t)b * P.nch3 + c], P.epoch, lane);
        } else {
            if (!wait_flag(&P.seq_flag[b], P.epoch, lane)) {
                if (lane == 0) atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
                continue;
            }
            const DrawDesc d = load_desc(&P.draw[b]);
            if (d.n < 0) continue;
            uint32_t ok = 1;
            const uint64_t t0 = global_ns();
            for (int c = lane; c < P.nch3; c += 32) {
                const uint32_t *f = &P.pass_flag[(int64_t)b * P.nch3 + c];
                while (ok && ld_acquire_u32(f) != P.epoch) {
                    __nanosleep(200);
                    if (global_ns() - t0 > kWaitNs) ok = 0;
                }
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) atomicOr(P.status, SPECVERIFY_STATUS_TIMEOUT);
                continue;
            }
            finalize_task<DT>(P, b, d, tab, lane);
        }
    }
}

template <int DT>
__global__ void __launch_bounds__(kFusedWarps * 32, 1) fused_kernel(Params P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kFusedStreamWarps][kStages];
    float2 *tab = reinterpret_cast<float2 *>(smem + kFusedRingBytes);
    float2 *ct = tab + kExpTab;
    for (int i = threadIdx.x; i < kExpTab; i += blockDim.x) tab[i] = P.exp2_tab[i];
    if (P.code_tab)
        for (int i = threadIdx.x; i < kCodeTab; i += blockDim.x) ct[i] = __ldcg(&P.code_tab[i]);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (warp < kFusedStreamWarps && lane == 0) {
        const uint32_t bar0 = smem_u32(&bars[warp][0]);
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp < kFusedStreamWarps)
        stream_items<DT, 0>(P, smem + warp * (kStages * kStageBytes), smem_u32(&bars[warp][0]),
                            (int64_t)blockIdx.x * kFusedStreamWarps + warp,
                            (int64_t)gridDim.x * kFusedStreamWarps, lane);
    run_tasks<DT>(P, tab, P.code_tab ? ct : nullptr, lane);
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
