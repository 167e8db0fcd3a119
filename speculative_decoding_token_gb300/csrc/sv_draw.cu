// sv_draw.cu -- the final-token draw of the verify step.
//
// "DistillSpec" Algorithm A.1 ("sample from the adjusted distribution"
// norm(max(0, p_{n+1} - q_{n+1})) after a rejection, otherwise sample the
// bonus token from p_{gamma+1}); "Speculative Decoding and Distillation"
// (Kadimisetty notes) Part 1 steps 4-5. The draw is the inverse CDF in token
// index order: k = min{k : C_k > u * R}.
//
// Exactness of the decision needs the CDF to roughly 40 bits, far beyond
// fp32 sums of fp32 exponentials, so every weight is a float-float
// e = 2^((l - M) log2(e)/T) (relative error near 2^-43) and every sum is
// compensated. With rho = S_p / S_q the residual weight of token v is
// proportional to max(0, e_p(v) - rho e_q(v)). One pass per (chunk, sequence)
// CTA accumulates S_p, S_q and, over the tokens whose sign is certain under
// the row-statistics estimate of rho (window 2^-15), P_A = sum e_p and
// Q_A = sum e_q of the positive ones; the few tokens inside the window are
// listed. The CTA that finishes a sequence's last chunk then knows rho
// exactly, forms the chunk masses P_A - rho Q_A (+ the listed tokens, exact),
// locates t = u * R among the chunk prefix sums and rescans that one chunk
// token by token. A list overflow or an estimate outside the window makes it
// recompute every chunk mass with the exact rho (slow path, flagged).
#include "sv_common.cuh"

namespace sv {

// L1-bypassing loads of records written by other CTAs of the same launch
__device__ __forceinline__ Quad ldcg_quad(const Quad *p) {
    const double2 a = __ldcg(reinterpret_cast<const double2 *>(p));
    const double2 b = __ldcg(reinterpret_cast<const double2 *>(p) + 1);
    return Quad{a.x, a.y, b.x, b.y};
}

__device__ __forceinline__ ZoneEntry ldcg_zone(const ZoneEntry *p) {
    ZoneEntry z;
    const int4 a = __ldcg(reinterpret_cast<const int4 *>(p));
    const int4 b = __ldcg(reinterpret_cast<const int4 *>(p) + 1);
    *reinterpret_cast<int4 *>(&z) = a;
    *(reinterpret_cast<int4 *>(&z) + 1) = b;
    return z;
}

// exact-rho residual weight max(0, e_p - rho e_q) as a float-float
__device__ __forceinline__ void residual_weight(float eph, float epl, float eqh, float eql,
                                                float rh, float rl, float &wh, float &wl) {
    const float ph = rh * eqh;
    float pe = fmaf(rh, eqh, -ph);
    pe = fmaf(rh, eql, pe);
    pe = fmaf(rl, eqh, pe);
    float s, e;
    two_sum(eph, -ph, s, e);
    e += epl - pe;
    wh = s + e;
    wl = e - (wh - s);
    if (!(wh > 0.0f)) {
        wh = 0.0f;
        wl = 0.0f;
    }
}

template <int DT>
__device__ __forceinline__ void token_exp(const char *row, int64_t v, float M, const Params &P,
                                          const float2 *tab, float &eh, float &el) {
    float yh, yl;
    scaled_gap(load_logit<DT>(row, v), M, P.c2h, P.c2l, yh, yl);
    ff_exp2(yh, yl, tab, eh, el);
}

// weight of token v under the final (exact) rho; residual == 0: e_p
template <int DT>
__device__ __forceinline__ void token_weight(const char *prow, const char *qrow, int64_t v,
                                             const DrawDesc &d, int residual, float rh,
                                             float rl, const Params &P, const float2 *tab,
                                             float &wh, float &wl) {
    float eph, epl;
    token_exp<DT>(prow, v, d.Mp, P, tab, eph, epl);
    if (!residual) {
        wh = eph;
        wl = epl;
        return;
    }
    float eqh, eql;
    token_exp<DT>(qrow, v, d.Mq, P, tab, eqh, eql);
    residual_weight(eph, epl, eqh, eql, rh, rl, wh, wl);
}

// block-wide float-float reduction of NV pairs; the double results land in out[] for all threads
template <int NV>
__device__ void block_sum_ff(float (&h)[NV], float (&l)[NV], double *red /* [8][NV] */,
                             double *out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        float hh = h[k], ll = l[k];
        // renormalise the per-thread accumulator first
        float s = hh + ll;
        ll = ll - (s - hh);
        hh = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oh = __shfl_xor_sync(0xffffffffu, hh, off);
            const float ol = __shfl_xor_sync(0xffffffffu, ll, off);
            ff_add(hh, ll, oh, ol, hh, ll);
        }
        if (lane == 0) red[warp * NV + k] = ff_to_double(hh, ll);
    }
    __syncthreads();
    if (threadIdx.x < NV) {
        double acc = 0.0;
        for (int w = 0; w < kDrawThreads / 32; ++w) acc += red[w * NV + threadIdx.x];
        out[threadIdx.x] = acc;
    }
    __syncthreads();
}

template <int DT>
__device__ void finalize_draw(const Params &P, int b, const DrawDesc &d, const float2 *tab,
                              double rho_est) {
    __shared__ double mass[kMaxChunks3];
    __shared__ double red[kDrawThreads / 32 * 4];
    __shared__ double tot[4];
    __shared__ double scan[kDrawThreads];
    __shared__ ZoneEntry zsorted[kZoneMax];
    __shared__ double sh_rho, sh_tloc;
    __shared__ int sh_slow, sh_res, sh_cstar, sh_takelast, sh_k, sh_lastpos;
    const int tid = threadIdx.x;
    const int nch = P.nch3;
    const Quad *part = P.draw_part + (int64_t)b * P.nch3;
    const char *prow = P.target + d.p_phys * P.stride_bytes;
    const char *qrow = d.residual ? P.draft + d.q_phys * P.stride_bytes : nullptr;

    if (tid == 0) {
        double sp = 0.0, sq = 0.0;
        for (int c = 0; c < nch; ++c) {
            const Quad pc = ldcg_quad(&part[c]);
            sp += pc.x;
            sq += pc.y;
        }
        const double rho = d.residual ? sp / sq : 1.0;
        const uint32_t zc = __ldcg(&P.zone_cnt[b]);
        sh_rho = rho;
        sh_slow = d.residual && (zc > (uint32_t)kZoneMax ||
                                 !(fabs(rho / rho_est - 1.0) <= 0.5 * kRhoWindow));
        sh_res = d.residual;
        sh_k = -1;
        sh_lastpos = -1;
    }
    __syncthreads();
    const double rho = sh_rho;
    const float rh = (float)rho;
    const float rl = (float)(rho - (double)rh);

    if (sh_slow) {
        // exact chunk masses with the final rho
        for (int c = 0; c < nch; ++c) {
            float h[1] = {0.0f}, l[1] = {0.0f};
            const int64_t v0 = (int64_t)c * kDrawChunk, v1 = min(P.V, v0 + kDrawChunk);
            for (int64_t v = v0 + tid; v < v1; v += kDrawThreads) {
                float wh, wl;
                token_weight<DT>(prow, qrow, v, d, 1, rh, rl, P, tab, wh, wl);
                ff_accumulate(h[0], l[0], wh, wl);
            }
            block_sum_ff<1>(h, l, red, tot);
            if (tid == 0) mass[c] = tot[0];
        }
        if (tid == 0) atomicOr(P.status, SPECVERIFY_STATUS_DRAW_SLOW);
    } else if (d.residual) {
        const int zc = min((int)__ldcg(&P.zone_cnt[b]), kZoneMax);
        for (int i = tid; i < zc; i += kDrawThreads)
            zsorted[i] = ldcg_zone(&P.zone[(int64_t)b * kZoneMax + i]);
        for (int c = tid; c < nch; c += kDrawThreads) {
            const Quad pc = ldcg_quad(&part[c]);
            mass[c] = pc.z - rho * pc.w;
        }
        __syncthreads();
        if (tid == 0) {
            // insertion sort by token index: a fixed summation order
            for (int i = 1; i < zc; ++i) {
                const ZoneEntry z = zsorted[i];
                int j = i - 1;
                while (j >= 0 && zsorted[j].v > z.v) {
                    zsorted[j + 1] = zsorted[j];
                    --j;
                }
                zsorted[j + 1] = z;
            }
            for (int i = 0; i < zc; ++i) {
                const ZoneEntry z = zsorted[i];
                const double w = ff_to_double(z.eph, z.epl) - rho * ff_to_double(z.eqh, z.eql);
                if (w > 0.0) mass[z.v / kDrawChunk] += w;
            }
        }
    } else {
        for (int c = tid; c < nch; c += kDrawThreads) mass[c] = ldcg_quad(&part[c]).x;
    }
    __syncthreads();

    if (tid == 0) {
        double R = 0.0;
        for (int c = 0; c < nch; ++c) R += mass[c];
        if (!(R > 0.0) || !isfinite(R)) {
            // zero residual mass through rounding: draw from p_{n+1}
            R = 0.0;
            for (int c = 0; c < nch; ++c) {
                mass[c] = ldcg_quad(&part[c]).x;
                R += mass[c];
            }
            sh_res = 0;
            atomicOr(P.status, SPECVERIFY_STATUS_DRAW_ZERO_MASS);
        }
        const double u = draw_uniform(P.seed, (uint32_t)b, (uint32_t)(d.n + 1));
        const double t = u * R;
        double C = 0.0;
        int cstar = -1;
        for (int c = 0; c < nch; ++c) {
            const double Cn = C + mass[c];
            if (Cn > t) {
                cstar = c;
                break;
            }
            C = Cn;
        }
        int takelast = 0;
        if (cstar < 0) {
            takelast = 1;
            for (int c = nch - 1; c >= 0; --c)
                if (mass[c] > 0.0) {
                    cstar = c;
                    break;
                }
            if (cstar < 0) cstar = 0;
        }
        sh_cstar = cstar;
        sh_takelast = takelast;
        sh_tloc = t - C;
    }
    __syncthreads();

    // rescan chunk c*: thread tid owns kDrawPerThread consecutive tokens
    const int residual = sh_res;
    const int64_t c0 = (int64_t)sh_cstar * kDrawChunk;
    const int64_t cend = min(P.V, c0 + kDrawChunk);
    const int64_t r0 = c0 + (int64_t)tid * kDrawPerThread;
    const int64_t r1 = min(cend, r0 + kDrawPerThread);
    float sh = 0.0f, sl = 0.0f;
    int lastpos = -1;
    for (int64_t v = r0; v < r1; ++v) {
        float wh, wl;
        token_weight<DT>(prow, qrow, v, d, residual, rh, rl, P, tab, wh, wl);
        if (wh > 0.0f) lastpos = (int)v;
        ff_accumulate(sh, sl, wh, wl);
    }
    if (lastpos >= 0) atomicMax(&sh_lastpos, lastpos);
    scan[tid] = ff_to_double(sh, sl);
    __syncthreads();
    if (tid == 0) {
        double run = 0.0;
        for (int i = 0; i < kDrawThreads; ++i) {
            const double x = scan[i];
            scan[i] = run;  // exclusive prefix
            run += x;
        }
    }
    __syncthreads();
    if (!sh_takelast) {
        const double start = scan[tid];
        const double tl = sh_tloc;
        const double mine = ff_to_double(sh, sl);
        if (start <= tl && tl < start + mine) {
            double C = start;
            for (int64_t v = r0; v < r1; ++v) {
                float wh, wl;
                token_weight<DT>(prow, qrow, v, d, residual, rh, rl, P, tab, wh, wl);
                C += ff_to_double(wh, wl);
                if (C > tl) {
                    sh_k = (int)v;
                    break;
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        const int k = sh_k >= 0 ? sh_k : sh_lastpos;
        P.tok_out[(int64_t)b * (P.gamma_max + 1) + d.n] = k;
    }
}

template <int DT>
__global__ void __launch_bounds__(kDrawThreads) draw_kernel(Params P) {
    __shared__ float2 tab[256];
    __shared__ double red[kDrawThreads / 32 * 4];
    __shared__ double tot[4];
    __shared__ int last_s;
    const int tid = threadIdx.x;
    const int b = (int)(blockIdx.x / (uint32_t)P.nch3);
    const int c = (int)(blockIdx.x % (uint32_t)P.nch3);
    const DrawDesc d = P.draw[b];
    if (d.n < 0) return;
    for (int i = tid; i < 256; i += kDrawThreads) tab[i] = P.exp2_tab[i];
    __syncthreads();

    const char *prow = P.target + d.p_phys * P.stride_bytes;
    const char *qrow = d.residual ? P.draft + d.q_phys * P.stride_bytes : nullptr;
    const double rho_est = d.residual ? (double)d.Sp / (double)d.Sq : 1.0;
    const float rhi = (float)(rho_est * (1.0 + kRhoWindow));
    const float rlo = (float)(rho_est * (1.0 - kRhoWindow));
    const int64_t v0 = (int64_t)c * kDrawChunk;
    const int64_t v1 = min(P.V, v0 + kDrawChunk);

    // S_p, S_q, P_A, Q_A as float-float accumulators
    float h[4] = {0.0f, 0.0f, 0.0f, 0.0f}, l[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (d.residual) {
        for (int64_t v = v0 + tid; v < v1; v += kDrawThreads) {
            float eph, epl, eqh, eql;
            token_exp<DT>(prow, v, d.Mp, P, tab, eph, epl);
            token_exp<DT>(qrow, v, d.Mq, P, tab, eqh, eql);
            ff_accumulate(h[0], l[0], eph, epl);
            ff_accumulate(h[1], l[1], eqh, eql);
            if (eph > rhi * eqh) {
                ff_accumulate(h[2], l[2], eph, epl);
                ff_accumulate(h[3], l[3], eqh, eql);
            } else if (eqh > 0.0f && eph >= rlo * eqh) {
                const uint32_t slot = atomicAdd(&P.zone_cnt[b], 1u);
                if (slot < (uint32_t)kZoneMax) {
                    ZoneEntry z;
                    z.v = (int32_t)v;
                    z.eph = eph;
                    z.epl = epl;
                    z.eqh = eqh;
                    z.eql = eql;
                    z.pad[0] = z.pad[1] = z.pad[2] = 0;
                    P.zone[(int64_t)b * kZoneMax + slot] = z;
                }
            }
        }
    } else {
        for (int64_t v = v0 + tid; v < v1; v += kDrawThreads) {
            float eph, epl;
            token_exp<DT>(prow, v, d.Mp, P, tab, eph, epl);
            ff_accumulate(h[0], l[0], eph, epl);
        }
    }
    __threadfence();  // zone entries before this CTA's completion is counted
    block_sum_ff<4>(h, l, red, tot);
    if (tid == 0) {
        P.draw_part[(int64_t)b * P.nch3 + c] = Quad{tot[0], tot[1], tot[2], tot[3]};
        __threadfence();
        last_s = (atomicAdd(&P.draw_cnt[b], 1u) + 1u == (uint32_t)P.nch3);
    }
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    finalize_draw<DT>(P, b, d, tab, rho_est);
}

cudaError_t launch_draw(const Params &p, int dtype, cudaStream_t s) {
    const dim3 grid((uint32_t)p.nch3 * (uint32_t)p.B), block(kDrawThreads);
    if (dtype == SV_DT_FP32)
        draw_kernel<SV_DT_FP32><<<grid, block, 0, s>>>(p);
    else
        draw_kernel<SV_DT_BF16><<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t prepare_draw() { return cudaSuccess; }

}  // namespace sv
