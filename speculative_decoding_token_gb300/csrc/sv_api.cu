// sv_api.cu -- the C ABI of the verify step (declared in include/specverify.h):
// handle and workspace ownership, host-side argument checks, kernel launches
// on the caller's stream, device status and optional kernel timing.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "sv_internal.h"
#include "sv_rows_params.h"
#include "sv_small.h"

namespace {

struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) {
            err = cudaSetDevice(dev);
            changed = err == cudaSuccess;
        }
    }
    ~DeviceGuard() {
        if (changed) cudaSetDevice(prev);
    }
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kNumKernels = 9;  // timing ids, see specverify_set_timing
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // about two seconds

struct TimedLaunch {
    cudaEvent_t start, stop;
    int kernel;
};

}  // namespace

struct specverify_ctx {
    int device = 0;
    int32_t max_batch = 0, max_gamma = 0;
    int64_t max_vocab = 0;
    int num_sms = 0;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    sv::Params base{};  // workspace pointers filled in at create time
    sv::RestrictParams rbase{};  // workspace of the restricted verify
    sv::FeatParams fbase{};      // workspace of the draft features (shares the pieces)
    int64_t max_rows = 0;        // rows of the largest batch: max_batch (2 max_gamma + 1)
    int timing = 0;
    std::vector<TimedLaunch> pending;
    std::vector<cudaEvent_t> pool;
    uint32_t epoch = 0;  // flag value of the last fused call
    uint64_t wait_ns = kDefaultWaitNs;  // bound of a fused-kernel wait on another warp
    double total_ms[kNumKernels] = {};
    int64_t launches[kNumKernels] = {};
};

namespace {

int map_cuda(cudaError_t e) {
    if (e == cudaSuccess) return SPECVERIFY_OK;
    if (e == cudaErrorMemoryAllocation) return SPECVERIFY_ERR_OOM;
    return SPECVERIFY_ERR_CUDA;
}

cudaEvent_t take_event(specverify_ctx *h) {
    if (!h->pool.empty()) {
        cudaEvent_t e = h->pool.back();
        h->pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Runs `launch` on stream s, bracketed by timing events when enabled.
template <class F>
cudaError_t timed(specverify_ctx *h, int kernel, cudaStream_t s, F &&launch) {
    if (!h->timing) return launch();
    cudaEvent_t a = take_event(h), b = take_event(h);
    if (!a || !b) return launch();
    cudaEventRecord(a, s);
    const cudaError_t e = launch();
    cudaEventRecord(b, s);
    h->pending.push_back({a, b, kernel});
    return e;
}

int check_batch(const specverify_ctx *h, const specverify_batch *in, bool sampling) {
    if (!h || !in) return SPECVERIFY_ERR_INVALID_ARG;
    if (in->B < 0 || in->B > h->max_batch) return SPECVERIFY_ERR_INVALID_ARG;
    if (in->gamma_max < 0 || in->gamma_max > h->max_gamma) return SPECVERIFY_ERR_INVALID_ARG;
    if (in->V < 1 || in->V > h->max_vocab) return SPECVERIFY_ERR_INVALID_ARG;
    if (in->dtype != SPECVERIFY_FP32 && in->dtype != SPECVERIFY_BF16)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (in->B == 0) return SPECVERIFY_OK;
    const int64_t esz = in->dtype == SPECVERIFY_FP32 ? 4 : 2;
    if (in->row_stride < in->V || (in->row_stride * esz) % 16 != 0)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (!in->target_logits || (reinterpret_cast<uintptr_t>(in->target_logits) & 15) != 0 ||
        in->target_rows < 1)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (!in->p_row_off || !in->gamma) return SPECVERIFY_ERR_INVALID_ARG;
    if (in->gamma_max > 0 && !in->draft_tokens) return SPECVERIFY_ERR_INVALID_ARG;
    if (sampling && in->gamma_max > 0) {
        if (!in->draft_logits || (reinterpret_cast<uintptr_t>(in->draft_logits) & 15) != 0 ||
            in->draft_rows < 1 || !in->q_row_off)
            return SPECVERIFY_ERR_INVALID_ARG;
    }
    return SPECVERIFY_OK;
}

int run_verify(specverify_ctx *h, const specverify_batch *in, bool sampling, float T,
               uint64_t seed, int32_t len_kind, float eps, int32_t *n_out, int32_t *tok_out,
               float *p_lse, float *q_lse, void *stream) {
    int rc = check_batch(h, in, sampling);
    if (rc != SPECVERIFY_OK) return rc;
    if (sampling && !(T > 0.0f && std::isfinite(T))) return SPECVERIFY_ERR_INVALID_ARG;
    if (len_kind < SPECVERIFY_LENIENCE_NONE || len_kind > SPECVERIFY_LENIENCE_EXP)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (len_kind != SPECVERIFY_LENIENCE_NONE && !(eps > 0.0f && eps <= 1.0f))
        return SPECVERIFY_ERR_INVALID_ARG;
    if (in->B == 0) return SPECVERIFY_OK;  // nothing to write: outputs may be NULL
    if (!n_out || !tok_out) return SPECVERIFY_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return SPECVERIFY_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    sv::Params P = h->base;
    const int64_t esz = in->dtype == SPECVERIFY_FP32 ? 4 : 2;
    P.target = static_cast<const char *>(in->target_logits);
    P.draft = static_cast<const char *>(sampling ? in->draft_logits : in->target_logits);
    if (!P.draft) P.draft = P.target;
    P.stride_bytes = in->row_stride * esz;
    P.V = in->V;
    P.row_bytes = in->V * esz;
    P.p_row_off = in->p_row_off;
    P.q_row_off = sampling ? in->q_row_off : in->p_row_off;
    P.tokens = in->draft_tokens;
    P.gamma = in->gamma;
    P.target_rows = in->target_rows;
    P.draft_rows = sampling ? in->draft_rows : 0;
    P.B = in->B;
    P.gamma_max = in->gamma_max;
    P.sampling = sampling ? 1 : 0;
    const double c2 = 1.4426950408889634073599 / (sampling ? (double)T : 1.0);  // log2(e)/T
    P.c2 = (float)c2;
    P.c2h = (float)c2;
    P.c2l = (float)(c2 - (double)P.c2h);
    P.lspan = (float)(1000.0 / c2);
    P.invT = sampling ? 1.0 / (double)T : 1.0;
    P.invTh = (float)P.invT;
    P.invTl = (float)(P.invT - (double)P.invTh);
    P.seed = seed;
    P.len_kind = len_kind;
    P.len_c = len_kind == SPECVERIFY_LENIENCE_LIN  ? -std::log((double)eps)
              : len_kind == SPECVERIFY_LENIENCE_SQ ? -2.0 * std::log((double)eps)
              : len_kind == SPECVERIFY_LENIENCE_EXP ? (double)eps
                                                    : 0.0;
    P.len_cf = (float)P.len_c;
    P.n_out = n_out;
    P.tok_out = tok_out;
    P.p_lse = sampling ? p_lse : nullptr;
    P.q_lse = sampling ? q_lse : nullptr;
    P.cpr = (int32_t)((P.row_bytes + sv::kItemBytes - 1) / sv::kItemBytes);
    P.nch3 = (int32_t)((in->V + sv::kDrawChunk - 1) / sv::kDrawChunk);
    // chunks per pass task: kTaskChunks when the batch gives every warp of
    // the GPU several tasks, down to one for small batches
    {
        const int64_t warps = (int64_t)h->num_sms * sv::kFusedWarps;
        const int64_t chunks = (int64_t)in->B * P.nch3;
        int64_t tc = chunks / (2 * warps);
        tc = tc < 1 ? 1 : (tc > sv::kTaskChunks ? sv::kTaskChunks : tc);
        P.task_chunks = (int32_t)tc;
    }
    P.ntask = (P.nch3 + P.task_chunks - 1) / P.task_chunks;
    if (!sampling || in->dtype != SPECVERIFY_BF16) P.code_tab = nullptr;

    if (sampling) {
        // one persistent kernel: plan, stream, accept tests and draw
        if (++h->epoch == 0) {
            // the flags hold epochs of earlier calls: after 2^32 calls clear
            // them, so that no stale flag can match the restarted epoch
            h->epoch = 1;
            const int64_t G = (int64_t)h->max_gamma + 1;
            const int64_t nch = (h->max_vocab + sv::kDrawChunk - 1) / sv::kDrawChunk;
            cudaError_t e = cudaMemsetAsync(P.rq_slot, 0,
                                            sizeof(unsigned long long) * h->max_batch * G, s);
            if (e == cudaSuccess)
                e = cudaMemsetAsync(P.dq_slot, 0,
                                    sizeof(unsigned long long) * h->max_batch * nch, s);
            if (e == cudaSuccess) e = cudaMemsetAsync(P.abort_flag, 0, sizeof(uint32_t), s);
            if (e == cudaSuccess)
                e = cudaMemsetAsync(P.grid_bar, 0, sizeof(unsigned long long) * 2 * sv::kCtrStride, s);
            if (e != cudaSuccess) return map_cuda(e);
        }
        P.epoch = h->epoch;
        P.G = in->gamma_max + 1;
        // no logsumexp output requested: stream only the rows the result needs
        P.skip = (p_lse == nullptr && q_lse == nullptr) ? 1 : 0;
        P.wait_ns = h->wait_ns;
        // a small batch: one cluster per sequence, no grid-wide machinery
        if (in->B <= sv::kSmallMaxB && in->gamma_max <= sv::kSmallMaxGamma &&
            sv::small_smem_bytes(P) <= sv::kSmallSmem) {
            const cudaError_t e = timed(h, 8, s, [&] { return sv::launch_small(P, in->dtype, s); });
            return map_cuda(e);
        }
        // one launch: the kernel's prologue validates and plans the call
        const cudaError_t e =
            timed(h, 4, s, [&] { return sv::launch_fused(P, in->dtype, h->num_sms, s); });
        return map_cuda(e);
    }
    // a small greedy batch: one cluster per sequence, one launch
    if (in->B <= sv::kSmallMaxB && in->gamma_max <= sv::kSmallMaxGamma) {
        const cudaError_t e =
            timed(h, 8, s, [&] { return sv::launch_small_greedy(P, in->dtype, s); });
        return map_cuda(e);
    }
    cudaError_t e = timed(h, 0, s, [&] { return sv::launch_plan(P, s); });
    if (e != cudaSuccess) return map_cuda(e);
    e = timed(h, 1, s, [&] { return sv::launch_rowstats(P, in->dtype, h->num_sms, s); });
    if (e != cudaSuccess) return map_cuda(e);
    e = timed(h, 3, s, [&] { return sv::launch_accept(P, in->dtype, s); });
    return map_cuda(e);
}

}  // namespace

extern "C" {

int specverify_create(specverify_t *out, int device, int32_t max_batch, int32_t max_gamma,
                      int64_t max_vocab) {
    if (!out) return SPECVERIFY_ERR_INVALID_ARG;
    *out = nullptr;
    if (max_batch < 1 || max_gamma < 0 || max_gamma > sv::kMaxGamma || max_vocab < 1 ||
        max_vocab > sv::kMaxVocab)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (device < 0) return SPECVERIFY_ERR_INVALID_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) return SPECVERIFY_ERR_CUDA;
    DeviceGuard guard(device);
    if (guard.err != cudaSuccess) return SPECVERIFY_ERR_CUDA;

    specverify_ctx *h = new (std::nothrow) specverify_ctx();
    if (!h) return SPECVERIFY_ERR_OOM;
    h->device = device;
    h->max_batch = max_batch;
    h->max_gamma = max_gamma;
    h->max_vocab = max_vocab;
    cudaError_t e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = sv::prepare_rowstats();
    if (e == cudaSuccess) e = sv::prepare_fused();
    if (e == cudaSuccess) e = sv::prepare_draw();
    if (e == cudaSuccess) e = sv::prepare_features();
    if (e == cudaSuccess) e = sv::prepare_restricted();
    if (e == cudaSuccess) e = sv::prepare_small();
    if (e != cudaSuccess) {
        delete h;
        return map_cuda(e);
    }

    const int64_t rows = (int64_t)max_batch * (2 * (int64_t)max_gamma + 1);
    const int64_t cpr = (max_vocab * 4 + sv::kItemBytes - 1) / sv::kItemBytes;
    const int64_t nch3 = (max_vocab + sv::kDrawChunk - 1) / sv::kDrawChunk;
    struct Piece {
        void **dst;
        size_t bytes;
    };
    sv::Params &P = h->base;
    const int64_t G = (int64_t)max_gamma + 1;
    void *p_rows = nullptr, *p_seq_base = nullptr, *p_seq_rows = nullptr, *p_total = nullptr,
         *p_part = nullptr, *p_stat = nullptr, *p_draw = nullptr, *p_draw_chunk = nullptr,
         *p_draw_mass = nullptr, *p_zone = nullptr, *p_zone_cnt = nullptr, *p_tab = nullptr,
         *p_status = nullptr, *p_code_tab = nullptr, *p_order = nullptr, *p_pos_cnt = nullptr,
         *p_pos_res = nullptr, *p_first_rej = nullptr, *p_decided = nullptr,
         *p_pass_left = nullptr, *p_dq_slot = nullptr, *p_rq_slot = nullptr,
         *p_ctr = nullptr, *p_abort = nullptr,
         *p_seq_state = nullptr, *p_grid_bar = nullptr, *p_seq_info = nullptr,
         *p_rr_rows = nullptr, *p_rr_total = nullptr, *p_rr_parts = nullptr,
         *p_rr_seq = nullptr, *p_rr_flag = nullptr, *p_rr_fin = nullptr,
         *p_feat_stat = nullptr;
    // restricted verify: every range of the row pass's stage split holds at
    // most cap row pieces
    const int64_t rr_ranges =
        (int64_t)h->num_sms * sv::kRestrictWarps * sv::kRestrictRangesPerWarp;
    const int64_t rr_cap = (rows + rr_ranges - 1) / rr_ranges + 2;
    Piece pieces[] = {
        {&p_rows, sizeof(sv::RowRef) * rows},
        {&p_seq_base, sizeof(int32_t) * max_batch},
        {&p_seq_rows, sizeof(int32_t) * max_batch},
        {&p_total, sizeof(int32_t)},
        {&p_part, sizeof(float2) * rows * cpr},
        {&p_stat, sizeof(float2) * rows},
        {&p_draw, sizeof(sv::DrawDesc) * max_batch},
        {&p_draw_chunk, sizeof(sv::ChunkTot) * max_batch * nch3},
        {&p_draw_mass, sizeof(double) * max_batch * nch3},
        {&p_zone, sizeof(sv::ZoneEntry) * max_batch * sv::kZoneMax},
        {&p_zone_cnt, sizeof(uint32_t) * max_batch},
        {&p_tab, sizeof(float2) * sv::kExpTab},
        {&p_status, sizeof(int32_t)},
        {&p_code_tab, sizeof(float2) * sv::kCodeTab},
        {&p_order, sizeof(sv::OrderRef) * max_batch * 2 * G},
        {&p_pos_cnt, sizeof(uint32_t) * max_batch * G},
        {&p_pos_res, sizeof(uint32_t) * max_batch * G},
        {&p_first_rej, sizeof(int32_t) * max_batch},
        {&p_decided, sizeof(uint32_t) * max_batch},
        {&p_pass_left, sizeof(uint32_t) * max_batch},
        {&p_dq_slot, sizeof(unsigned long long) * max_batch * nch3},
        {&p_rq_slot, sizeof(unsigned long long) * max_batch * G},
        {&p_ctr, sizeof(uint32_t) * sv::kNumCtr * sv::kCtrStride},
        {&p_abort, sizeof(uint32_t)},
        {&p_seq_state, sizeof(unsigned long long) * max_batch},
        {&p_grid_bar, sizeof(unsigned long long) * 2 * sv::kCtrStride},
        {&p_seq_info, sizeof(int32_t) * max_batch},
        {&p_rr_rows, sizeof(sv::RRow) * rows},
        {&p_rr_total, sizeof(int32_t)},
        {&p_rr_parts, sizeof(sv::RTop) * rr_ranges * rr_cap * sv::kMaxRestrictK},
        {&p_rr_seq, sizeof(int2) * max_batch},
        {&p_rr_flag, sizeof(uint32_t) * max_batch},
        {&p_rr_fin, sizeof(uint32_t) * rows},
        {&p_feat_stat, sizeof(float4) * rr_ranges * rr_cap},
    };
    size_t total = 0;
    for (const Piece &pc : pieces) total = align_up(total, 256) + pc.bytes;
    e = cudaMalloc(&h->ws, total);
    if (e != cudaSuccess) {
        delete h;
        return map_cuda(e);
    }
    h->ws_bytes = total;
    size_t off = 0;
    for (const Piece &pc : pieces) {
        off = align_up(off, 256);
        *pc.dst = static_cast<char *>(h->ws) + off;
        off += pc.bytes;
    }
    P.rows = static_cast<sv::RowRef *>(p_rows);
    P.seq_base = static_cast<int32_t *>(p_seq_base);
    P.seq_rows = static_cast<int32_t *>(p_seq_rows);
    P.total_rows = static_cast<int32_t *>(p_total);
    P.partials = static_cast<float2 *>(p_part);
    P.row_stat = static_cast<float2 *>(p_stat);
    P.draw = static_cast<sv::DrawDesc *>(p_draw);
    P.draw_chunk = static_cast<sv::ChunkTot *>(p_draw_chunk);
    P.draw_mass = static_cast<double *>(p_draw_mass);
    P.code_tab = static_cast<float2 *>(p_code_tab);  // per call: null unless bf16 sampling
    P.order = static_cast<sv::OrderRef *>(p_order);
    P.pos_cnt = static_cast<uint32_t *>(p_pos_cnt);
    P.pos_res = static_cast<uint32_t *>(p_pos_res);
    P.first_rej = static_cast<int32_t *>(p_first_rej);
    P.decided = static_cast<uint32_t *>(p_decided);
    P.pass_left = static_cast<uint32_t *>(p_pass_left);
    P.dq_slot = static_cast<unsigned long long *>(p_dq_slot);
    P.rq_slot = static_cast<unsigned long long *>(p_rq_slot);
    P.ctr = static_cast<uint32_t *>(p_ctr);
    P.abort_flag = static_cast<uint32_t *>(p_abort);
    P.seq_state = static_cast<unsigned long long *>(p_seq_state);
    P.grid_bar = static_cast<unsigned long long *>(p_grid_bar);
    P.seq_info = static_cast<int32_t *>(p_seq_info);
    P.zone = static_cast<sv::ZoneEntry *>(p_zone);
    P.zone_cnt = static_cast<uint32_t *>(p_zone_cnt);
    P.exp2_tab = static_cast<const float2 *>(p_tab);
    P.status = static_cast<int32_t *>(p_status);
    sv::RestrictParams &RP = h->rbase;
    RP.rows = static_cast<sv::RRow *>(p_rr_rows);
    RP.total_rows = static_cast<int32_t *>(p_rr_total);
    RP.parts = static_cast<sv::RTop *>(p_rr_parts);
    RP.cap = (int32_t)rr_cap;
    RP.seq_rows = static_cast<int2 *>(p_rr_seq);
    RP.row_grid = h->num_sms;
    h->fbase.parts = RP.parts;
    h->fbase.pstat = static_cast<float4 *>(p_feat_stat);
    h->fbase.cap = RP.cap;
    h->fbase.row_grid = h->num_sms;
    h->max_rows = rows;
    RP.seq_flag = static_cast<uint32_t *>(p_rr_flag);
    RP.row_fin = static_cast<uint32_t *>(p_rr_fin);
    RP.status = P.status;
    RP.exp2_tab = P.exp2_tab;

    std::vector<float2> tab(sv::kExpTab);
    sv::fill_exp2_table(tab.data());
    e = cudaMemcpy(p_tab, tab.data(), sizeof(float2) * sv::kExpTab, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(p_status, 0, sizeof(int32_t));
    // the fused kernel's flags hold the epoch of the call that set them
    if (e == cudaSuccess) e = cudaMemset(p_rq_slot, 0, sizeof(unsigned long long) * max_batch * G);
    if (e == cudaSuccess)
        e = cudaMemset(p_dq_slot, 0, sizeof(unsigned long long) * max_batch * nch3);
    if (e == cudaSuccess) e = cudaMemset(p_abort, 0, sizeof(uint32_t));
    if (e == cudaSuccess)
        e = cudaMemset(p_grid_bar, 0, sizeof(unsigned long long) * 2 * sv::kCtrStride);
    // the restricted verify's flags start (and are left) at zero
    if (e == cudaSuccess) e = cudaMemset(p_rr_flag, 0, sizeof(uint32_t) * max_batch);
    if (e == cudaSuccess) e = cudaMemset(p_rr_fin, 0, sizeof(uint32_t) * rows);
    if (e != cudaSuccess) {
        cudaFree(h->ws);
        delete h;
        return map_cuda(e);
    }
    *out = h;
    return SPECVERIFY_OK;
}

int specverify_destroy(specverify_t h) {
    if (!h) return SPECVERIFY_OK;
    {
        DeviceGuard guard(h->device);
        for (auto &t : h->pending) {
            cudaEventDestroy(t.start);
            cudaEventDestroy(t.stop);
        }
        for (auto ev : h->pool) cudaEventDestroy(ev);
        if (h->ws) cudaFree(h->ws);
    }
    delete h;
    return SPECVERIFY_OK;
}

int specverify_verify(specverify_t h, const specverify_batch *in, float temperature,
                      uint64_t seed, int32_t *n_accepted, int32_t *out_tokens, float *p_lse,
                      float *q_lse, void *cuda_stream) {
    return run_verify(h, in, true, temperature, seed, SPECVERIFY_LENIENCE_NONE, 1.0f, n_accepted,
                      out_tokens, p_lse, q_lse, cuda_stream);
}

int specverify_verify_lossy(specverify_t h, const specverify_batch *in, float temperature,
                            uint64_t seed, int32_t lenience, float eps, int32_t *n_accepted,
                            int32_t *out_tokens, float *p_lse, float *q_lse, void *cuda_stream) {
    return run_verify(h, in, true, temperature, seed, lenience, eps, n_accepted, out_tokens, p_lse,
                      q_lse, cuda_stream);
}

int specverify_verify_greedy(specverify_t h, const specverify_batch *in, int32_t *n_accepted,
                             int32_t *out_tokens, void *cuda_stream) {
    return run_verify(h, in, false, 0.0f, 0, SPECVERIFY_LENIENCE_NONE, 1.0f, n_accepted,
                      out_tokens, nullptr, nullptr, cuda_stream);
}

int specverify_verify_restricted(specverify_t h, const specverify_batch *in,
                                 const float *temperature, const int32_t *top_k,
                                 const float *top_p, uint64_t seed, int32_t *n_accepted,
                                 int32_t *out_tokens, void *cuda_stream) {
    int rc = check_batch(h, in, true);
    if (rc != SPECVERIFY_OK) return rc;
    if (in->B == 0) return SPECVERIFY_OK;
    if (!temperature || !top_k || !n_accepted || !out_tokens) return SPECVERIFY_ERR_INVALID_ARG;
    const int64_t esz0 = in->dtype == SPECVERIFY_FP32 ? 4 : 2;
    const int64_t max_rows = (int64_t)in->B * (2 * (int64_t)in->gamma_max + 1);
    const int64_t stages = max_rows * ((in->V * esz0 + 4095) / 4096);
    if (max_rows > INT32_MAX || stages > INT32_MAX) return SPECVERIFY_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return SPECVERIFY_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const int64_t esz = in->dtype == SPECVERIFY_FP32 ? 4 : 2;
    sv::RestrictParams R = h->rbase;
    R.target = static_cast<const char *>(in->target_logits);
    R.draft = static_cast<const char *>(in->draft_logits);
    R.stride_bytes = in->row_stride * esz;
    R.V = in->V;
    R.row_bytes = in->V * esz;
    R.target_rows = in->target_rows;
    R.draft_rows = in->draft_rows;
    R.B = in->B;
    R.gamma_max = in->gamma_max;
    R.p_row_off = in->p_row_off;
    R.q_row_off = in->q_row_off;
    R.tokens = in->draft_tokens;
    R.gamma = in->gamma;
    R.temperature = temperature;
    R.top_k = top_k;
    R.top_p = top_p;
    R.seed = seed;
    R.n_out = n_accepted;
    R.tok_out = out_tokens;
    cudaError_t e = timed(h, 5, s, [&] { return sv::launch_restrict_plan(R, s); });
    if (e == cudaSuccess)
        e = timed(h, 6, s, [&] { return sv::launch_restrict_rows(R, in->dtype, s); });
    if (e == cudaSuccess) e = timed(h, 7, s, [&] { return sv::launch_restrict_final(R, s); });
    return map_cuda(e);
}

int specverify_acceptance_stats(specverify_t h, const specverify_batch *in, float temperature,
                                float *beta, float *tvd, void *cuda_stream) {
    int rc = check_batch(h, in, true);
    if (rc != SPECVERIFY_OK) return rc;
    if (!(temperature > 0.0f && std::isfinite(temperature))) return SPECVERIFY_ERR_INVALID_ARG;
    if (in->B == 0 || in->gamma_max == 0) return SPECVERIFY_OK;
    if (!beta || !tvd) return SPECVERIFY_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return SPECVERIFY_ERR_CUDA;
    const int64_t esz = in->dtype == SPECVERIFY_FP32 ? 4 : 2;
    sv::FeatParams F{};
    F.rows = static_cast<const char *>(in->target_logits);
    F.rows2 = static_cast<const char *>(in->draft_logits);
    F.stride_bytes = in->row_stride * esz;
    F.V = in->V;
    F.row_bytes = in->V * esz;
    F.nrows = in->B;
    F.p_row_off = in->p_row_off;
    F.q_row_off = in->q_row_off;
    F.gamma = in->gamma;
    F.target_rows = in->target_rows;
    F.draft_rows = in->draft_rows;
    F.gamma_max = in->gamma_max;
    F.c2 = (float)(1.4426950408889634073599 / (double)temperature);
    F.beta = beta;
    F.tvd = tvd;
    F.status = h->base.status;
    return map_cuda(sv::launch_pairs(F, in->dtype, h->num_sms, static_cast<cudaStream_t>(cuda_stream)));
}

int specverify_row_features(specverify_t h, const void *rows, int32_t dtype, int64_t nrows,
                            int64_t V, int64_t row_stride, float temperature, int32_t k,
                            float *entropy, float *topk_prob, int32_t *topk_idx,
                            void *cuda_stream) {
    if (!h || nrows < 0 || V < 1 || V > INT32_MAX || k < 0 || k > sv::kMaxTopK)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (dtype != SPECVERIFY_FP32 && dtype != SPECVERIFY_BF16) return SPECVERIFY_ERR_INVALID_ARG;
    if (!(temperature > 0.0f && std::isfinite(temperature))) return SPECVERIFY_ERR_INVALID_ARG;
    if (nrows == 0) return SPECVERIFY_OK;
    const int64_t esz = dtype == SPECVERIFY_FP32 ? 4 : 2;
    if (!rows || (reinterpret_cast<uintptr_t>(rows) & 15) != 0 || row_stride < V ||
        (row_stride * esz) % 16 != 0 || !entropy || (k > 0 && (!topk_prob || !topk_idx)))
        return SPECVERIFY_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return SPECVERIFY_ERR_CUDA;
    // the row pass splits at most max_rows rows at a time (its pieces fit the workspace)
    sv::FeatParams F = h->fbase;
    F.stride_bytes = row_stride * esz;
    F.V = V;
    F.row_bytes = V * esz;
    F.k = k;
    F.c2 = (float)(1.4426950408889634073599 / (double)temperature);
    {
        // the most negative bf16 logit s with s * c2 finite and far below any
        // real logit: -7.5e37 / c2, at least -3.3e38, rounded toward zero
        const double sv = std::max(-3.3e38, -7.5e37 / (double)F.c2);
        const float sf = (float)sv;
        uint32_t bits;
        std::memcpy(&bits, &sf, 4);
        const uint32_t b16 = bits >> 16;  // truncation: toward zero, so finite
        F.ninf_sub = b16 | (b16 << 16);
    }
    F.status = h->base.status;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    for (int64_t r0 = 0; r0 < nrows; r0 += h->max_rows) {
        F.rows = static_cast<const char *>(rows) + r0 * F.stride_bytes;
        F.nrows = std::min(h->max_rows, nrows - r0);
        F.entropy = entropy + r0;
        F.topk_prob = k > 0 ? topk_prob + r0 * k : nullptr;
        F.topk_idx = k > 0 ? topk_idx + r0 * k : nullptr;
        const cudaError_t e = sv::launch_features(F, dtype, s);
        if (e != cudaSuccess) return map_cuda(e);
    }
    return SPECVERIFY_OK;
}

int specverify_device_status(specverify_t h, void *cuda_stream, int32_t *status_out) {
    if (!h || !status_out) return SPECVERIFY_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return SPECVERIFY_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, h->base.status, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->base.status, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return map_cuda(e);
    *status_out = v;
    return SPECVERIFY_OK;
}

const char *specverify_status_string(int status) {
    switch (status) {
        case SPECVERIFY_OK: return "ok";
        case SPECVERIFY_ERR_INVALID_ARG: return "invalid argument";
        case SPECVERIFY_ERR_CUDA: return "CUDA runtime error";
        case SPECVERIFY_ERR_OOM: return "out of device memory";
        case SPECVERIFY_ERR_DEVICE_INPUT: return "bad input detected on the device";
        case SPECVERIFY_ERR_TIMEOUT: return "a bounded device wait gave up";
        case SPECVERIFY_ERR_TOO_LARGE:
            return "batch larger than the fixed scratch of the no-allocation entry point";
        default: return "unknown status";
    }
}

int specverify_workspace_bytes(specverify_t h, size_t *out) {
    if (!h || !out) return SPECVERIFY_ERR_INVALID_ARG;
    *out = h->ws_bytes;
    return SPECVERIFY_OK;
}

int specverify_set_timing(specverify_t h, int enable) {
    if (!h) return SPECVERIFY_ERR_INVALID_ARG;
    h->timing = enable ? 1 : 0;
    return SPECVERIFY_OK;
}

int specverify_set_wait_limit(specverify_t h, uint64_t ns) {
    if (!h) return SPECVERIFY_ERR_INVALID_ARG;
    h->wait_ns = ns == 0 ? kDefaultWaitNs : ns;
    return SPECVERIFY_OK;
}

int specverify_get_timing(specverify_t h, int kernel, double *total_ms, int64_t *launches,
                          int reset) {
    if (!h || kernel < 0 || kernel >= kNumKernels) return SPECVERIFY_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return SPECVERIFY_ERR_CUDA;
    for (auto &t : h->pending) {
        if (cudaEventSynchronize(t.stop) != cudaSuccess) return SPECVERIFY_ERR_CUDA;
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, t.start, t.stop) != cudaSuccess) return SPECVERIFY_ERR_CUDA;
        h->total_ms[t.kernel] += ms;
        h->launches[t.kernel] += 1;
        h->pool.push_back(t.start);
        h->pool.push_back(t.stop);
    }
    h->pending.clear();
    if (total_ms) *total_ms = h->total_ms[kernel];
    if (launches) *launches = h->launches[kernel];
    if (reset) {
        for (int k = 0; k < kNumKernels; ++k) {
            h->total_ms[k] = 0.0;
            h->launches[k] = 0;
        }
    }
    return SPECVERIFY_OK;
}

}  // extern "C"
