// sv_noalloc.cu -- specverify_verify_noalloc: the sampling verify step for
// callers that may not allocate device memory.
//
// Some callers cannot call cudaMalloc: a serving process whose memory pool
// has already reserved all free device memory for its KV cache and forbids
// other allocators, or code on a latency-critical path where an allocation's
// implicit device-wide synchronisation would stall other streams. They
// cannot create a handle (the handle's workspace is allocated), so this entry
// point runs the verify step -- plan, row statistics, accept scan and the two
// draw kernels as separate launches, the same tasks that specverify_verify
// runs in its fused kernel -- with their workspace carved out of one fixed
// file-scope device array. The array exists on every
// GPU that loads the library, from load until process exit, whether or not
// this entry point is used.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "sv_internal.h"

namespace {

// Limits of the fixed scratch (the caller still owns inputs and outputs).
constexpr int32_t kNaMaxBatch = 64;
constexpr int32_t kNaMaxGamma = 16;
constexpr int64_t kNaMaxVocab = 262144;

constexpr int64_t kNaRows = (int64_t)kNaMaxBatch * (2 * kNaMaxGamma + 1);
constexpr int64_t kNaCpr = (kNaMaxVocab * 4 + sv::kItemBytes - 1) / sv::kItemBytes;
constexpr int64_t kNaNch3 = (kNaMaxVocab + sv::kDrawChunk - 1) / sv::kDrawChunk;

constexpr size_t al256(size_t x) { return (x + 255) / 256 * 256; }

// Byte offsets of the workspace pieces inside the scratch array.
constexpr size_t kOffRows = 0;
constexpr size_t kOffSeqBase = al256(kOffRows + sizeof(sv::RowRef) * kNaRows);
constexpr size_t kOffSeqRows = al256(kOffSeqBase + sizeof(int32_t) * kNaMaxBatch);
constexpr size_t kOffTotal = al256(kOffSeqRows + sizeof(int32_t) * kNaMaxBatch);
constexpr size_t kOffPart = al256(kOffTotal + sizeof(int32_t));
constexpr size_t kOffStat = al256(kOffPart + sizeof(float2) * kNaRows * kNaCpr);
constexpr size_t kOffDraw = al256(kOffStat + sizeof(float2) * kNaRows);
constexpr size_t kOffDrawChunk = al256(kOffDraw + sizeof(sv::DrawDesc) * kNaMaxBatch);
constexpr size_t kOffDrawMass = al256(kOffDrawChunk + sizeof(sv::ChunkTot) * kNaMaxBatch * kNaNch3);
constexpr size_t kOffZone = al256(kOffDrawMass + sizeof(double) * kNaMaxBatch * kNaNch3);
constexpr size_t kOffZoneCnt = al256(kOffZone + sizeof(sv::ZoneEntry) * kNaMaxBatch * sv::kZoneMax);
constexpr size_t kOffTab = al256(kOffZoneCnt + sizeof(uint32_t) * kNaMaxBatch);
constexpr size_t kOffStatus = al256(kOffTab + sizeof(float2) * sv::kExpTab);
constexpr size_t kOffCodeTab = al256(kOffStatus + sizeof(int32_t));
constexpr size_t kScratchBytes = al256(kOffCodeTab + sizeof(float2) * sv::kCodeTab);
static_assert(kScratchBytes <= (size_t)4 << 20, "the fixed scratch must stay modest");

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    std::mutex mu;
    bool ready = false;    // set once the set-up below has succeeded
    char *base = nullptr;  // device address of the scratch array on this device
    int num_sms = 0;
};

DeviceSetup g_setup[kMaxDevices];

}  // namespace

// The fixed scratch. In host code this name is only a stand-in for the
// device symbol, never a usable address: host code must take the device
// address with cudaGetSymbolAddress (done once per device below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

// Once per device, with that device current: the scratch's device address,
// the SM count, the kernels' shared-memory attribute, the exp2 table and a
// cleared status word. The copies here are synchronous. Returns a status
// code; a failure leaves the device not set up, so a later call tries again
// (for example one made after a stream capture that made this one fail).
int setup_device(DeviceSetup &s) {
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return SPECVERIFY_ERR_CUDA;
    int dev = 0, num_sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = sv::prepare_rowstats();
    if (e == cudaSuccess) e = sv::prepare_draw();
    float2 tab[sv::kExpTab];  // host staging of the table, private to this call
    sv::fill_exp2_table(tab);
    char *base = static_cast<char *>(ptr);
    if (e == cudaSuccess) e = cudaMemcpy(base + kOffTab, tab, sizeof(tab), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(base + kOffStatus, 0, sizeof(int32_t));
    if (e != cudaSuccess) return SPECVERIFY_ERR_CUDA;
    s.base = base;
    s.num_sms = num_sms;
    s.ready = true;
    return SPECVERIFY_OK;
}

}  // namespace

extern "C" int specverify_verify_noalloc(const specverify_batch *in, float temperature,
                                         uint64_t seed, int32_t *n_accepted,
                                         int32_t *out_tokens, float *p_lse, float *q_lse,
                                         void *cuda_stream) {
    if (!in) return SPECVERIFY_ERR_INVALID_ARG;
    if (!(temperature > 0.0f && std::isfinite(temperature))) return SPECVERIFY_ERR_INVALID_ARG;
    if (in->B < 0 || in->gamma_max < 0 || in->V < 1) return SPECVERIFY_ERR_INVALID_ARG;
    if (in->B > kNaMaxBatch || in->gamma_max > kNaMaxGamma || in->V > kNaMaxVocab)
        return SPECVERIFY_ERR_TOO_LARGE;
    if (in->dtype != SPECVERIFY_FP32 && in->dtype != SPECVERIFY_BF16)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (in->B == 0) return SPECVERIFY_OK;
    const int64_t esz = in->dtype == SPECVERIFY_FP32 ? 4 : 2;
    if (in->row_stride < in->V || (in->row_stride * esz) % 16 != 0)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (!in->target_logits || (reinterpret_cast<uintptr_t>(in->target_logits) & 15) != 0 ||
        in->target_rows < 1 || !in->p_row_off || !in->gamma)
        return SPECVERIFY_ERR_INVALID_ARG;
    if (in->gamma_max > 0 &&
        (!in->draft_tokens || !in->draft_logits || !in->q_row_off || in->draft_rows < 1 ||
         (reinterpret_cast<uintptr_t>(in->draft_logits) & 15) != 0))
        return SPECVERIFY_ERR_INVALID_ARG;
    if (!n_accepted || !out_tokens) return SPECVERIFY_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return SPECVERIFY_ERR_CUDA;
    DeviceSetup &s = g_setup[dev];
    {
        std::lock_guard<std::mutex> lock(s.mu);
        if (!s.ready) {
            const int rc = setup_device(s);
            if (rc != SPECVERIFY_OK) return rc;
        }
    }

    char *w = s.base;
    sv::Params P{};
    P.target = static_cast<const char *>(in->target_logits);
    P.draft = in->draft_logits ? static_cast<const char *>(in->draft_logits) : P.target;
    P.stride_bytes = in->row_stride * esz;
    P.V = in->V;
    P.row_bytes = in->V * esz;
    P.p_row_off = in->p_row_off;
    P.q_row_off = in->q_row_off ? in->q_row_off : in->p_row_off;
    P.tokens = in->draft_tokens;
    P.gamma = in->gamma;
    P.target_rows = in->target_rows;
    P.draft_rows = in->draft_rows;
    P.B = in->B;
    P.gamma_max = in->gamma_max;
    P.sampling = 1;
    const double c2 = 1.4426950408889634073599 / (double)temperature;  // log2(e)/T
    P.c2 = (float)c2;
    P.c2h = (float)c2;
    P.c2l = (float)(c2 - (double)P.c2h);
    P.lspan = (float)(1000.0 / c2);
    P.invT = 1.0 / (double)temperature;
    P.invTh = (float)P.invT;
    P.invTl = (float)(P.invT - (double)P.invTh);
    P.seed = seed;
    P.wait_ns = 2000000000ull;
    P.len_kind = SPECVERIFY_LENIENCE_NONE;
    P.len_c = 0.0;
    P.len_cf = (float)P.len_c;
    P.n_out = n_accepted;
    P.tok_out = out_tokens;
    P.p_lse = p_lse;
    P.q_lse = q_lse;
    P.rows = reinterpret_cast<sv::RowRef *>(w + kOffRows);
    P.seq_base = reinterpret_cast<int32_t *>(w + kOffSeqBase);
    P.seq_rows = reinterpret_cast<int32_t *>(w + kOffSeqRows);
    P.total_rows = reinterpret_cast<int32_t *>(w + kOffTotal);
    P.partials = reinterpret_cast<float2 *>(w + kOffPart);
    P.row_stat = reinterpret_cast<float2 *>(w + kOffStat);
    P.draw = reinterpret_cast<sv::DrawDesc *>(w + kOffDraw);
    P.draw_chunk = reinterpret_cast<sv::ChunkTot *>(w + kOffDrawChunk);
    P.draw_mass = reinterpret_cast<double *>(w + kOffDrawMass);
    P.zone = reinterpret_cast<sv::ZoneEntry *>(w + kOffZone);
    P.zone_cnt = reinterpret_cast<uint32_t *>(w + kOffZoneCnt);
    P.exp2_tab = reinterpret_cast<const float2 *>(w + kOffTab);
    P.status = reinterpret_cast<int32_t *>(w + kOffStatus);
    P.code_tab = in->dtype == SPECVERIFY_BF16 ? reinterpret_cast<float2 *>(w + kOffCodeTab) : nullptr;
    P.cpr = (int32_t)((P.row_bytes + sv::kItemBytes - 1) / sv::kItemBytes);
    P.nch3 = (int32_t)((in->V + sv::kDrawChunk - 1) / sv::kDrawChunk);
    P.task_chunks = sv::kTaskChunks;
    P.ntask = (P.nch3 + sv::kTaskChunks - 1) / sv::kTaskChunks;

    // Every counter the kernels read is reset by the plan kernel of this call
    // (the draw completion counters, the ambiguous-sign list lengths);
    // every other piece is written before it is read within the call.
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e = sv::launch_plan(P, st);
    if (e == cudaSuccess) e = sv::launch_rowstats(P, in->dtype, s.num_sms, st);
    if (e == cudaSuccess) e = sv::launch_accept(P, in->dtype, st);
    if (e == cudaSuccess) e = sv::launch_draw(P, in->dtype, s.num_sms, st);
    return e == cudaSuccess ? SPECVERIFY_OK : SPECVERIFY_ERR_CUDA;
}
