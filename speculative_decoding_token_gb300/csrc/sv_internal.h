// sv_internal.h -- types and tile constants shared by the host library and
// the kernels of the verify step (not part of the public C ABI).
#pragma once

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "specverify.h"

#define SV_DT_FP32 0
#define SV_DT_BF16 1

namespace sv {

// Row-statistics kernel tiling: every row is cut into chunks of kItemBytes
// (the unit one warp reduces to a partial), each streamed through that
// warp's private ring of kStages shared-memory buffers of kStageBytes by 1-D
// bulk asynchronous copies. One persistent CTA of kWarps warps per SM.
constexpr int kItemBytes = 32768;
constexpr int kStageBytes = 4096;
constexpr int kStages = 3;
constexpr int kWarps = 16;
constexpr int kRowStatsSmem = kWarps * kStages * kStageBytes;  // 192 KiB

// Accept kernel: one CTA per sequence.
constexpr int kAcceptThreads = 256;

// Draw: the draw rows are cut into chunks of kDrawChunk tokens, each with
// its own totals (the finalize rescans one chunk, so smaller chunks shorten
// it; 1024 measured faster than 2048 or 4096). A pass walks its chunks in
// blocks of 256 tokens of which lane L owns tokens 8L .. 8L + 7 (coalesced
// 16-byte loads). The standalone draw kernels run CTAs of kDrawWarps warps
// sharing the tables in shared memory.
constexpr int kDrawChunk = 1024;
constexpr int kDrawBlock = 256;
// A pass task covers up to kTaskChunks consecutive draw chunks (its fixed
// costs -- claim, descriptor, epilogue -- amortise over 4096 tokens), still
// recording one total per chunk. Small batches use fewer chunks a task, so
// that a sequence's draw rows spread over more warps (one warp's pass is
// latency-bound: ~20 us for 4096 tokens on an otherwise idle SM).
constexpr int kTaskChunks = 4;
constexpr int kDrawWarps = 8;
// Each warp that runs draw tasks owns a ring of kPassRingBytes of shared
// memory through which its blocks arrive ahead of use (8 blocks of bf16
// rows, 4 of fp32).
constexpr int kPassRingBytes = 8192;
constexpr int kZoneMax = 256;         // ambiguous-sign residual entries kept per sequence
// 2^(j/4096), j = 0..4095, as float-float pairs
constexpr int kExpTab = 4096;
constexpr int kMaxChunks3 = 2048;     // draw chunks per row: V <= 2 Mi tokens
constexpr int64_t kMaxVocab = (int64_t)kDrawChunk * kMaxChunks3;
constexpr int kMaxGamma = 256;

// bf16 weight table: the float-float weight 2^(l log2(e)/T) of every bf16
// logit l with 2^-6 <= |l| < 2^10 (16 binades of 128 mantissas per sign),
// built once per call. Index: magnitude bits - kCodeBase, + kCodeHalf if l < 0.
constexpr uint32_t kCodeBase = 121u << 7;  // bf16 bits of 2^-6
constexpr int kCodeHalf = 2048;
constexpr int kCodeTab = 2 * kCodeHalf;

// Fused sampling kernel: one cooperative CTA per SM; kFusedStreamWarps warps
// stream the rows (each with its ring of kFusedStages stages of
// kFusedStageBytes), one warp tests positions, the rest (if any) start on
// the draw tasks at once, and every warp takes draw tasks once its stream is
// done. Dynamic shared memory: the stream rings (a streaming warp's draw ring
// is the start of its stream ring, free once its stream is done), the draw
// rings of the task warps, then one 32 KiB table (the bf16 weight table, or
// the exponential table when the call has no weight table; the exponential
// table is then read from global memory on its rare path). 16 warps leave
// 128 registers a thread. The split was measured on the ragged B = 256,
// V = 152064 bf16 batch (and the B = 64, V = 128256 one): every warp but the
// tester streaming, with two 4 KiB stages each (199.5 us), beat 12 to 14
// streaming warps with two stages (200-202 us), 10 with three (204-206 us)
// and every split with fewer streaming warps or deeper rings (up to 229 us).
// The stream's per-warp control path is latency-bound, so it wants many
// warps; fewer bytes in flight keep the memory queues, and with them every
// round trip of the tests and the draw, short.
constexpr int kFusedStreamWarps = 15;
constexpr int kFusedStages = 2;
constexpr int kFusedStageBytes = 4096;
constexpr int kFusedWarps = 16;
constexpr int kTesterWarp = kFusedStreamWarps;  // serves position tests only
constexpr int kFusedTaskWarps = kFusedWarps - kFusedStreamWarps - 1;
constexpr int kFusedRingBytes = kFusedStreamWarps * kFusedStages * kFusedStageBytes;
constexpr int kFusedDrawRingOff = kFusedRingBytes;
constexpr int kFusedTabOff = kFusedDrawRingOff + kFusedTaskWarps * kPassRingBytes;
constexpr int kSmemTab = kExpTab > kCodeTab ? kExpTab : kCodeTab;  // float2 entries
constexpr int kFusedSmem = kFusedTabOff + kSmemTab * 8;
static_assert(kItemBytes % kFusedStageBytes == 0, "stages tile a chunk");
static_assert(kFusedStages * kFusedStageBytes >= kPassRingBytes, "a stream ring holds a draw ring");
static_assert(kFusedSmem <= 227 * 1024 - 2048, "dynamic shared memory of one CTA");
static_assert(kExpTab == kCodeTab, "either table fills the shared table region");
// the standalone draw kernels: both tables, then one draw ring per warp, in
// dynamic shared memory
constexpr int kDrawRingOff = kExpTab * 8 + kCodeTab * 8;
constexpr int kDrawSmem = kDrawRingOff + kDrawWarps * kPassRingBytes;
// .y of a chunk partial whose chunk has not been streamed yet (a stored
// partial's .y is a sum of exponentials: >= 0 or NaN)
constexpr float kPartialPending = -1.0f;

// Half-width of the window around the row-statistics estimate of
// rho = S_p / S_q inside which a token's residual sign is decided only once
// the exact rho is known (2^-15).
constexpr double kRhoWindow = 1.0 / 32768.0;

// Logical row of the batch: sequence b, and j >= 0 for target row p_{j+1}
// or j < 0 for draft row q_{-j}; phys is the row index in its logit buffer.
struct RowRef {
    int64_t phys;
    int32_t b;
    int32_t j;
};

// What the accept scan hands to the draw kernel for sequence b.
struct __align__(16) DrawDesc {
    int32_t n;          // accepted count, -1 for a bad sequence
    int32_t residual;   // 1: draw from norm(max(0, p_{n+1} - q_{n+1})); 0: bonus from p
    int64_t p_phys;     // target row p_{n+1}
    int64_t q_phys;     // draft row q_{n+1} (residual only)
    float Mp, Sp;       // raw-logit max and sum of exp((l - Mp)/T) of the p row
    float Mq, Sq;       // the same for the q row
    float ip, iq;       // integer exponent shifts of the p and q rows (0 unless shift)
    int32_t shift;      // 1: a row lies far from 0 in the 2^(l log2(e)/T) scale
    int32_t pad;
    float rho_est;      // row-statistics estimate of S_p / S_q in the shifted scale
    int32_t pad2;
};

// Four doubles: per-chunk S_p, S_q, P_A, Q_A of a draw, as the finalize
// uses them.
struct __align__(16) Quad {
    double x, y, z, w;
};

// The same totals as a pass stores them: float-float pairs (head, tail), so
// that the pass itself needs no FP64 instruction (FP64 runs at a small
// fraction of the FP32 rate). s = (S_p, S_q), a = (P_A, Q_A); a bonus pass
// stores S_p only.
struct __align__(16) ChunkTot {
    float4 s, a;
};

// A token whose residual sign the draw kernel could not decide with the
// estimated rho: its exact exponentials, as float-float pairs.
struct __align__(16) ZoneEntry {
    int32_t v;
    float eph, epl, eqh, eql;
    int32_t pad[3];
};

// A row in the fused kernel's stream order.
struct __align__(16) OrderRef {
    int64_t phys;   // row index in its logit buffer
    int32_t b;      // sequence
    int32_t j;      // >= 0: target row p_{j+1}; < 0: draft row q_{-j}
    int32_t lrow;   // sequence-major logical row (partials, row statistics)
    int32_t pos;    // position of the row: j + 1, or -j
    int32_t need;   // chunk partials that complete the position (cpr x its rows)
    int32_t pad;
};

// counters of the fused kernel, each on its own 128-byte line (index k at
// ctr[k * kCtrStride]): the position-test queue, the pass-task queue, the
// sequences completed, the stream tickets
constexpr int kCtrRqHead = 0, kCtrRqTail = 1, kCtrDqHead = 2, kCtrDqTail = 3, kCtrDone = 4,
              kCtrTicket = 5;
constexpr int kNumCtr = 6;
// Items per stream ticket of the fused kernel: ticket c covers the items
// (c / NW) kStreamWin NW + (c mod NW) + j NW, j < kStreamWin, of the
// position-major order (NW: the kernel's streaming warps). With tickets
// dealt round robin, warp gw takes tickets gw, gw + NW, ..., so it streams
// items gw, gw + NW, ... whatever kStreamWin is; kStreamWin sets how many it
// holds at once (2 measured as fast as 4 and faster than 8).
constexpr int kStreamWin = 2;
// Up to this many items a streaming warp, tickets are dealt round robin;
// beyond it they are claimed from a shared counter.
constexpr int kDealtItemsPerWarp = 48;
constexpr int kCtrStride = 32;

struct Params {
    // inputs (device)
    const char *target;
    const char *draft;
    int64_t stride_bytes;
    int64_t V;
    int64_t row_bytes;        // V * element size
    const int64_t *p_row_off;
    const int64_t *q_row_off;
    const int32_t *tokens;
    const int32_t *gamma;
    int64_t target_rows, draft_rows;
    int32_t B, gamma_max;
    int32_t sampling;
    float c2;                 // log2(e) / T, rounded to float
    float c2h, c2l;           // log2(e) / T as a float-float
    float lspan;              // 1000 / (log2(e) / T): logits below max - lspan weigh 0
    double invT;
    float invTh, invTl;       // 1 / T as a float-float
    uint64_t seed;
    // outputs (device)
    int32_t *n_out;
    int32_t *tok_out;
    float *p_lse;
    float *q_lse;
    // workspace (device)
    RowRef *rows;
    int32_t *seq_base;
    int32_t *seq_rows;
    int32_t *total_rows;
    float2 *partials;         // [rows, cpr]
    float2 *row_stat;         // [rows]: (max, sum) or (max value, argmax bits)
    DrawDesc *draw;
    ChunkTot *draw_chunk;     // [B, nch3]: S_p, S_q, P_A, Q_A of each draw chunk
    double *draw_mass;        // [B, nch3]: chunk masses of the final draw
    ZoneEntry *zone;          // [B, kZoneMax]
    uint32_t *zone_cnt;
    const float2 *exp2_tab;   // kExpTab entries 2^(j/kExpTab) as float-float
    float2 *code_tab;         // kCodeTab bf16 weights (bf16 sampling only, else null)
    int32_t *status;
    int32_t cpr;              // chunks per row in the row-statistics kernel
    int32_t nch3;             // chunks per row in the draw kernel
    int32_t task_chunks;      // draw chunks per pass task (1 .. kTaskChunks)
    int32_t ntask;            // pass tasks per row: ceil(nch3 / task_chunks)
    // fused kernel only
    int32_t skip;             // 1: stream only rows the verify needs (no logsumexp outputs)
    int32_t G;                // positions per sequence: gamma_max + 1
    uint32_t epoch;           // this call's flag value (never 0; flags start at 0)
    OrderRef *order;          // [total_rows]: the dense position-major stream order
    uint32_t *pos_cnt;        // [B, G]: chunk partials of position k's rows stored so far
    uint32_t *pos_res;        // [B, G]: 0 untested, 1 accepted / bonus row ready, 2 rejected, 3 bad
    int32_t *first_rej;       // [B]: lowest rejected position known so far (G + 1: none)
    uint32_t *decided;        // [B]: 1 once sequence b is decided (or bad)
    unsigned long long *seq_state;  // [B] (G <= 32): bit k-1 position k accepted, bit 31+k
                                    // rejected, both bad
    uint32_t *pass_left;      // [B]: pass tasks of sequence b not yet finished; the warp
                              // that finishes the last one runs b's finalize
    unsigned long long *dq_slot;  // [B * ntask]: pass tasks (b * ntask + t) once published
    // queue slots: (epoch << 32) | item once published
    unsigned long long *rq_slot;  // [B * G]: positions ready for their test (b * G + k - 1)
    uint32_t *ctr;            // kCtrRqHead .. kCtrDone
    uint32_t *abort_flag;     // == epoch once a wait of this call gave up
    unsigned long long *grid_bar;  // two grid-barrier counters, kCtrStride words apart
    int32_t *seq_info;        // [B]: gamma of a valid sequence, -1 for bad input
    uint64_t wait_ns;         // bound of a wait on another warp (nanoseconds)
    int32_t len_kind;         // SPECVERIFY_LENIENCE_*: the accept test's f(p, eps)
    double len_c;             // -log eps (lin), -2 log eps (sq), eps (exp)
    float len_cf;             // len_c rounded to float
};

// Kernel launchers (sv_rowstats.cu, sv_draw.cu, sv_fused.cu)
cudaError_t launch_plan(const Params &p, cudaStream_t s);
cudaError_t launch_rowstats(const Params &p, int dtype, int num_ctas, cudaStream_t s);
cudaError_t launch_accept(const Params &p, int dtype, cudaStream_t s);
cudaError_t launch_draw(const Params &p, int dtype, int num_sms, cudaStream_t s);
cudaError_t launch_fused(const Params &p, int dtype, int num_ctas, cudaStream_t s);
cudaError_t prepare_rowstats();
cudaError_t prepare_draw();
cudaError_t prepare_fused();

// Host: fill the exponential table, 2^(j/kExpTab) from the host's double exp2,
// split into a float head and a float tail.
inline void fill_exp2_table(float2 *tab) {
    for (int j = 0; j < kExpTab; ++j) {
        const double v = std::exp2((double)j / (double)kExpTab);
        const float hi = (float)v;
        tab[j] = make_float2(hi, (float)(v - (double)hi));
    }
}

}  // namespace sv
