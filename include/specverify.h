/*
 * specverify.h -- C ABI of the GB300 (sm_103a) speculative-sampling verify step.
 *
 * The operation (page title, then section / algorithm):
 *   "DistillSpec: Improving Speculative Decoding via Knowledge Distillation",
 *   Sec. 3 "Speculative sampling" and App. A.3, Algorithm A.1 "Speculative
 *   decoding step"; "How speculative decoding lets a small model draft and a
 *   large one check" (the quoted rule n = min({i-1 : r_i > p_i(x)/q_i(x)} U
 *   {gamma})); "Speculative Decoding and Distillation" (Kadimisetty notes),
 *   Part 1 steps 1-5 and "Greedy vs sampling"; "Dynamic Speculation Lookahead
 *   Accelerates Speculative Decoding of Large Language Models" Sec. 3 (a
 *   lookahead gamma chosen per iteration, hence a ragged gamma per sequence).
 *
 * For each sequence b with gamma_b draft tokens x_1..x_gamma_b, target logit
 * rows p_1..p_{gamma_b+1} and draft logit rows q_1..q_gamma_b:
 *   p_i = softmax(target_i / T), q_i = softmax(draft_i / T)  (one T for both);
 *   r_i = U24(Philox4x32-10(key = seed, counter = (b, i, 0, 0)).word0);
 *   n   = min({i-1 : r_i > p_i(x_i) / q_i(x_i)} U {gamma_b});
 *   if n < gamma_b the final token is drawn from norm(max(0, p_{n+1} - q_{n+1})),
 *   otherwise (the bonus token) from p_{gamma_b+1}; the draw is the inverse CDF
 *   in token-index order, k = min{k : C_k > u * R}, with
 *   u = U52(Philox4x32-10(seed, (b, n+1, 1, 0)).words 0-1);
 *   the emitted tokens are x_1..x_n followed by the final token.
 * U24(x) = (2*(x>>9)+1) * 2^-24 and U52(x0,x1) = (2*k+1) * 2^-53 with
 * k = (x0<<20) | (x1>>12); key = (seed & 0xffffffff, seed >> 32). Ties
 * r_i == ratio accept. Greedy mode keeps the longest prefix with
 * x_i == argmax p_i (lowest index on ties, compared on the raw logits) and
 * appends argmax p_{n+1}; it reads no draft logits.
 *
 * All calls are asynchronous on the caller's CUDA stream; no call inside
 * verify synchronises the host. PyTorch (or any caller) owns every input and
 * output buffer; the handle owns only its workspace.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct specverify_ctx *specverify_t;

typedef enum {
    SPECVERIFY_FP32 = 0, /* IEEE binary32 logits */
    SPECVERIFY_BF16 = 1  /* bfloat16 logits (top 16 bits of a binary32) */
} specverify_dtype;

/* Return codes. Host-checkable errors are returned synchronously and launch
 * nothing. */
enum {
    SPECVERIFY_OK = 0,
    SPECVERIFY_ERR_INVALID_ARG = -1, /* bad pointer, size, alignment, dtype or temperature */
    SPECVERIFY_ERR_CUDA = -2,        /* a CUDA runtime call failed */
    SPECVERIFY_ERR_OOM = -3,         /* workspace allocation failed */
    SPECVERIFY_ERR_DEVICE_INPUT = -4,/* reported by specverify_device_status only */
    SPECVERIFY_ERR_TIMEOUT = -5,     /* reported by specverify_device_status only */
    SPECVERIFY_ERR_TOO_LARGE = -6    /* batch exceeds the fixed scratch of specverify_verify_noalloc */
};

/* Lenience of the accept test ("DistillSpec" Sec. 4 "DistillSpec with lossy
 * SD"; App. A.3 Algorithm A.1, rejection threshold f(p_i(y), eps) / q_i(y)):
 * f_lin(p, eps) = p / eps, f_sq(p, eps) = p / eps^2, f_exp(p, eps) = p^eps,
 * eps in (0, 1]; NONE (and any f at eps = 1) is lossless speculative
 * sampling. The residual after a rejection stays norm(max(0, p - q)). */
enum {
    SPECVERIFY_LENIENCE_NONE = 0,
    SPECVERIFY_LENIENCE_LIN = 1,
    SPECVERIFY_LENIENCE_SQ = 2,
    SPECVERIFY_LENIENCE_EXP = 3
};

/* Bits of the sticky device status word (specverify_device_status). A
 * sequence whose input is bad gets n_accepted[b] = -1 and all its output
 * tokens -1; the other sequences are unaffected. No kernel ever traps. */
enum {
    SPECVERIFY_STATUS_BAD_GAMMA = 1 << 0,   /* gamma[b] outside [0, gamma_max] */
    SPECVERIFY_STATUS_BAD_ROW = 1 << 1,     /* a row offset outside the logit buffer */
    SPECVERIFY_STATUS_BAD_TOKEN = 1 << 2,   /* a draft token outside [0, V) */
    SPECVERIFY_STATUS_BAD_LOGIT = 1 << 3,   /* NaN or +inf logit, or a row of all -inf, in a
                                               row the call reads: without logsumexp outputs,
                                               specverify_verify does not read the rows after
                                               a sequence's first rejection, so bad logits
                                               there go unreported */
    SPECVERIFY_STATUS_TIMEOUT = 1 << 4,     /* a bounded wait in a kernel gave up */
    SPECVERIFY_STATUS_BAD_PARAM = 1 << 5,   /* specverify_verify_restricted: a temperature,
                                               top-k or top-p outside its range */
    SPECVERIFY_STATUS_DRAW_SLOW = 1 << 8,   /* informational: a draw took the exact slow path */
    SPECVERIFY_STATUS_DRAW_ZERO_MASS = 1 << 9 /* informational: a residual had zero mass after
                                                 rounding; the token was drawn from p_{n+1} */
};

/* One batch, all pointers DEVICE pointers owned by the caller.
 *   target p_{b,i} (i = 1..gamma[b]+1) is row p_row_off[b] + i-1 of target_logits;
 *   draft  q_{b,i} (i = 1..gamma[b])   is row q_row_off[b] + i-1 of draft_logits;
 *   draft token x_{b,i} is draft_tokens[b * gamma_max + i-1].
 * Rows are row_stride elements apart; the logit buffers must be 16-byte
 * aligned and row_stride * element size a multiple of 16 bytes (rows are
 * streamed with bulk asynchronous copies). Rows of different sequences may
 * be packed ragged, shared or interleaved; the library only reads them. */
typedef struct {
    int32_t B;                   /* sequences in the batch, 0 <= B <= max_batch */
    int32_t gamma_max;           /* row length of draft_tokens, <= max_gamma */
    int64_t V;                   /* vocabulary size, 1 <= V <= max_vocab */
    int32_t dtype;               /* specverify_dtype of both logit buffers */
    const void *target_logits;   /* [target_rows, row_stride] */
    const void *draft_logits;    /* [draft_rows, row_stride]; may be NULL for greedy */
    int64_t row_stride;          /* elements between consecutive rows, >= V */
    int64_t target_rows;         /* rows in target_logits (offsets are checked against it) */
    int64_t draft_rows;          /* rows in draft_logits */
    const int64_t *p_row_off;    /* [B] */
    const int64_t *q_row_off;    /* [B]; may be NULL for greedy */
    const int32_t *draft_tokens; /* [B, gamma_max]; may be NULL when gamma_max == 0 */
    const int32_t *gamma;        /* [B], per-sequence lookahead, 0 <= gamma[b] <= gamma_max */
} specverify_batch;

/* Create a handle on CUDA device `device` whose workspace fits any batch with
 * B <= max_batch, gamma_max <= max_gamma (<= 256) and V <= max_vocab. The
 * workspace is device memory owned by the handle until specverify_destroy.
 * The handle is not thread-safe: use one per concurrently used stream. */
int specverify_create(specverify_t *out, int device, int32_t max_batch, int32_t max_gamma,
                      int64_t max_vocab);

/* Release the handle and its workspace. Work still queued on a stream that
 * uses the handle must have completed. NULL is accepted. */
int specverify_destroy(specverify_t h);

/* Sampling verify (temperature > 0, finite). Outputs (device, caller-owned):
 *   n_accepted [B]              accepted draft count n in [0, gamma[b]]; emitted = n+1;
 *                               -1 for a sequence with bad input;
 *   out_tokens [B, gamma_max+1] x_1..x_n, the final token, then -1 padding;
 *   p_lse, q_lse (nullable)     natural-log logsumexp of target_i / T (resp. draft_i / T),
 *                               written at the row's index in its logit buffer, for every
 *                               row the batch uses.
 * When both p_lse and q_lse are NULL, only the rows the result depends on are
 * read: p_1..p_{n+1} and q_1..q_{min(n+1, gamma)} of each sequence (rows after
 * the first rejection cannot change n or any token, as the accept scan stops
 * there). Bad logits in rows that are not read are then not detected. With
 * either output requested, every row is read and validated. A small batch
 * (B <= 8, gamma_max <= 16, at most 16 MiB of logits) runs as one cluster of
 * 8 CTAs per sequence (timing id 8) that reads every row; its bad-logit check
 * still covers only the rows above unless an lse output is requested, so the
 * results are the same as the large-batch kernel's.
 * seed keys the counter-based uniforms; pass a fresh seed per call. */
int specverify_verify(specverify_t h, const specverify_batch *in, float temperature,
                      uint64_t seed, int32_t *n_accepted, int32_t *out_tokens, float *p_lse,
                      float *q_lse, void *cuda_stream);

/* Lossy sampling verify: specverify_verify with the accept test
 * r_i <= f(p_i(x_i), eps) / q_i(x_i) for lenience in SPECVERIFY_LENIENCE_*
 * and eps in (0, 1] (anything else returns SPECVERIFY_ERR_INVALID_ARG).
 * The output distribution then differs from the target's unless eps = 1;
 * everything else -- arguments, outputs, rows read, errors -- is as in
 * specverify_verify, which equals this call with SPECVERIFY_LENIENCE_NONE. */
int specverify_verify_lossy(specverify_t h, const specverify_batch *in, float temperature,
                            uint64_t seed, int32_t lenience, float eps, int32_t *n_accepted,
                            int32_t *out_tokens, float *p_lse, float *q_lse, void *cuda_stream);

/* Greedy verify (temperature 0): reads the target rows only. Outputs as
 * specverify_verify. A batch of at most 8 sequences with gamma_max <= 16
 * takes one cluster kernel (8 CTAs per sequence, timing id 8): each CTA the
 * first argmax of its column slice of every target row, folded in column
 * order, then the exact-match scan; larger batches take the plan, row
 * statistics and accept kernels. Both give the same results. */
int specverify_verify_greedy(specverify_t h, const specverify_batch *in, int32_t *n_accepted,
                             int32_t *out_tokens, void *cuda_stream);

/* Restricted sampling verify ("Speculative Decoding and Distillation"
 * (Kadimisetty notes), "Greedy vs sampling": temperature, top-k and top-p
 * apply to the target and the draft alike, and the accept / residual rule
 * runs on the restricted distributions). Per sequence b (device arrays,
 * caller-owned): temperature[b] > 0 and finite, top_k[b] in [1, 32], top_p[b]
 * in (0, 1] (top_p NULL: 1). A row l restricted with (T, k, p) keeps its
 * min(k, V) largest logits (ties: the lower token index first), weighs them
 * w_j = exp(l_j / T - l_max / T), keeps the shortest prefix in that order
 * whose weight reaches p times the top-k total, and normalises over it; every
 * other token has probability 0. p'_i and q'_i are the restricted target and
 * draft rows; the accept test is r_i <= p'_i(x_i) / q'_i(x_i) (+inf when
 * q'_i(x_i) = 0 < p'_i(x_i), 0 when both are 0), the residual is
 * norm(max(0, p'_{n+1} - q'_{n+1})) and the bonus token comes from
 * p'_{gamma+1}; uniforms, index-order draw and outputs as in
 * specverify_verify. Every row of every valid sequence is read once; a
 * sequence with a bad gamma, row offset, token, parameter
 * (SPECVERIFY_STATUS_BAD_PARAM) or logit in any of its rows gets
 * n_accepted[b] = -1 and tokens -1. The restricted weights come from a
 * table-driven float-float exponential (relative error about 1e-13); their
 * prefix sums, the top-p cut, the probabilities and the draw are
 * float-float (about 48 bits), the accept ratio float (about 1e-7).
 * Three kernel launches (timing ids 5, 6 and 7) on cuda_stream;
 * B * (2 gamma_max + 1) rows, and that many times ceil(V * element size /
 * 4096), must stay below 2^31. */
int specverify_verify_restricted(specverify_t h, const specverify_batch *in,
                                 const float *temperature, const int32_t *top_k,
                                 const float *top_p, uint64_t seed, int32_t *n_accepted,
                                 int32_t *out_tokens, void *cuda_stream);

/* Acceptance statistics of every position ("DistillSpec" Sec. 3: the
 * acceptance rate beta = sum_x min(p(x), q(x)), the probability that the
 * accept test passes when x ~ q; Sec. 4: the total variation distance
 * TVD = 1/2 sum_x |p(x) - q(x)| = 1 - beta as its proxy), with
 * p = softmax(p_{b,i} / T) and q = softmax(q_{b,i} / T) for i = 1..gamma[b].
 * Outputs (device, caller-owned, float): beta[b * gamma_max + i-1] and
 * tvd[b * gamma_max + i-1]; NaN for i > gamma[b] and for a position whose
 * rows are bad (sticky status bits as in specverify_verify). tvd is computed
 * as 1 - beta (at least 0). Both rows of every position are read twice, the
 * second time partly from L2. Sums are fp32: absolute error about 1e-6.
 * Asynchronous on cuda_stream. */
int specverify_acceptance_stats(specverify_t h, const specverify_batch *in, float temperature,
                                float *beta, float *tvd, void *cuda_stream);

/* Draft-distribution features ("Dynamic Speculation Lookahead ..." Sec. 3
 * Eq. 2 and App. D.1: the lookahead classifier's inputs): for each of the
 * nrows rows of `rows` (device, dtype, row_stride elements apart, 16-byte
 * aligned rows), with q = softmax(row / T):
 *   entropy[r]                 -sum_v q_v ln q_v (nats);
 *   topk_prob[r * k + j]       the j-th largest q_v, j < k <= 32;
 *   topk_idx[r * k + j]        its token index (ties: the lower index first);
 *                              -1 (probability 0) past V.
 * A row with a NaN or +inf logit, or with every logit -inf, gets NaN and
 * -1 and sets SPECVERIFY_STATUS_BAD_LOGIT. One pass over every row (in
 * blocks of max_batch (2 max_gamma + 1) rows: two launches per block, the
 * row pass and the per-row merge). Asynchronous on cuda_stream; uses the
 * handle's device, status and workspace (one stream per handle, as for the
 * verify calls). V < 2^31. */
int specverify_row_features(specverify_t h, const void *rows, int32_t dtype, int64_t nrows,
                            int64_t V, int64_t row_stride, float temperature, int32_t k,
                            float *entropy, float *topk_prob, int32_t *topk_idx,
                            void *cuda_stream);

/* Synchronise `cuda_stream`, return the sticky status bits accumulated since
 * the last call in *status_out (0 = clean) and clear them. */
int specverify_device_status(specverify_t h, void *cuda_stream, int32_t *status_out);

/* Human-readable text of a return code. Never NULL. */
const char *specverify_status_string(int status);

/* Device workspace bytes held by the handle. */
int specverify_workspace_bytes(specverify_t h, size_t *out);

/* Kernel timing (diagnostics for roofline accounting). When enabled, every
 * verify call records CUDA events on its stream around each kernel. Kernel
 * ids: 0 = plan, 1 = row statistics, 2 = residual/bonus draw (standalone, not
 * launched by these entry points), 3 = row combine and accept scan, 4 =
 * fused sampling kernel, 5 = restricted-verify plan, 6 = restricted-verify
 * row pass, 7 = restricted-verify finalisation, 8 = small-batch sampling or
 * greedy kernel. specverify_verify launches 4 only, or 8 for a small batch
 * (plan, row statistics, accept tests and draw in one persistent kernel);
 * specverify_verify_greedy launches 0, 1 and 3, or 8 for a small batch;
 * specverify_verify_restricted launches 5, 6 and 7.
 * specverify_get_timing waits for the recorded events, returns the summed
 * milliseconds and the launch count of kernel `kernel` since the last reset,
 * and resets them when reset != 0. Timing adds no synchronisation to verify. */
int specverify_set_timing(specverify_t h, int enable);
int specverify_get_timing(specverify_t h, int kernel, double *total_ms, int64_t *launches,
                          int reset);

/* Bound, in nanoseconds of GPU wall time, on every wait of specverify_verify's
 * fused kernel for another warp (a position's chunk partials, an idle task
 * loop); 0 restores the default of about two seconds. A wait that runs out
 * sets SPECVERIFY_STATUS_TIMEOUT, every other wait of that call then returns
 * at once, and the kernel returns with the sequences it had not decided left
 * at n_accepted[b] = -1 (tokens -1). A warp's waits on its own bulk copies
 * keep their fixed bound of about two seconds, so no kernel exits with a copy
 * in flight. A limit far below the call's duration makes calls time out:
 * this exists for failure-detection tests and watchdog tuning. */
int specverify_set_wait_limit(specverify_t h, uint64_t ns);

/* Sampling verify that allocates nothing. The paper has no counterpart: this
 * entry point exists for callers that may not call cudaMalloc -- a serving
 * process whose memory pool has already taken all free device memory, or a
 * latency-critical path where an allocation's implicit device-wide
 * synchronisation would stall other streams. It needs no handle: the verify
 * step runs as separate plan, row-statistics, accept and draw kernels (the
 * same arithmetic as specverify_verify's fused kernel, so the same results)
 * with their workspace in one fixed device array of about 1.8 MiB that every
 * GPU loading the library holds until the process exits. Every row is read.
 * Inputs, outputs, their meaning and layout are those of specverify_verify;
 * the device is the current CUDA device.
 * Limits: B <= 64, gamma_max <= 16, V <= 262144; larger batches return
 * SPECVERIFY_ERR_TOO_LARGE and launch nothing.
 * The first call on each device sets that device up (it looks up the array's
 * device address and copies a 32 KiB table into it, synchronously), so make
 * that first call before any stream capture; a set-up that fails returns its
 * error and the next call on that device tries again. Calls share the one array:
 * calls that can overlap on the GPU (different streams, different host
 * threads) corrupt each other, so keep them on one stream. Bad input gives
 * n_accepted[b] = -1 for its sequence; this entry point reports no status
 * word. */
int specverify_verify_noalloc(const specverify_batch *in, float temperature, uint64_t seed,
                              int32_t *n_accepted, int32_t *out_tokens, float *p_lse,
                              float *q_lse, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
