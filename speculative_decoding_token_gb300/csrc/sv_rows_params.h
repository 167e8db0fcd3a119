// sv_rows_params.h -- parameters of the per-row kernels beside the verify
// step: the row diagnostics (sv_features.cu) and the restricted verify
// (sv_restrict.cu), with their launchers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// A (logit, token) entry of a row's top list.
struct RTop {
    float v;
    int32_t i;
};

// Row diagnostics (sv_features.cu): acceptance statistics of position pairs
// and draft features of rows.
struct FeatParams {
    const char *rows;       // features: the rows; pairs: the target rows
    const char *rows2;      // pairs: the draft rows
    int64_t stride_bytes;
    int64_t V;
    int64_t row_bytes;
    int64_t nrows;          // features: rows; pairs: B
    const int64_t *p_row_off, *q_row_off;
    const int32_t *gamma;
    int64_t target_rows, draft_rows;
    int32_t gamma_max;
    int32_t k;              // top-k size (features)
    float c2;               // log2(e) / T
    uint32_t ninf_sub;      // features, bf16: a finite bf16 pair that stands in for logits
                            // below it in the sums (-inf among them), see features_rows_kernel
    float *entropy;         // [nrows]
    float *topk_prob;       // [nrows, k]
    int32_t *topk_idx;      // [nrows, k]
    float *beta, *tvd;      // [B, gamma_max]
    int32_t *status;        // sticky status word (may be null)
    // features: the row pass's pieces (workspace shared with the restricted verify)
    RTop *parts;            // [ranges, cap, 32] each piece's best (logit, token) pairs
    float4 *pstat;          // [ranges, cap] each piece's (max, sum, entropy sum, flags)
    int32_t cap;            // pieces per range of the split
    int32_t row_grid;       // CTAs of the row pass
};

constexpr int kMaxTopK = 32;

// Restricted sampling (sv_restrict.cu): per sequence a temperature, a top-k
// (1..kMaxRestrictK) and a top-p.
constexpr int kMaxRestrictK = 32;

// One logical row of a restricted verify: sequence b's rows are p_0..p_gamma
// (j = 0..gamma) then q_0..q_{gamma-1} (j = gamma+1..2 gamma), cnt = 2 gamma + 1.
struct RRow {
    const char *addr;
    int32_t b;
    uint16_t j;
    uint16_t cnt;
};

struct RestrictParams {
    const char *target, *draft;
    int64_t stride_bytes;
    int64_t V;
    int64_t row_bytes;
    int64_t target_rows, draft_rows;
    int32_t B, gamma_max;
    const int64_t *p_row_off, *q_row_off;
    const int32_t *tokens, *gamma;
    const float *temperature;    // [B]
    const int32_t *top_k;        // [B]
    const float *top_p;          // [B] or null (1)
    uint64_t seed;
    int32_t *n_out, *tok_out;
    int32_t *status;
    const float2 *exp2_tab;      // 2^(j/4096) as float-float pairs (handle workspace)
    // workspace
    RRow *rows;                  // [max rows]
    int32_t *total_rows;         // rows of the call (plan output)
    RTop *parts;                 // [ranges, cap, kMaxRestrictK]: the list of each row piece
    int32_t cap;                 // list slots per range of the stage split
    int2 *seq_rows;              // [max_batch] (first row, rows); rows 0: a bad sequence
    int32_t row_grid;            // CTAs of the row pass (the split depends on it)
    uint32_t *seq_flag;          // [max_batch] 1: a bad logit, 2: a wait gave up; reset by
                                 // the finalisation
    uint32_t *row_fin;           // [max rows] 1: the row holds a finite logit; reset likewise
};

// warps per CTA of the restricted kernel (one CTA per SM)
constexpr int kRestrictWarps = 16;
// Ranges of the restricted kernel's stage split per warp: the split has this
// many ranges per warp and warp w streams ranges w, w + W, w + 2W, ... (W
// warps). One range per warp measured fastest: every row piece starts its
// top-32 list cold, so fewer, longer pieces cost less, and the streaming
// itself ran at the same speed for 1 and 4 ranges.
constexpr int kRestrictRangesPerWarp = 1;

// Kernel launchers (sv_features.cu, sv_restrict.cu)
cudaError_t launch_features(const FeatParams &p, int dtype, cudaStream_t s);
cudaError_t launch_pairs(const FeatParams &p, int dtype, int num_sms, cudaStream_t s);
cudaError_t launch_restrict_plan(const RestrictParams &p, cudaStream_t s);
cudaError_t launch_restrict_rows(const RestrictParams &p, int dtype, cudaStream_t s);
cudaError_t launch_restrict_final(const RestrictParams &p, cudaStream_t s);
cudaError_t prepare_features();
cudaError_t prepare_restricted();

}  // namespace sv
