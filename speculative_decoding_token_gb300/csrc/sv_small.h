// sv_small.h -- the small-batch sampling and greedy kernels (sv_small.cu): one cluster of
// kSmallCtas CTAs per sequence, used for batches small enough that the fused
// kernel's grid-wide machinery (grid barriers, queues, tickets) would be most
// of the step.
#pragma once

#include "sv_internal.h"

namespace sv {

constexpr int kSmallCtas = 8;       // CTAs per sequence (a portable cluster size)
constexpr int kSmallWarps = 16;     // warps per CTA
constexpr int kSmallMaxGamma = 16;  // gamma_max of a small batch
constexpr int kSmallMaxB = 8;       // sequences of a small batch
// dynamic shared memory of a CTA: the exp2 table, then its slice of every row
constexpr int kSmallSmem = 200 * 1024;

// Bytes of dynamic shared memory the small kernel needs for a call: the table
// and (2 gamma_max + 1) row slices of ceil(V / kSmallCtas) elements rounded up
// to whole 16-byte vectors.
inline int64_t small_smem_bytes(const Params &p) {
    const int64_t esz = p.row_bytes / (p.V > 0 ? p.V : 1);
    const int64_t pv = 16 / esz;
    const int64_t per = ((p.V + kSmallCtas - 1) / kSmallCtas + pv - 1) / pv * pv;
    return (int64_t)kExpTab * 8 + (2 * (int64_t)p.gamma_max + 1) * (per / pv) * 16;
}

cudaError_t prepare_small();
cudaError_t launch_small(const Params &p, int dtype, cudaStream_t s);
// the greedy step for a batch of at most kSmallMaxB sequences with gamma_max
// at most kSmallMaxGamma (rows read from global memory: no size limit of its own)
cudaError_t launch_small_greedy(const Params &p, int dtype, cudaStream_t s);

}  // namespace sv
