// Host-side launch entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "params.h"

namespace fl {

// maps: Q0, K0, V, Q1, K1, O, PB, MB (Q1/K1 are the second branch for
// differential attention and copies of Q0/K0 otherwise; O is the output,
// stored by TMA; PB / MB are the Evoformer pair-bias and mask-bias maps,
// copies of Q0 when unused).
#define FL_DECLARE_ATTN(D, DV)                                                                      \
  cudaError_t launch_attn_d##D##_dv##DV(int score_mod, const CUtensorMap* maps, const KParams& p, int grid, \
                                        cudaStream_t s);
FL_DECLARE_ATTN(32, 32)
FL_DECLARE_ATTN(32, 64)
FL_DECLARE_ATTN(32, 128)
FL_DECLARE_ATTN(64, 32)
FL_DECLARE_ATTN(64, 64)
FL_DECLARE_ATTN(64, 128)
FL_DECLARE_ATTN(128, 32)
FL_DECLARE_ATTN(128, 64)
FL_DECLARE_ATTN(128, 128)
#undef FL_DECLARE_ATTN

cudaError_t launch_diff_d64(const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s);
cudaError_t launch_evo_row(const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s);
cudaError_t launch_evo_col(int d, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s);

}  // namespace fl
