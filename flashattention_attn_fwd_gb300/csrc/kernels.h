// Host-side launch entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "params.h"

namespace fl {

// maps: Q0, K0, V, Q1, K1, O (Q1/K1 are the second branch for differential
// attention and copies of Q0/K0 otherwise; O is the output, stored by TMA).
using LaunchFn = cudaError_t (*)(const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t stream);

cudaError_t launch_attn_d32(int score_mod, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s);
cudaError_t launch_attn_d64(int score_mod, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s);
cudaError_t launch_attn_d128(int score_mod, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s);
cudaError_t launch_diff_d64(const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s);
cudaError_t launch_evo(int d, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s);

}  // namespace fl
