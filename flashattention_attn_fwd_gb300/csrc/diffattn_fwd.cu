// Differential attention forward: two query/key branches of head dim 64
// sharing one value tile of 128 channels; out = O1/l1 - lambda O2/l2.
#include "launch.cuh"

namespace fl {
cudaError_t launch_diff_d64(const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s) {
  return launch_fused<64, 128, KIND_DIFF, SCORE_NONE>(maps, p, grid, s);
}
}  // namespace fl
