// Fused attention forward, head dim 32.
#include "launch.cuh"

namespace fl {
cudaError_t launch_attn_d32(int score_mod, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s) {
  return launch_attn_by_score<32>(score_mod, maps, p, grid, s);
}
}  // namespace fl
