// Fused attention forward, head dim 32, value head dim 32 (vanilla / ALiBi / softcap score, any mask).
#include "launch.cuh"

namespace fl {
cudaError_t launch_attn_d32_dv32(int score_mod, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s) {
  return launch_attn_by_score<32, 32>(score_mod, maps, p, grid, s);
}
}  // namespace fl
