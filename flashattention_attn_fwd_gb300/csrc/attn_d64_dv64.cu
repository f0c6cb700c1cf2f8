// Fused attention forward, head dim 64, value head dim 64 (vanilla / ALiBi / softcap score, any mask).
#include "launch.cuh"

namespace fl {
cudaError_t launch_attn_d64_dv64(int score_mod, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s) {
  return launch_attn_by_score<64, 64>(score_mod, maps, p, grid, s);
}
}  // namespace fl
