// Evoformer MSA gated attention: row-wise (head dim 32; pair bias staged per
// key tile and shared by two MSA rows) and column-wise (head dim 32 or 64).
#include "launch.cuh"

namespace fl {
cudaError_t launch_evo_row(const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s) {
  return launch_fused<32, 32, KIND_EVO, SCORE_NONE>(maps, p, grid, s);
}
cudaError_t launch_evo_col(int d, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s) {
  return d == 32 ? launch_fused<32, 32, KIND_EVO_COL, SCORE_NONE>(maps, p, grid, s)
                 : launch_fused<64, 64, KIND_EVO_COL, SCORE_NONE>(maps, p, grid, s);
}
}  // namespace fl
