// Evoformer MSA row-wise gated self-attention forward (pair bias broadcast
// over the MSA rows, per-row residue mask bias, sigmoid gate epilogue).
#include "launch.cuh"

namespace fl {
cudaError_t launch_evo(int d, const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t s) {
  if (d == 32) return launch_fused<32, 32, KIND_EVO, SCORE_NONE>(maps, p, grid, s);
  if (d == 64) return launch_fused<64, 64, KIND_EVO, SCORE_NONE>(maps, p, grid, s);
  return cudaErrorInvalidValue;
}
}  // namespace fl
