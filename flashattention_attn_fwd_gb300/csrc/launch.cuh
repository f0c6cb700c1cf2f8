// Launch helper shared by the kernel translation units.
#pragma once

#include "fused_attn.cuh"
#include "kernels.h"

namespace fl {

template <int D, int DV, int KIND, int SCORE>
cudaError_t launch_fused(const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t stream) {
  auto kern = fused_attn_fwd_kernel<D, DV, KIND, SCORE>;
  constexpr int smem = Layout<D, DV, KIND>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_attn_by_score(int score_mod, const CUtensorMap* maps, const KParams& p, int grid,
                                 cudaStream_t s) {
  switch (score_mod) {
    case SCORE_NONE: return launch_fused<D, D, KIND_ATTN, SCORE_NONE>(maps, p, grid, s);
    case SCORE_ALIBI: return launch_fused<D, D, KIND_ATTN, SCORE_ALIBI>(maps, p, grid, s);
    case SCORE_SOFTCAP: return launch_fused<D, D, KIND_ATTN, SCORE_SOFTCAP>(maps, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fl
