// Launch helper shared by the kernel translation units.
#pragma once

#include "fused_attn.cuh"
#include "kernels.h"

namespace fl {

template <int D, int DV, int KIND, int SCORE>
cudaError_t launch_fused(const CUtensorMap* maps, const KParams& p, int grid, cudaStream_t stream) {
  auto kern = fused_attn_fwd_kernel<D, DV, KIND, SCORE>;
  constexpr int smem = Layout<D, DV, KIND, SCORE>::SMEM_BYTES;
  // The register split (setmaxnreg) hands the control warpgroup's registers
  // to the softmax warpgroups; it needs exactly kLaunchRegs per thread at
  // launch, or the softmax warpgroups would wait for registers forever.
  static const cudaError_t checked = [&]() {
    cudaFuncAttributes a{};
    cudaError_t e = cudaFuncGetAttributes(&a, kern);
    if (e != cudaSuccess) return e;
    if (a.numRegs != kLaunchRegs) return cudaErrorInvalidDeviceFunction;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  }();
  if (checked != cudaSuccess) return checked;
  kern<<<grid, kThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7],
                                         p);
  return cudaGetLastError();
}

template <int D, int DV>
cudaError_t launch_attn_by_score(int score_mod, const CUtensorMap* maps, const KParams& p, int grid,
                                 cudaStream_t s) {
  switch (score_mod) {
    case SCORE_NONE: return launch_fused<D, DV, KIND_ATTN, SCORE_NONE>(maps, p, grid, s);
    case SCORE_ALIBI: return launch_fused<D, DV, KIND_ATTN, SCORE_ALIBI>(maps, p, grid, s);
    case SCORE_SOFTCAP: return launch_fused<D, DV, KIND_ATTN, SCORE_SOFTCAP>(maps, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fl
