// Backward pass of the fused attention: parameters shared by the host
// launcher and the kernels (internal header).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fl {

struct BwdParams {
  const void* out;        // bf16 [B, Hq, Lq, DV] forward output
  const void* dout;       // bf16 [B, Hq, Lq, DV] gradient of the output
  const float* lse;       // fp32 [B, Hq, Lq] forward log-sum-exp (natural log)
  void* dq;               // bf16 [B, Hq, Lq, D]
  void* dk;               // bf16 [B, Hkv, Lk, D]
  void* dv;               // bf16 [B, Hkv, Lk, DV]
  float* dq_acc;          // fp32 [B, Hq, Lq, D] workspace
  float* dvec;            // fp32 [B, Hq, Lq] workspace: rowsum(dO * O)
  float* l2;              // fp32 [B, Hq, Lq] workspace: LSE * log2(e)
  const float* slopes;    // ALiBi slopes [Hq]
  const int32_t* doc_offsets;
  uint32_t* status;
  uint64_t timeout_ns;
  int B, Hq, Hkv, Lq, Lk;
  int n_ktiles;           // ceil(Lk / 128)
  int64_t rows;           // B * Hq * Lq
  float scale, softcap;
  // softcap on the FMA pipe, as in the forward: cap*log2(e)*tanh(s*scale/cap)
  // = s * (q0 + q1 s^2 + q2 s^4 + q3 s^6) while |s| <= sc_smax
  float sc_q[4];
  float sc_smax;
  int mask_kind, doc_causal, window, prefix, num_docs;
  // the gradients are those of dout_scale * dout (1 for the plain backward;
  // -lambda for the second branch of differential attention), and with
  // dv_accumulate the kernel adds its dV to the bf16 values already in dv
  float dout_scale;
  int dv_accumulate;
};

// (d, dv): (32, 32), (64, 64), (128, 128) or (64, 128)
cudaError_t launch_bwd(int d, int dv, int score_mod, const CUtensorMap* maps, const BwdParams& p, cudaStream_t s);

}  // namespace fl
