// Decode-phase (key/value cache) attention: parameters shared by the host
// launcher and the kernels (internal header).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fl {

// Query rows one CTA serves: the (Hq / Hkv) heads of a group times Lq.
constexpr int kDecodeMaxRows = 64;

struct DecodeParams {
  const void* q;          // bf16 [B, Hq, Lq, D]
  void* out;              // bf16 [B, Hq, Lq, D]
  float* lse;             // fp32 [B, Hq, Lq] (natural log) or null
  const int32_t* kv_len;  // int32 [B] or null (= Lmax)
  const float* slopes;    // ALiBi slopes [Hq]
  float* opart;           // fp32 [n_split, rows, D] normalised partial outputs
  float* lpart;           // fp32 [n_split, rows] partial log-sum-exp (log2)
  uint32_t* status;       // device status words
  uint64_t timeout_ns;
  int B, Hq, Hkv, Lq, Lmax;
  int n_split, chunk;     // key splits and keys per split (a multiple of 128)
  int64_t rows;           // B * Hq * Lq
  float scale, softcap;
  int score_mod, causal;
};

// Query rows one CTA of the warp-level decode kernel serves (larger M uses
// the block-phase kernel).
constexpr int kDecodeWarpRows = 8;

// Number of key splits and keys per split for a problem on `sm_count` SMs
// with M = (Hq / Hkv) * Lq query rows per CTA: enough CTAs for several waves
// (cache lengths differ per sequence, and a split past a sequence's length
// has no work) -- four per SM for the warp-level kernel, whose CTAs stream
// longer ranges well, sixteen for the block-phase kernel -- and whole
// 128-key tiles per split.
inline void decode_split(int B, int Hkv, int Lmax, int M, int sm_count, int* n_split, int* chunk) {
  const int tiles = (Lmax + 127) / 128;
  const int heads = B * Hkv;
  const int per_sm = M <= kDecodeWarpRows ? 4 : 16;
  int ns = (per_sm * sm_count + heads - 1) / heads;
  ns = ns < 1 ? 1 : (ns > tiles ? tiles : ns);
  const int tiles_per = (tiles + ns - 1) / ns;
  *chunk = tiles_per * 128;
  *n_split = (tiles + tiles_per - 1) / tiles_per;
}

cudaError_t launch_decode(int d, const CUtensorMap* maps, const DecodeParams& p, cudaStream_t stream);

}  // namespace fl
