// Decode-phase attention over a key/value cache, split over the key axis.
//
// A few new query rows per sequence (Lq, e.g. one generated token) attend to
// a long cache of kv_len[b] keys.  The work per key is a handful of
// multiply-adds per query row, so the kernel is bound by reading the cache
// from HBM, not by arithmetic: it streams K/V tiles with TMA into an
// mbarrier ring and computes on the CUDA cores (a 128-row tensor-core tile
// would be mostly padding here).  Each CTA owns one (batch, key/value head,
// key range); all G = Hq / Hkv query heads of the group and their Lq rows
// (M = G * Lq rows) share every K/V tile it loads.  With M <= 8 (the usual
// serving case) each warp takes its own 16 keys of every tile and keeps its
// own online-softmax state, merged once per CTA (decode_warp_kernel); larger
// M uses block-wide phases per tile (decode_split_kernel).  Every split writes its
// normalised partial output and log-sum-exp; a second kernel merges the
// splits with weights 2^(LSE_s - LSE).  This is the split-K/V forward with
// an LSE merge that the Flashlight wiki summary's critical analysis (批判性分析,
// serving path) names for the decode phase; the online softmax inside a
// split is the one the technical summary's Methodology ("Semantic Fusion
// with Algebraic Transformation") describes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "decode.h"
#include "ptx.cuh"

namespace fl {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecTileN = 128;  // keys per tile
constexpr float kDLog2e = 1.4426950408889634f;
constexpr float kDLn2 = 0.6931471805599453f;

template <int D>
struct DecLayout {
  static constexpr int STAGES = D == 128 ? 2 : 3;
  static constexpr int NBOX = D / 64;                     // 64-channel TMA boxes per row
  static constexpr int TILE_BYTES = kDecTileN * D * 2;    // one K (or V) tile
  static constexpr int OFF_K = 0;                          // K[stage]
  static constexpr int OFF_V = STAGES * TILE_BYTES;        // V[stage]
  static constexpr int OFF_Q = 2 * STAGES * TILE_BYTES;    // then, sized by the M rows:
  // fp32 Q [M][D] (pre-scaled), fp32 P [M][128], m / l / alpha [M], barriers
  static int smem_bytes(int M) { return OFF_Q + M * (D + kDecTileN) * 4 + 3 * M * 4 + 8 * STAGES + 16 + 1024; }
};

struct DecCtl {
  uint32_t* status;
  uint64_t timeout_ns;
};

// Bounded wait on a TMA barrier; on expiry the status word records a timeout.
__device__ __forceinline__ bool dec_wait(uint64_t* bar, uint32_t parity, const DecCtl& c, volatile int* abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (ptx::globaltimer_ns() - t0 > c.timeout_ns) {
      *abort = 1;
      atomicOr(c.status, 1u);
      atomicExch(c.status + 1, 40u);
      return false;
    }
  }
  return true;
}

// D: head dim; MR: rows per CTA rounded up to a power of two (>= M).
template <int D, int MR>
__global__ void __launch_bounds__(kDecThreads, MR <= 16 ? 2 : 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ DecodeParams p) {
  using L = DecLayout<D>;
  constexpr int S = L::STAGES;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int split = blockIdx.x % p.n_split;
  const int bh = blockIdx.x / p.n_split;
  const int hkv = bh % p.Hkv;
  const int b = bh / p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int M = G * p.Lq;
  float* qs = reinterpret_cast<float*>(sm + L::OFF_Q);
  float* ps = qs + M * D;
  float* rm = ps + M * kDecTileN;
  float* rl = rm + M;
  float* ra = rl + M;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + ((L::OFF_Q + (M * (D + kDecTileN) + 3 * M) * 4 + 7) & ~7));
  volatile int* abort = reinterpret_cast<volatile int*>(full + S);
  const int kv_len = p.kv_len ? min(max(__ldg(p.kv_len + b), 0), p.Lmax) : p.Lmax;
  const int key_lo = split * p.chunk;
  const int key_hi = min(key_lo + p.chunk, kv_len);  // exclusive
  const int n_tiles = key_hi > key_lo ? (key_hi - key_lo + kDecTileN - 1) / kDecTileN : 0;
  const DecCtl ctl{p.status, p.timeout_ns};

  if (tid == 0) {
    for (int st = 0; st < S; ++st) ptx::mbar_init(&full[st], 1);
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  // query rows m = (head in group) * Lq + i, pre-scaled into the log2 domain
  const float qscale = p.scale * kDLog2e;
  for (int e = tid; e < M * D; e += kDecThreads) {
    const int m = e / D, c = e % D;
    const int h = hkv * G + m / p.Lq, i = m % p.Lq;
    const __nv_bfloat16* qr = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                              ((static_cast<int64_t>(b) * p.Hq + h) * p.Lq + i) * D;
    qs[m * D + c] = __bfloat162float(qr[c]) * qscale;
  }
  if (tid < M) {
    rm[tid] = -CUDART_INF_F;
    rl[tid] = 0.f;
  }
  __syncthreads();

  // thread 0 streams the split's K/V tiles (read once: L2 evict-first)
  int issued = 0;
  auto issue = [&](int t) {
    const int st = t % S;
    const uint64_t pol = ptx::policy_evict_first();
    ptx::mbar_arrive_expect_tx(&full[st], 2u * L::TILE_BYTES);
#pragma unroll
    for (int bx = 0; bx < L::NBOX; ++bx) {
      ptx::tma_load_4d(sm + L::OFF_K + st * L::TILE_BYTES + bx * kDecTileN * 128, &tmK, &full[st], 64 * bx,
                       key_lo + t * kDecTileN, hkv, b, pol);
      ptx::tma_load_4d(sm + L::OFF_V + st * L::TILE_BYTES + bx * kDecTileN * 128, &tmV, &full[st], 64 * bx,
                       key_lo + t * kDecTileN, hkv, b, pol);
    }
    issued = t + 1;
  };
  if (tid == 0)
    for (int t = 0; t < S && t < n_tiles; ++t) issue(t);

  // P V: thread -> channel pair cp and key group g (keys j = g mod NG), with
  // accumulators for all rows; the key groups are summed once at the end
  constexpr int CP = D / 2;                        // channel pairs
  constexpr int NG = kDecThreads / CP;             // key groups: 8 (D=64) or 4 (D=128)
  const int cp = tid % CP;
  const int g = tid / CP;
  float2 acc[MR];
#pragma unroll
  for (int k = 0; k < MR; ++k) acc[k] = make_float2(0.f, 0.f);

  bool ok = true;
  int t = 0;
  for (; t < n_tiles; ++t) {
    const int st = t % S;
    if (!dec_wait(&full[st], (t / S) & 1u, ctl, abort)) ok = false;
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    const uint8_t* ks = sm + L::OFF_K + st * L::TILE_BYTES;
    const uint8_t* vs = sm + L::OFF_V + st * L::TILE_BYTES;
    const int j0 = key_lo + t * kDecTileN;
    // ---- scores: thread -> key j, rows m = mhalf, mhalf + 2, ...
    {
      const int j = tid % kDecTileN;
      const int mhalf = tid / kDecTileN;
      const int jg = j0 + j;
#pragma unroll 1
      for (int m0 = mhalf; m0 < M; m0 += 2 * 4) {
        // two packed accumulators per row: four independent FMA chains per
        // 8-channel chunk and row
        float2 acc2[4][2];
#pragma unroll
        for (int r = 0; r < 4; ++r) acc2[r][0] = acc2[r][1] = make_float2(0.f, 0.f);
#pragma unroll 2
        for (int c = 0; c < D / 8; ++c) {
          const int bx = c >> 3, cq = c & 7;
          const uint4 kw = *reinterpret_cast<const uint4*>(ks + bx * kDecTileN * 128 + j * 128 + ((cq ^ (j & 7)) << 4));
          const float2 k01 = make_float2(__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xffff0000u));
          const float2 k23 = make_float2(__uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xffff0000u));
          const float2 k45 = make_float2(__uint_as_float(kw.z << 16), __uint_as_float(kw.z & 0xffff0000u));
          const float2 k67 = make_float2(__uint_as_float(kw.w << 16), __uint_as_float(kw.w & 0xffff0000u));
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int m = m0 + 2 * r;
            if (m < M) {
              const float4 qa = *reinterpret_cast<const float4*>(qs + m * D + 8 * c);
              const float4 qb = *reinterpret_cast<const float4*>(qs + m * D + 8 * c + 4);
              acc2[r][0] = ptx::fma2(make_float2(qa.x, qa.y), k01, acc2[r][0]);
              acc2[r][1] = ptx::fma2(make_float2(qa.z, qa.w), k23, acc2[r][1]);
              acc2[r][0] = ptx::fma2(make_float2(qb.x, qb.y), k45, acc2[r][0]);
              acc2[r][1] = ptx::fma2(make_float2(qb.z, qb.w), k67, acc2[r][1]);
            }
          }
        }
        float sacc[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) sacc[r] = (acc2[r][0].x + acc2[r][0].y) + (acc2[r][1].x + acc2[r][1].y);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int m = m0 + 2 * r;
          if (m >= M) break;
          const int h = hkv * G + m / p.Lq, i = m % p.Lq;
          const int pos = kv_len - p.Lq + i;  // position of this query row
          float x = sacc[r];                  // log2 units
          if (p.score_mod == 2) {
            const float kc = p.softcap * kDLog2e;
            x = kc * tanhf(x / kc);
          } else if (p.score_mod == 1) {
            x = fmaf(__ldg(p.slopes + h) * kDLog2e, static_cast<float>(jg - pos), x);
          }
          const bool vis = jg < key_hi && (!p.causal || jg <= pos);
          ps[m * kDecTileN + j] = vis ? x : -CUDART_INF_F;
        }
      }
    }
    __syncthreads();
    // ---- online softmax: one warp per row
    {
      const int w = tid >> 5, lane = tid & 31;
      for (int m = w; m < M; m += kDecThreads / 32) {
        float4 v = *reinterpret_cast<float4*>(ps + m * kDecTileN + 4 * lane);
        float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_old = rm[m];
        const float m_new = fmaxf(m_old, mx);
        const float msub = m_new == -CUDART_INF_F ? 0.f : m_new;
        v.x = exp2f(v.x - msub);
        v.y = exp2f(v.y - msub);
        v.z = exp2f(v.z - msub);
        v.w = exp2f(v.w - msub);
        *reinterpret_cast<float4*>(ps + m * kDecTileN + 4 * lane) = v;
        float sum = (v.x + v.y) + (v.z + v.w);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) {
          const float alpha = m_old == -CUDART_INF_F ? 0.f : exp2f(m_old - msub);
          ra[m] = alpha;
          rl[m] = rl[m] * alpha + sum;
          rm[m] = m_new;
        }
      }
    }
    __syncthreads();
    // ---- O += P V over this thread's key group
    {
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        if (m < M) {
          const float a = ra[m];
          acc[m].x *= a;
          acc[m].y *= a;
        }
      }
      const int bx = cp >> 5;                 // 64-channel box
      const int cq = (cp & 31) >> 2;          // 16-byte chunk in the 128-byte row
      const int cw = (cp & 3) * 4;            // byte offset in the chunk
#pragma unroll 2
      for (int j = g; j < kDecTileN; j += NG) {
        const uint32_t vw = *reinterpret_cast<const uint32_t*>(vs + bx * kDecTileN * 128 + j * 128 +
                                                              ((cq ^ (j & 7)) << 4) + cw);
        const float v0 = __uint_as_float(vw << 16), v1 = __uint_as_float(vw & 0xffff0000u);
        const float2 v01 = make_float2(v0, v1);
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          if (m < M) {
            const float pj = ps[m * kDecTileN + j];
            acc[m] = ptx::fma2(make_float2(pj, pj), v01, acc[m]);
          }
        }
      }
    }
    __syncthreads();
    // the stage is free: refill it with tile t + S
    if (tid == 0 && t + S < n_tiles) issue(t + S);
  }
  if (!ok) {
    // let the copies this CTA started land before it exits (bounded)
    if (tid == 0) {
      for (int tt = t; tt < issued; ++tt) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(&full[tt % S], (tt / S) & 1u))
          if (ptx::globaltimer_ns() - t0 > 50ull * 1000ull * 1000ull) break;
      }
    }
    __syncthreads();
    return;
  }
  // ---- sum the key groups (shared-memory atomics into the P area), then
  // write the partial (or, with one split, final) results
  float* osum = ps;  // [M][D] fp32
  for (int e = tid; e < M * D; e += kDecThreads) osum[e] = 0.f;
  __syncthreads();
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    if (m < M) {
      atomicAdd(&osum[m * D + 2 * cp], acc[m].x);
      atomicAdd(&osum[m * D + 2 * cp + 1], acc[m].y);
    }
  }
  __syncthreads();
  for (int e = tid; e < M * CP; e += kDecThreads) {
    const int m = e / CP, c2 = e % CP;
    const int h = hkv * G + m / p.Lq, i = m % p.Lq;
    const int64_t row = (static_cast<int64_t>(b) * p.Hq + h) * p.Lq + i;
    const float l = rl[m];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse2 = l > 0.f ? rm[m] + __log2f(l) : -CUDART_INF_F;
    const float o0 = osum[m * D + 2 * c2] * inv, o1 = osum[m * D + 2 * c2 + 1] * inv;
    if (p.n_split == 1) {
      reinterpret_cast<__nv_bfloat162*>(p.out)[row * CP + c2] = __floats2bfloat162_rn(o0, o1);
      if (c2 == 0 && p.lse) p.lse[row] = lse2 * kDLn2;
    } else {
      const int64_t prow = static_cast<int64_t>(split) * p.rows + row;
      reinterpret_cast<float2*>(p.opart)[prow * CP + c2] = make_float2(o0, o1);
      if (c2 == 0) p.lpart[prow] = lse2;
    }
  }
}

// ---------------------------------------------------------------------------
// Decode with independent warps (M = G * Lq <= 8 query rows per CTA, the
// usual serving case).  Each of the eight warps owns 16 keys of every
// 128-key tile and keeps its own online-softmax state (m, l, O) for the M
// rows.  Per tile and warp both products are one warp-level tile each:
//   S (16 x 16 keys) = Q (16 rows, M used) K^T      mma.m16n8k16, K by ldmatrix
//   O (16 x D)      += P (bf16, from S's registers) V    V by ldmatrix.trans
// -- a 16-key by 8-row contraction is far below the 64/128-row granularity of
// tcgen05, and the kernel is bound by reading the cache, so the warp-level
// MMA is the cheap way to keep the instruction count per byte low.  The last
// warp to finish with a stage (a shared counter) refills it by TMA, so no
// warp waits for the others between tiles; the warps' states are merged once
// at the end with weights 2^(m_w - m).
constexpr int kDwWarps = 8;
constexpr int kDwThreads = 32 * kDwWarps;
constexpr int kDwKeys = kDecTileN / kDwWarps;  // keys per warp per tile (16)
constexpr int kDwRows = kDecodeWarpRows;       // query rows per CTA (rows 8..15 of the MMA tile stay empty)

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a b, m16n8k16, bf16 inputs, fp32 accumulators.  Rows 8..15 of A are
// zero here, so only a0 (row g, k 2t..2t+1) and a2 (row g, k 8+2t..) are passed.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

template <int D>
struct DwLayout {
  static constexpr int STAGES = D == 128 ? 2 : 3;  // two CTAs per SM at D = 64
  static constexpr int NBOX = D / 64;
  static constexpr int TILE_BYTES = kDecTileN * D * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = STAGES * TILE_BYTES;
  static constexpr int OFF_BAR = 2 * STAGES * TILE_BYTES;  // full[S], done[S], issued, abort
  static constexpr int SMEM = OFF_BAR + 16 * STAGES + 16 + 1024;
  // merge area after the loop (reuses the K/V ring): (m, l) [warp][row][2]
  // then O [warp][row][D]
  static constexpr int OFF_MST = 0;
  static constexpr int OFF_MO = kDwWarps * kDwRows * 2 * 4;
  static_assert(OFF_MO + kDwWarps * kDwRows * D * 4 <= 2 * STAGES * TILE_BYTES, "merge area");
};

// Byte offset of the 16-byte chunk (8 channels, block cb) of key row j in a
// K or V tile: 64-channel boxes of 128 rows x 128 bytes, 128-byte swizzle.
__device__ __forceinline__ uint32_t dw_chunk(int j, int cb) {
  return static_cast<uint32_t>((cb >> 3) * kDecTileN * 128 + j * 128 + (((cb & 7) ^ (j & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kDwThreads, D == 64 ? 2 : 1)
    decode_warp_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ DecodeParams p) {
  using L = DwLayout<D>;
  constexpr int S = L::STAGES;
  constexpr int KS = D / 16;  // k-steps of Q K^T; dim tiles of P V: D / 8
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;  // MMA fragment row and column pair
  const int split = blockIdx.x % p.n_split;
  const int bh = blockIdx.x / p.n_split;
  const int hkv = bh % p.Hkv;
  const int b = bh / p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int M = G * p.Lq;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  int* done = reinterpret_cast<int*>(full + S);  // warps finished with each stage (cumulative)
  int* issued = done + S;                        // tiles whose loads were started
  volatile int* abort = reinterpret_cast<volatile int*>(issued + 1);
  const int kv_len = p.kv_len ? min(max(__ldg(p.kv_len + b), 0), p.Lmax) : p.Lmax;
  const int key_lo = split * p.chunk;
  const int key_hi = min(key_lo + p.chunk, kv_len);  // exclusive
  const int n_tiles = key_hi > key_lo ? (key_hi - key_lo + kDecTileN - 1) / kDecTileN : 0;
  const DecCtl ctl{p.status, p.timeout_ns};

  // K and V tile t of the split into its stage (read once: L2 evict-first)
  auto issue = [&](int t) {
    const int st = t % S;
    const uint64_t pol = ptx::policy_evict_first();
    ptx::mbar_arrive_expect_tx(&full[st], 2u * L::TILE_BYTES);
#pragma unroll
    for (int bx = 0; bx < L::NBOX; ++bx) {
      ptx::tma_load_4d(sm + L::OFF_K + st * L::TILE_BYTES + bx * kDecTileN * 128, &tmK, &full[st], 64 * bx,
                       key_lo + t * kDecTileN, hkv, b, pol);
      ptx::tma_load_4d(sm + L::OFF_V + st * L::TILE_BYTES + bx * kDecTileN * 128, &tmV, &full[st], 64 * bx,
                       key_lo + t * kDecTileN, hkv, b, pol);
    }
    atomicMax(issued, t + 1);
  };
  if (tid == 0) {
    for (int st = 0; st < S; ++st) {
      ptx::mbar_init(&full[st], 1);
      done[st] = 0;
    }
    *issued = 0;
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
    for (int t = 0; t < S && t < n_tiles; ++t) issue(t);
  }
  // this lane's query row g (rows >= M are zero): the A fragments of every
  // k-step, bf16 pairs (channels 16 kk + 2 tq, +1 and 16 kk + 8 + 2 tq, +1)
  uint32_t qa[KS][2];
  {
    const bool qv = g < M;
    const int h = hkv * G + (qv ? g : 0) / p.Lq, i = (qv ? g : 0) % p.Lq;
    const uint32_t* qr = reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                          ((static_cast<int64_t>(b) * p.Hq + h) * p.Lq + i) * D);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      qa[kk][0] = qv ? __ldg(qr + 8 * kk + tq) : 0u;
      qa[kk][1] = qv ? __ldg(qr + 8 * kk + 4 + tq) : 0u;
    }
  }
  __syncthreads();
  // this lane's row g: position, ALiBi slope; its state (reference max, sum,
  // O fragments: o[dt][0..1] = O[g][8 dt + 2 tq, +1]; [2..3] stay zero)
  const int gm = g < M ? g : 0;
  const int pos = kv_len - p.Lq + gm % p.Lq;
  const float slope2 = p.score_mod == 1 ? __ldg(p.slopes + hkv * G + gm / p.Lq) * kDLog2e : 0.f;
  const float scale_log2 = p.scale * kDLog2e;
  const float kc = p.softcap * kDLog2e;
  float mrow = -CUDART_INF_F, lrow = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
  const int jw = kDwKeys * warp;                           // this warp's first key in a tile
  const int q8 = lane >> 3, i8 = lane & 7;                 // ldmatrix: matrix and row of this lane
  const int kkey = jw + 8 * (q8 >> 1) + i8;                // K rows: n-tile q8 >> 1
  const int vkey = jw + 8 * (q8 & 1) + i8;                 // V rows: key half q8 & 1
  const uint32_t smb = ptx::smem_u32(sm);
  for (int t = 0; t < n_tiles; ++t) {
    const int st = t % S;
    if (!dec_wait(&full[st], (t / S) & 1u, ctl, abort)) break;
    const uint32_t kb = smb + L::OFF_K + st * L::TILE_BYTES;
    const uint32_t vb = smb + L::OFF_V + st * L::TILE_BYTES;
    // S = Q K^T over the warp's 16 keys (n-tiles of 8 keys)
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t r[4];
      ldsm_x4(r, kb + dw_chunk(kkey, 2 * kk + (q8 & 1)));
      mma_bf16_16816(s0, qa[kk][0], qa[kk][1], r[0], r[1]);
      mma_bf16_16816(s1, qa[kk][0], qa[kk][1], r[2], r[3]);
    }
    // scores of row g at keys j0 + {2tq, 2tq+1, 8+2tq, 9+2tq} (log2 units)
    const int jb = key_lo + t * kDecTileN + jw + 2 * tq;
    float x[4] = {s0[0], s0[1], s1[0], s1[1]};
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = jb + (e >> 1) * 8 + (e & 1);
      float v = x[e] * scale_log2;
      if (p.score_mod == 2) v = kc * tanhf(v / kc);
      else if (p.score_mod == 1) v = fmaf(slope2, static_cast<float>(j - pos), v);
      const bool vis = g < M && j < key_hi && (!p.causal || j <= pos);
      x[e] = vis ? v : -CUDART_INF_F;
      mx = fmaxf(mx, x[e]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // the reference max moves only by more than 2^8 (O rescaled then)
    if (mx > mrow + 8.f || (mrow == -CUDART_INF_F && mx != -CUDART_INF_F)) {
      const float alpha = ptx::ex2(mrow - mx);  // 0 when mrow = -inf
      lrow *= alpha;
      mrow = mx;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        o[dt][0] *= alpha;
        o[dt][1] *= alpha;
      }
    }
    const float mref = mrow == -CUDART_INF_F ? 0.f : mrow;
    float pe[4], sum = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      pe[e] = ptx::ex2(x[e] - mref);
      sum += pe[e];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    lrow += sum;
    // O += P V: P is the A fragment straight from S's registers (row g,
    // keys 2tq.. and 8 + 2tq..); V fragments by transposing loads
    const uint32_t pa0 = ptx::pack_bf16x2(pe[0], pe[1]), pa2 = ptx::pack_bf16x2(pe[2], pe[3]);
#pragma unroll
    for (int dd = 0; dd < D / 16; ++dd) {
      uint32_t r[4];
      ldsm_x4_t(r, vb + dw_chunk(vkey, 2 * dd + (q8 >> 1)));
      mma_bf16_16816(o[2 * dd], pa0, pa2, r[0], r[1]);
      mma_bf16_16816(o[2 * dd + 1], pa0, pa2, r[2], r[3]);
    }
    // the last warp done with this stage refills it with tile t + S
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&done[st], 1) % kDwWarps == kDwWarps - 1 && t + S < n_tiles) issue(t + S);
    }
  }
  __syncthreads();
  if (*abort) {
    // let the copies still in flight land before the block exits (bounded)
    if (tid == 0) {
      const int n = *issued;
      for (int tt = n > S ? n - S : 0; tt < n; ++tt) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(&full[tt % S], (tt / S) & 1u))
          if (ptx::globaltimer_ns() - t0 > 50ull * 1000ull * 1000ull) break;
      }
    }
    return;
  }
  // ---- each warp hands its state to the merge (the ring is idle now)
  float* mst = reinterpret_cast<float*>(sm + L::OFF_MST);
  float* mo = reinterpret_cast<float*>(sm + L::OFF_MO);
  if (tq == 0) {
    mst[(warp * kDwRows + g) * 2] = mrow;
    mst[(warp * kDwRows + g) * 2 + 1] = lrow;
  }
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt)
    *reinterpret_cast<float2*>(mo + (warp * kDwRows + g) * D + 8 * dt + 2 * tq) = make_float2(o[dt][0], o[dt][1]);
  __syncthreads();
  // ---- merge the warps: row max over the warps, weights 2^(m_w - m); then
  // the partial (or, with one split, final) results as in the kernel above
  constexpr int CP = D / 2;
  for (int e = tid; e < M * CP; e += kDwThreads) {
    const int m = e / CP, c2 = e % CP;
    float mrow = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kDwWarps; ++w) mrow = fmaxf(mrow, mst[(w * kDwRows + m) * 2]);
    const float ms = mrow == -CUDART_INF_F ? 0.f : mrow;
    float lsum = 0.f;
    float2 o = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kDwWarps; ++w) {
      const float mw_ = mst[(w * kDwRows + m) * 2];
      const float wt = mw_ == -CUDART_INF_F ? 0.f : ptx::ex2(mw_ - ms);
      lsum = fmaf(wt, mst[(w * kDwRows + m) * 2 + 1], lsum);
      const float2 ow = *reinterpret_cast<const float2*>(mo + (w * kDwRows + m) * D + 2 * c2);
      o = make_float2(fmaf(wt, ow.x, o.x), fmaf(wt, ow.y, o.y));
    }
    const int h = hkv * G + m / p.Lq, i = m % p.Lq;
    const int64_t row = (static_cast<int64_t>(b) * p.Hq + h) * p.Lq + i;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const float lse2 = lsum > 0.f ? ms + __log2f(lsum) : -CUDART_INF_F;
    if (p.n_split == 1) {
      reinterpret_cast<__nv_bfloat162*>(p.out)[row * CP + c2] = __floats2bfloat162_rn(o.x * inv, o.y * inv);
      if (c2 == 0 && p.lse) p.lse[row] = lse2 * kDLn2;
    } else {
      const int64_t prow = static_cast<int64_t>(split) * p.rows + row;
      reinterpret_cast<float2*>(p.opart)[prow * CP + c2] = make_float2(o.x * inv, o.y * inv);
      if (c2 == 0) p.lpart[prow] = lse2;
    }
  }
}

// Merge of the splits: one warp per query row.
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const __grid_constant__ DecodeParams p) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.rows) return;
  float L = -CUDART_INF_F;
  for (int s = 0; s < p.n_split; ++s) L = fmaxf(L, p.lpart[static_cast<int64_t>(s) * p.rows + row]);
  const float Ls = L == -CUDART_INF_F ? 0.f : L;
  constexpr int PER = D / 32;  // channels per lane
  float o[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) o[c] = 0.f;
  float wsum = 0.f;
  for (int s = 0; s < p.n_split; ++s) {
    const int64_t prow = static_cast<int64_t>(s) * p.rows + row;
    const float ls = p.lpart[prow];
    const float w = ls == -CUDART_INF_F ? 0.f : exp2f(ls - Ls);
    wsum += w;
    const float* op = p.opart + prow * D + lane * PER;
#pragma unroll
    for (int c = 0; c < PER; ++c) o[c] = fmaf(w, op[c], o[c]);
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + row * D + lane * PER;
#pragma unroll
  for (int c = 0; c < PER; c += 2)
    *reinterpret_cast<__nv_bfloat162*>(orow + c) = __floats2bfloat162_rn(o[c] * inv, o[c + 1] * inv);
  if (lane == 0 && p.lse) p.lse[row] = wsum > 0.f ? (Ls + __log2f(wsum)) * kDLn2 : -CUDART_INF_F;
}

template <int D, int MR>
cudaError_t launch_decode_dm(const CUtensorMap* maps, const DecodeParams& p, cudaStream_t stream) {
  const int smem = DecLayout<D>::smem_bytes(p.Hq / p.Hkv * p.Lq);
  static const cudaError_t attr = cudaFuncSetAttribute(decode_split_kernel<D, MR>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       DecLayout<D>::smem_bytes(MR));
  if (attr != cudaSuccess) return attr;
  const int grid = p.B * p.Hkv * p.n_split;
  decode_split_kernel<D, MR><<<grid, kDecThreads, smem, stream>>>(maps[0], maps[1], p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split == 1) return e;
  const int mgrid = static_cast<int>((p.rows + 7) / 8);
  decode_merge_kernel<D><<<mgrid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_warp(const CUtensorMap* maps, const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = DwLayout<D>::SMEM;
  static const cudaError_t attr =
      cudaFuncSetAttribute(decode_warp_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  const int grid = p.B * p.Hkv * p.n_split;
  decode_warp_kernel<D><<<grid, kDwThreads, smem, stream>>>(maps[0], maps[1], p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split == 1) return e;
  const int mgrid = static_cast<int>((p.rows + 7) / 8);
  decode_merge_kernel<D><<<mgrid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const CUtensorMap* maps, const DecodeParams& p, cudaStream_t stream) {
  const int M = p.Hq / p.Hkv * p.Lq;
  if (M <= kDwRows) return launch_decode_warp<D>(maps, p, stream);
  if (M <= 16) return launch_decode_dm<D, 16>(maps, p, stream);
  if (M <= 32) return launch_decode_dm<D, 32>(maps, p, stream);
  return launch_decode_dm<D, 64>(maps, p, stream);
}

}  // namespace

cudaError_t launch_decode(int d, const CUtensorMap* maps, const DecodeParams& p, cudaStream_t stream) {
  return d == 64 ? launch_decode_d<64>(maps, p, stream) : launch_decode_d<128>(maps, p, stream);
}

}  // namespace fl
