// Backward pass of the fused attention (dQ, dK, dV) for sm_103a.
//
// The derivative of softmax(score_mod(scale QK^T) + mask) V, recomputing P
// from the forward's log-sum-exp instead of storing it (the same recompute
// the fused forward's single pass makes possible; the Flashlight wiki
// summary lists the training backward as future work, 局限与 Future Work):
//
//   P^T  = exp(T^T - LSE)          dV += P^T dO
//   dP^T = V dO^T                  dS^T = P^T * (dP^T - D) * dT/dS
//   dK  += dS^T Q                  dQ  += dS K        (D = rowsum(dO * O))
//
// One CTA owns one (batch, key/value head, 128-key tile) and walks every
// query tile of every query head of its GQA group that sees those keys;
// dK and dV stay in TMEM for the whole walk, and each query tile's dQ
// contribution is added to an fp32 accumulator in global memory.  All five
// products run on tcgen05 with accumulators in TMEM:
//   S^T  = K Q^T   (A = K, B = Q smem)              TMEM [0,128)
//   P^T  (bf16, written by the compute warps)        over S^T: [0,32), [64,96)
//   dP^T = V dO^T  (A = V smem, B = dO smem)        TMEM [192,320)
//   dS^T (bf16; queries 0-63 over dP^T's [192,224), 64-127 over [256,288))
//   dV  += P^T dO  (A = P^T TMEM, B = dO smem)      TMEM [320,320+D)
//   dK  += dS^T Q  (A = dS^T TMEM, B = Q smem)      TMEM [320+D,320+2D)
//   dQ   = dS K    (A = dS smem, M-major; B = K)    TMEM [320+2D,320+3D)
// P^T goes over the first half of each half-tile's S^T columns, so that
// TMEM [128,192) holds either K and V (constant over the walk; the A
// operands of S^T and dP^T, which then read only Q and dO from shared
// memory, whose bandwidth the products contend for) or, with softcap,
// sech^2 of the tile's scores as fp16 pairs for the dS step.  With d = 128,
// dV and dK take 256 columns: dP^T moves to [128,256) and dQ shares those
// columns (dP^T of the next tile waits until the dQ warps have read dQ),
// sech^2 goes over the second half of each half-tile's S^T columns, and K, V
// stay in shared memory, as does one dO buffer (two do not fit beside the
// rest).  With d = 64 and dv = 128 (the branches of differential
// attention) dP^T is at [128,256), dV [256,384), dK [384,448), dQ
// [448,512), sech^2 as at d = 128.  The gradients may be those of a scaled
// output gradient (dout_scale, applied to dP, D and dV), and dV may be added
// to what dv holds: the differential backward's second branch takes
// -lambda dout and adds its dV to the first branch's.
// Warp roles (512 threads): warp 0 TMA, warp 1 TMEM + MMA issue, warps 4-11
// compute P and dS (one thread per key row and half of the query columns:
// two warps per scheduler), warps 12-15 add dQ into the accumulator (one
// thread per query row): they stage the fp32 tile in shared memory and one
// thread adds it to global memory with a TMA bulk reduction.  Every wait is
// bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>
#include <type_traits>

#include "bwd.h"
#include "fused_attn.cuh"

namespace fl {
namespace {

constexpr int kBwdThreads = 512;

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}
// registers: 128 per thread at launch, then 56 (TMA / MMA warps), 168 (P and
// dS), 120 (dQ) -- together exactly the launch's 512 x 128
constexpr int kBwdLaunchRegs = 128, kBwdCtlRegs = 56, kBwdComputeRegs = 168, kBwdDQRegs = 120;
static_assert(128 * kBwdCtlRegs + 256 * kBwdComputeRegs + 128 * kBwdDQRegs <= kBwdThreads * kBwdLaunchRegs,
              "backward register split");

template <int D, int DV>
struct BwdLayout {
  static_assert((D == DV && (D == 32 || D == 64 || D == 128)) || (D == 64 && DV == 128), "backward head dims");
  static constexpr int ROWB = D * 2;
  // Q and K: D channels; V and dO: DV channels; each in boxes of at most 64
  // channels (128-byte rows)
  static constexpr int BOXW = D < 64 ? D : 64;
  static constexpr int NBOX = D / BOXW;
  static constexpr int BOXB = BOXW * 2;                // bytes per row of one box
  static constexpr int BOX = 128 * BOXB;               // one box of 128 rows
  static constexpr int TILE = NBOX * BOX;              // one 128-row tile of K or Q
  static constexpr uint32_t SWZ = BOXB == 128 ? 2u : 4u;
  static constexpr int BOXW_V = DV < 64 ? DV : 64;
  static constexpr int NBOX_V = DV / BOXW_V;
  static constexpr int BOXB_V = BOXW_V * 2;
  static constexpr int BOX_V = 128 * BOXB_V;
  static constexpr int TILE_V = NBOX_V * BOX_V;        // one 128-row tile of V or dO
  static constexpr uint32_t SWZ_V = BOXB_V == 128 ? 2u : 4u;
  // d = 128: one dO buffer and one 32-channel dQ staging box; two of each
  // would not fit in a block's 227 KB
  static constexpr int NDO = D == 128 ? 1 : 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = TILE + TILE_V;          // Q[2]
  static constexpr int OFF_DO = OFF_Q + 2 * TILE;      // dO[NDO]
  static constexpr int OFF_DS = OFF_DO + NDO * TILE_V; // dS tile: 2 boxes [128 keys][64 queries], 128B swizzle
  static constexpr int DQS = D == 128 ? 128 * 32 * 4 : 128 * D * 4;  // fp32 boxes [128 rows][32], 128B swizzle
  static constexpr int OFF_DQS = OFF_DS + 2 * 128 * 128;  // dQ staging (the previous tile's reduction
                                                          // has a whole tile period to read it out)
  static constexpr int OFF_VEC = OFF_DQS + DQS;        // fp32 L2[2][128], Dv[2][128]
  static constexpr int OFF_BAR = OFF_VEC + 4 * 128 * 4;
  static constexpr int NBARS = 16;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  static_assert(SMEM <= 227 * 1024, "backward shared memory");
  static_assert(OFF_Q % 1024 == 0 && OFF_DO % 1024 == 0 && OFF_DS % 1024 == 0 && OFF_DQS % 1024 == 0,
                "swizzled tiles on 1024-byte boundaries");
  // k-step kb (16 channels) of a K-major Q / K tile: box kb * 16 / BOXW, 32
  // bytes per step within the box's 128-byte swizzled rows (descriptor
  // units of 16 B); koff_v likewise for V / dO
  __host__ __device__ static constexpr uint32_t koff(int kb) {
    return ((kb * 16 / BOXW) * BOX + (kb * 16 % BOXW) * 2) >> 4;
  }
  __host__ __device__ static constexpr uint32_t koff_v(int kb) {
    return ((kb * 16 / BOXW_V) * BOX_V + (kb * 16 % BOXW_V) * 2) >> 4;
  }
};

// Queries that see key k form one interval [qlo, qhi] for every mask kind
// (the mirror of row_bounds: the visible-key intervals of the rows are
// non-decreasing in the row).
__device__ __forceinline__ void col_bounds(const BwdParams& p, int b, int k, int& qlo, int& qhi) {
  qlo = 0;
  qhi = p.Lq - 1;
  switch (p.mask_kind) {
    case MASK_NONE: break;
    case MASK_CAUSAL: qlo = k; break;
    case MASK_WINDOW: qlo = k; qhi = k + p.window - 1; break;
    case MASK_PREFIX: qlo = k < p.prefix ? 0 : k; break;
    default: {
      const int32_t* off = p.doc_offsets + static_cast<int64_t>(b) * (p.num_docs + 1);
      int a = 0, z = p.num_docs - 1;
      while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (__ldg(off + mid) <= k) a = mid; else z = mid - 1;
      }
      qlo = __ldg(off + a);
      qhi = __ldg(off + a + 1) - 1;
      if (p.doc_causal) qlo = k > qlo ? k : qlo;
    }
  }
  qhi = qhi > p.Lq - 1 ? p.Lq - 1 : qhi;
}

template <int D, int DV, int SCORE>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmL2, const __grid_constant__ CUtensorMap tmDv,
                    const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ BwdParams p) {
  using L = BwdLayout<D, DV>;
  // d = dv <= 64: S^T [0,128), K V or sech^2 [128,192), dP^T [192,320), dV,
  // dK, dQ after.  d = 128 (dV and dK take 256 columns): S^T [0,128), dP^T
  // [128,256) shared with dQ, dV [256,384), dK [384,512).  d = 64 with dv =
  // 128: S^T [0,128), dP^T [128,256), dV [256,384), dK [384,448), dQ
  // [448,512).  In the last two maps softcap's sech^2 goes over the second
  // half of each half-tile's S^T columns (P^T holds the first).
  constexpr bool kWide = D == 128;
  constexpr bool kSechInS = D == 128 || DV != D;
  constexpr uint32_t kColS = 0, kColDP = kSechInS ? 128 : 192, kColDV = kSechInS ? 256 : 320;
  constexpr uint32_t kColDK = kColDV + DV, kColDQ = kWide ? kColDP : kColDK + D;
  static_assert(kColDK + D <= 512 && kColDQ + D <= 512, "backward TMEM map");
  // TMEM [128,192) (d = dv <= 64): K and V without softcap, the tile's sech^2 with it
  constexpr bool kKVT = SCORE != SCORE_SOFTCAP && !kSechInS;
  constexpr uint32_t kColKT = 128, kColVT = 128 + D / 2;
  // softcap: sech^2, fp16 pairs, 32 columns per half
  constexpr uint32_t kColSech = kSechInS ? 32 : 128, kSechHalf = kSechInS ? 64 : 32;
  // sech^2 in the S^T columns: the next S^T waits for the dS step
  constexpr bool kLateS = kSechInS && SCORE == SCORE_SOFTCAP;
  extern __shared__ uint8_t bsm_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(bsm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;    // [2]
  uint64_t* q_empty = bars + 3;   // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* dp_full = bars + 6;
  uint64_t* p_full = bars + 7;
  uint64_t* ds_full = bars + 8;
  uint64_t* dq_full = bars + 9;
  uint64_t* dq_free = bars + 10;
  uint64_t* done = bars + 11;
  uint64_t* kvt_ready = bars + 12;  // K and V copied into TMEM
  uint64_t* do_full = bars + 13;    // d = 128: the single dO buffer loaded ...
  uint64_t* do_empty = bars + 14;   // ... and read by dV
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  float* vec = reinterpret_cast<float*>(smem + L::OFF_VEC);  // L2[buf][128] then Dv[buf][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA: (batch b, key/value head hkv, key tile jt), key tiles in the
  // outer order so that the first tiles of every head (the longest walks
  // under causal and prefix masks) start first and the short ones end the grid
  const int jt = blockIdx.x / (p.B * p.Hkv);
  const int bh = blockIdx.x % (p.B * p.Hkv);
  const int hkv = bh % p.Hkv, b = bh / p.Hkv;
  const int j0 = jt * 128;
  const int group = p.Hq / p.Hkv;
  // query tiles that see any key of the tile (intervals are monotone in k)
  int qlo0, qhi0, qlo1, qhi1;
  col_bounds(p, b, j0, qlo0, qhi0);
  col_bounds(p, b, min(j0 + 127, p.Lk - 1), qlo1, qhi1);
  const int it_lo = qlo0 / 128;
  const int it_hi = qhi1 >= qlo0 ? qhi1 / 128 : it_lo - 1;
  const int nq = it_hi - it_lo + 1;
  const int n_tiles = nq > 0 ? nq * group : 0;

  if (threadIdx.x == 0) {
    ptx::mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&q_full[i], 1);
      ptx::mbar_init(&q_empty[i], 1);
    }
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(dp_full, 1);
    ptx::mbar_init(p_full, 8);
    ptx::mbar_init(ds_full, 8);
    ptx::mbar_init(dq_full, 1);
    ptx::mbar_init(dq_free, 4);
    ptx::mbar_init(done, 1);
    ptx::mbar_init(kvt_ready, 8);
    ptx::mbar_init(do_full, 1);
    ptx::mbar_init(do_empty, 1);
    misc[1] = 0u;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&misc[0], 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const Ctl ctl{reinterpret_cast<volatile uint32_t*>(&misc[1]), p.status, p.timeout_ns};
  const uint64_t drain_ns = 50ull * 1000ull * 1000ull;

  if (warp < 4) {
    ptx::setmaxnreg_dec<kBwdCtlRegs>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- TMA
      const uint64_t pol_keep = ptx::policy_evict_last();
      if (n_tiles > 0) {
        ptx::mbar_arrive_expect_tx(kv_full, static_cast<uint32_t>(L::TILE + L::TILE_V));
#pragma unroll
        for (int bx = 0; bx < L::NBOX; ++bx)
          ptx::tma_load_4d(smem + L::OFF_K + bx * L::BOX, &tmK, kv_full, bx * L::BOXW, j0, hkv, b, pol_keep);
#pragma unroll
        for (int bx = 0; bx < L::NBOX_V; ++bx)
          ptx::tma_load_4d(smem + L::OFF_V + bx * L::BOX_V, &tmV, kv_full, bx * L::BOXW_V, j0, hkv, b, pol_keep);
      }
      int issued = 0, do_issued = 0;
      bool ok = true;
      for (int n = 0; n < n_tiles && ok; ++n) {
        const int h = hkv * group + n / nq, i0 = (it_lo + n % nq) * 128;
        const int buf = n & 1;
        if (!wait_bar(&q_empty[buf], ((n >> 1) & 1u) ^ 1u, ctl, 50)) { ok = false; break; }
        ptx::mbar_arrive_expect_tx(&q_full[buf],
                                   static_cast<uint32_t>(L::TILE + (L::NDO == 2 ? L::TILE_V : 0)) + 2u * 512u);
#pragma unroll
        for (int bx = 0; bx < L::NBOX; ++bx)
          ptx::tma_load_4d(smem + L::OFF_Q + buf * L::TILE + bx * L::BOX, &tmQ, &q_full[buf], bx * L::BOXW, i0, h, b,
                           pol_keep);
        if (L::NDO == 2) {
#pragma unroll
          for (int bx = 0; bx < L::NBOX_V; ++bx)
            ptx::tma_load_4d(smem + L::OFF_DO + buf * L::TILE_V + bx * L::BOX_V, &tmDO, &q_full[buf], bx * L::BOXW_V,
                             i0, h, b, pol_keep);
        }
        const int row = b * p.Hq + h;
        ptx::tma_load_2d(vec + buf * 128, &tmL2, &q_full[buf], i0, row, pol_keep);
        ptx::tma_load_2d(vec + 256 + buf * 128, &tmDv, &q_full[buf], i0, row, pol_keep);
        issued = n + 1;
        if (L::NDO == 1) {
          // one dO buffer: tile n's once dV(n - 1) has read tile n - 1's
          if (!wait_bar(do_empty, (n & 1u) ^ 1u, ctl, 56)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(do_full, L::TILE_V);
#pragma unroll
          for (int bx = 0; bx < L::NBOX_V; ++bx)
            ptx::tma_load_4d(smem + L::OFF_DO + bx * L::BOX_V, &tmDO, do_full, bx * L::BOXW_V, i0, h, b, pol_keep);
          do_issued = n + 1;
        }
      }
      if (*ctl.abort) {
        if (n_tiles > 0) wait_drain(kv_full, 0u, drain_ns);
        for (int n = issued - 2 < 0 ? 0 : issued - 2; n < issued; ++n) wait_drain(&q_full[n & 1], (n >> 1) & 1u, drain_ns);
        if (do_issued > 0) wait_drain(do_full, (do_issued - 1) & 1u, drain_ns);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------------- MMA
      constexpr uint32_t ID_SS = ptx::idesc_bf16_f32(128, 128, false);        // S^T, dP^T
      constexpr uint32_t ID_DV = ptx::idesc_bf16_f32(128, DV, true);         // dV (B = dO, N-major)
      constexpr uint32_t ID_DK = ptx::idesc_bf16_f32(128, D, true);          // dK (B = Q, N-major)
      constexpr uint32_t ID_DQ = ptx::idesc_bf16_f32(128, D, true) | (1u << 15);  // dQ: A = dS, M-major
      const uint32_t k_a = ptx::smem_u32(smem + L::OFF_K), v_a = ptx::smem_u32(smem + L::OFF_V);
      const uint32_t ds_a = ptx::smem_u32(smem + L::OFF_DS);
      const uint64_t dsa = ptx::smem_desc(ds_a, 128 * 128, 1024, 2u);
      // N-major B operands (N = D channels across NBOX boxes, LBO = box
      // stride) and K-major operands (k-steps through ::koff)
      const uint64_t kn = ptx::smem_desc(k_a, L::BOX, 8 * L::BOXB, L::SWZ);
      const uint64_t ka = ptx::smem_desc(k_a, 16, 8 * L::BOXB, L::SWZ);
      const uint64_t va = ptx::smem_desc(v_a, 16, 8 * L::BOXB_V, L::SWZ_V);
      // S^T = K Q^T and dP^T = V dO^T of query tile n (K-major, k-steps of 16
      // channels), each once its Q / dO tile has landed
      auto issue_s = [&](int n) -> bool {
        const int buf = n & 1;
        if (!wait_bar(&q_full[buf], (n >> 1) & 1u, ctl, 52)) return false;
        ptx::tc_fence_after();
        const uint64_t qb = ptx::smem_desc(ptx::smem_u32(smem + L::OFF_Q + buf * L::TILE), 16, 8 * L::BOXB, L::SWZ);
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb) {
          if (kKVT) ptx::mma_ts(tmem + kColS, tmem + kColKT + kb * 8, qb + L::koff(kb), ID_SS, kb > 0);
          else ptx::mma_ss(tmem + kColS, ka + L::koff(kb), qb + L::koff(kb), ID_SS, kb > 0);
        }
        ptx::mma_commit(s_full);
        return true;
      };
      auto issue_dp = [&](int n) -> bool {
        if (L::NDO == 1) {
          if (!wait_bar(do_full, n & 1u, ctl, 57)) return false;
          ptx::tc_fence_after();
        }
        const uint64_t dob = ptx::smem_desc(
            ptx::smem_u32(smem + L::OFF_DO + (L::NDO == 2 ? (n & 1) : 0) * L::TILE_V), 16, 8 * L::BOXB_V, L::SWZ_V);
#pragma unroll
        for (int kb = 0; kb < DV / 16; ++kb) {
          if (kKVT) ptx::mma_ts(tmem + kColDP, tmem + kColVT + kb * 8, dob + L::koff_v(kb), ID_SS, kb > 0);
          else ptx::mma_ss(tmem + kColDP, va + L::koff_v(kb), dob + L::koff_v(kb), ID_SS, kb > 0);
        }
        ptx::mma_commit(dp_full);
        return true;
      };
      // The products of tile n + 1 are issued as soon as the compute warps
      // are done with the TMEM they overwrite, so that the next P and dS find
      // them ready: S^T(n+1) right after dV(n) (d = 128 softcap: after the dS
      // step, which reads sech^2 from the S^T columns), dP^T(n+1) right after
      // dK(n) (d = 128: once the dQ warps have read dQ(n) from the same
      // columns).  One thread's MMAs run in issue order, so dV(n) has read P^T
      // (over the S^T columns) and dK(n) dS^T before the next products
      // overwrite those columns, and a commit covers every product issued
      // before it.
      bool ok = n_tiles == 0 ||
                (wait_bar(kv_full, 0u, ctl, 51) && (!kKVT || wait_bar(kvt_ready, 0u, ctl, 58)) && issue_s(0) &&
                 issue_dp(0));
      for (int n = 0; n < n_tiles && ok; ++n) {
        const int buf = n & 1;
        const uint32_t ph = n & 1;
        const bool more = n + 1 < n_tiles;
        const uint32_t q_a = ptx::smem_u32(smem + L::OFF_Q + buf * L::TILE);
        const uint32_t do_a = ptx::smem_u32(smem + L::OFF_DO + (L::NDO == 2 ? buf : 0) * L::TILE_V);
        // dV += P^T dO (B = dO as [queries][D], N contiguous)
        if (!wait_bar(p_full, ph, ctl, 53)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t don = ptx::smem_desc(do_a, L::BOX_V, 8 * L::BOXB_V, L::SWZ_V);
#pragma unroll
        for (int kb = 0; kb < 8; ++kb)
          ptx::mma_ts(tmem + kColDV, tmem + kColS + kb * 8 + (kb >= 4 ? 32 : 0), don + ((kb * 16 * L::BOXB_V) >> 4),
                      ID_DV, (n > 0 || kb > 0));
        if (L::NDO == 1) ptx::mma_commit(do_empty);
        if (!kLateS && more && !issue_s(n + 1)) { ok = false; break; }
        // dK += dS^T Q (dS^T of queries 64-127 sits 64 columns further on)
        if (!wait_bar(ds_full, ph, ctl, 54)) { ok = false; break; }
        ptx::tc_fence_after();
        if (kLateS && more && !issue_s(n + 1)) { ok = false; break; }
        const uint64_t qn = ptx::smem_desc(q_a, L::BOX, 8 * L::BOXB, L::SWZ);
#pragma unroll
        for (int kb = 0; kb < 8; ++kb)
          ptx::mma_ts(tmem + kColDK, tmem + kColDP + kb * 8 + (kb >= 4 ? 32 : 0), qn + ((kb * 16 * L::BOXB) >> 4),
                      ID_DK, (n > 0 || kb > 0));
        if (!kWide && more) issue_dp(n + 1);
        // dQ = dS K once the dQ warps have read the previous one
        if (!wait_bar(dq_free, ph ^ 1u, ctl, 55)) { ok = false; break; }
        ptx::tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 8; ++kb)
          ptx::mma_ss(tmem + kColDQ, dsa + ((kb * 16 * 128) >> 4), kn + ((kb * 16 * L::BOXB) >> 4), ID_DQ, kb > 0);
        ptx::mma_commit(dq_full);
        ptx::mma_commit(&q_empty[buf]);
        if (kWide && more) {
          if (!wait_bar(dq_free, ph, ctl, 59)) { ok = false; break; }
          ptx::tc_fence_after();
          if (!issue_dp(n + 1)) { ok = false; break; }
        }
      }
      ptx::mma_commit(done);
      wait_drain(done, 0u, drain_ns);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc(tmem, 512);
    }
  } else if (warp < 12) {
    // ---------------------------------------- P and dS (key rows, half tiles)
    // Thread (quad, lane) of half hf owns key row r and the query columns
    // [64 hf, 64 hf + 64) of every query tile: its S^T, P^T and dP^T columns.
    ptx::setmaxnreg_inc<kBwdComputeRegs>();
    const int quad = warp & 3;
    const int hf = (warp - 4) >> 2;
    const int r = quad * 32 + lane;          // key row of the tile
    const int kg = j0 + r;                   // key index
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t cS = kColS + 64 * hf;     // S^T
    const uint32_t cP = cS;                  // P^T, bf16 pairs, over the S^T just read
    const uint32_t cSech = kColSech + kSechHalf * hf;  // softcap: sech^2, fp16 pairs
    const uint32_t cDP = kColDP + 64 * hf;   // dP^T; dS^T as bf16 pairs over its first 32 columns
    int cqlo, cqhi;
    col_bounds(p, b, kg < p.Lk ? kg : p.Lk - 1, cqlo, cqhi);
    if (kg >= p.Lk) { cqlo = 1; cqhi = 0; }  // keys past the end see nothing
    const float scale_log2 = p.scale * kLog2e;
    const float2 sc2 = make_float2(scale_log2, scale_log2);
    const float kcap = p.softcap * kLog2e;
    const float zmul = SCORE == SCORE_SOFTCAP ? 2.0f * scale_log2 / p.softcap : 0.f;
    const float2 sq0 = make_float2(p.sc_q[0], p.sc_q[0]), sq1 = make_float2(p.sc_q[1], p.sc_q[1]);
    const float2 sq2 = make_float2(p.sc_q[2], p.sc_q[2]), sq3 = make_float2(p.sc_q[3], p.sc_q[3]);
    const float ikc = SCORE == SCORE_SOFTCAP ? 1.0f / kcap : 0.f;
    const float gsc = p.dout_scale;  // dP of the scaled dO (D comes scaled from the pre-kernel)
    const float2 ikc2 = make_float2(ikc, ikc);
    bool ok = true;
    if constexpr (kKVT) if (n_tiles > 0) {
      // this thread's key row of K (half 0) or V (half 1) into TMEM: 16-byte
      // chunk c of row r sits at c ^ (r & 7) (128-byte rows) or
      // c ^ ((r >> 1) & 3) (64-byte rows) of the swizzled tile
      ok = __all_sync(0xffffffffu, wait_bar(kv_full, 0u, ctl, 65));
      if (ok) {
        const uint8_t* row = smem + (hf ? L::OFF_V : L::OFF_K) + r * L::ROWB;
        uint32_t kv[D / 2];
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const int sc = L::ROWB == 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
          const uint4 v4 = *reinterpret_cast<const uint4*>(row + (sc << 4));
          kv[4 * c] = v4.x; kv[4 * c + 1] = v4.y; kv[4 * c + 2] = v4.z; kv[4 * c + 3] = v4.w;
        }
        const uint32_t ta = tl + (hf ? kColVT : kColKT);
        if constexpr (D == 64) ptx::tmem_st32(ta, kv);
        else ptx::tmem_st16(ta, kv);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(kvt_ready);
      }
    }
    for (int n = 0; n < n_tiles && ok; ++n) {
      const int h = hkv * group + n / nq, i0 = (it_lo + n % nq) * 128;
      const int q0 = i0 + 64 * hf;           // first query column of this half
      const int buf = n & 1;
      const uint32_t ph = n & 1;
      const float* l2 = vec + buf * 128 + 64 * hf;
      const float* dvec = vec + 256 + buf * 128 + 64 * hf;
      if (!__all_sync(0xffffffffu, wait_bar(s_full, ph, ctl, 60))) { ok = false; break; }
      // this tile's LSE and D rows came with Q (TMA); observe that barrier too
      if (!__all_sync(0xffffffffu, wait_bar(&q_full[buf], (n >> 1) & 1u, ctl, 64))) { ok = false; break; }
      ptx::tc_fence_after();
      float x[64];
      ptx::tmem_ld32f(tl + cS, &x[0]);
      ptx::tmem_ld32f(tl + cS + 32, &x[32]);
      ptx::tmem_ld_wait();
      ptx::reg_fence32f(&x[0]);
      ptx::reg_fence32f(&x[32]);
      const float slope2 = SCORE == SCORE_ALIBI ? __ldg(p.slopes + h) * kLog2e : 0.f;
      // ALiBi: slope2 (k - q) = abase - slope2 c for query q0 + c
      const float abase = slope2 * static_cast<float>(kg - q0);
      // the warp's rows all see all 64 columns (no per-element test), or some
      const bool all_vis = __all_sync(0xffffffffu, cqlo <= q0 && cqhi >= q0 + 63);
      const bool any_vis = __any_sync(0xffffffffu, cqlo <= q0 + 63 && cqhi >= q0);
      // P^T = 2^(t log2 e - L2_q) on visible (key, query) pairs; softcap also
      // leaves sech^2 of the scaled score over cap (fp16 pairs, cSech) for
      // the dS step, which the next tile's P step of these same warps
      // overwrites only afterwards.  When all of the warp's scores are in
      // the polynomial's range, tanh comes from the forward's FMA-pipe
      // polynomial (t = s q(s^2) = cap log2(e) tanh, sech^2 = 1 - tanh^2);
      // otherwise from d = 1 / (1 + e^(2 s / cap)): tanh = 1 - 2d,
      // sech^2 = 4 d (1 - d) (two MUFU operations more per score).
      bool poly = false;
      if (SCORE == SCORE_SOFTCAP) {
        float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 64; ++c) am[c & 3] = fmaxf(am[c & 3], fabsf(x[c]));
        poly = __all_sync(0xffffffffu, fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3])) <= p.sc_smax);
      }
      auto p_chunk = [&](int c0, auto full) {
        uint32_t sech[16];  // fp16 pairs
        if (SCORE == SCORE_SOFTCAP) {
          // t = cap log2(e) tanh(s scale / cap) in place, and sech^2 (one
          // form per chunk: the branch stays outside the loops)
          if (poly) {
#pragma unroll
            for (int e2 = 0; e2 < 32; e2 += 2) {
              const float2 xv = make_float2(x[c0 + e2], x[c0 + e2 + 1]);
              const float2 z = ptx::mul2(xv, xv);
              float2 q = ptx::fma2(sq3, z, sq2);
              q = ptx::fma2(q, z, sq1);
              q = ptx::fma2(q, z, sq0);
              const float2 t = ptx::mul2(xv, q);
              const float2 th = ptx::mul2(t, ikc2);
              const float2 sc = ptx::fma2(make_float2(-th.x, -th.y), th, make_float2(1.0f, 1.0f));
              x[c0 + e2] = t.x;
              x[c0 + e2 + 1] = t.y;
              sech[e2 >> 1] = pack_f16x2(sc.x, sc.y);
            }
          } else {
#pragma unroll
            for (int e2 = 0; e2 < 32; e2 += 2) {
              const float d0 = ptx::rcp(1.0f + ptx::ex2(x[c0 + e2] * zmul));
              const float d1 = ptx::rcp(1.0f + ptx::ex2(x[c0 + e2 + 1] * zmul));
              x[c0 + e2] = fmaf(-2.0f * kcap, d0, kcap);
              x[c0 + e2 + 1] = fmaf(-2.0f * kcap, d1, kcap);
              sech[e2 >> 1] = pack_f16x2(4.0f * d0 * (1.0f - d0), 4.0f * d1 * (1.0f - d1));
            }
          }
        }
#pragma unroll
        for (int c4 = 0; c4 < 32; c4 += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(l2 + c0 + c4);
#pragma unroll
          for (int e2 = 0; e2 < 4; e2 += 2) {
            const int c = c0 + c4 + e2;
            const float2 lq = e2 == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
            const float2 xv = make_float2(x[c], x[c + 1]);
            float2 arg;  // t log2 e - L2_q of the pair
            if (SCORE == SCORE_SOFTCAP) {
              arg = ptx::sub2(xv, lq);  // x holds t already
            } else if (SCORE == SCORE_ALIBI) {
              arg = ptx::fma2(xv, sc2,
                              make_float2(fmaf(-slope2, static_cast<float>(c), abase) - lq.x,
                                          fmaf(-slope2, static_cast<float>(c + 1), abase) - lq.y));
            } else {
              arg = ptx::fma2(xv, sc2, make_float2(-lq.x, -lq.y));
            }
            const float2 pv = make_float2(ptx::ex2(arg.x), ptx::ex2(arg.y));
            if (decltype(full)::value) {
              x[c] = pv.x;
              x[c + 1] = pv.y;
            } else {
              const int q = q0 + c;
              x[c] = any_vis && q >= cqlo && q <= cqhi ? pv.x : 0.f;
              x[c + 1] = any_vis && q + 1 >= cqlo && q + 1 <= cqhi ? pv.y : 0.f;
            }
          }
        }
        if (SCORE == SCORE_SOFTCAP) ptx::tmem_st16(tl + cSech + c0 / 2, sech);
      };
      if (all_vis) {
        p_chunk(0, std::true_type{});
        p_chunk(32, std::true_type{});
      } else {
        p_chunk(0, std::false_type{});
        p_chunk(32, std::false_type{});
      }
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = ptx::pack_bf16x2(x[c + 2 * e], x[c + 2 * e + 1]);
        ptx::tmem_st16(tl + cP + c / 2, pk);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(p_full);
      // dS^T = P^T (dP^T - D_q) (* sech^2 for softcap)
      if (!__all_sync(0xffffffffu, wait_bar(dp_full, ph, ctl, 61))) { ok = false; break; }
      // the previous dQ product must have read the dS tile in shared memory
      if (n > 0 && !__all_sync(0xffffffffu, wait_bar(dq_full, ph ^ 1u, ctl, 62))) { ok = false; break; }
      ptx::tc_fence_after();
      float dpv[64];
      ptx::tmem_ld32f(tl + cDP, &dpv[0]);
      if (SCORE != SCORE_SOFTCAP) ptx::tmem_ld32f(tl + cDP + 32, &dpv[32]);
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t sv[16];  // sech^2, fp16 pairs
        if (SCORE == SCORE_SOFTCAP) {
          if (c > 0) ptx::tmem_ld32f(tl + cDP + c, &dpv[c]);
          ptx::tmem_ld16(tl + cSech + c / 2, sv);
          ptx::tmem_ld_wait();
          ptx::reg_fence16(sv);
          ptx::reg_fence32f(&dpv[c]);
        } else if (c == 0) {
          ptx::tmem_ld_wait();
          ptx::reg_fence32f(&dpv[0]);
          ptx::reg_fence32f(&dpv[32]);
        }
        uint32_t pk[16];
#pragma unroll
        for (int e4 = 0; e4 < 32; e4 += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(dvec + c + e4);
          const float dq4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            float d0 = x[c + e4 + e] * fmaf(dpv[c + e4 + e], gsc, -dq4[e]);
            float d1 = x[c + e4 + e + 1] * fmaf(dpv[c + e4 + e + 1], gsc, -dq4[e + 1]);
            if (SCORE == SCORE_SOFTCAP) {
              const float2 sc = unpack_f16x2(sv[(e4 + e) >> 1]);
              d0 *= sc.x;
              d1 *= sc.y;
            }
            pk[(e4 + e) / 2] = ptx::pack_bf16x2(d0, d1);
          }
        }
        // dS^T over the first half of this half's dP^T columns (already read) ...
        ptx::tmem_st16(tl + cDP + c / 2, pk);
        // ... and dS into shared memory: row r (key) of box hf ([128][64],
        // 16-byte chunks at the 128-byte swizzle positions)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int chunk = (c >> 3) + w;
          *reinterpret_cast<uint4*>(smem + L::OFF_DS + hf * 128 * 128 + r * 128 + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
        }
      }
      ptx::tmem_st_wait();
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ds_full);
    }
    // dV (half 0) or dK (half 1) of this thread's key row, once every product
    // is done (the TMEM loads are warp-wide; only the stores depend on the row)
    if (ok && __all_sync(0xffffffffu, wait_bar(done, 0u, ctl, 63))) {
      ptx::tc_fence_after();
      const bool z = n_tiles == 0;
      const int64_t row = (static_cast<int64_t>(b) * p.Hkv + hkv) * p.Lk + kg;
      // NC columns of TMEM from col, times f, as bf16 into base's row (plus
      // what is there with acc)
      auto write_row = [&](auto nc, uint32_t col, void* base, float f, bool acc) {
        constexpr int NC = decltype(nc)::value;
        constexpr int EC = NC < 64 ? NC : 64;  // columns per TMEM read-out
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + row * NC);
#pragma unroll
        for (int c0 = 0; c0 < NC; c0 += EC) {
          float a[EC];
#pragma unroll
          for (int c = 0; c < EC; c += 32) ptx::tmem_ld32f(tl + col + c0 + c, &a[c]);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < EC; c += 32) ptx::reg_fence32f(&a[c]);
          if (kg < p.Lk) {
#pragma unroll
            for (int c = 0; c < EC; c += 8) {
              float o[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] = z ? 0.f : a[c + e] * f;
              if (acc) {
                const uint4 prev = dst[(c0 + c) / 8];
                const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&prev);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 pf = __bfloat1622float2(p2[e]);
                  o[2 * e] += pf.x;
                  o[2 * e + 1] += pf.y;
                }
              }
              dst[(c0 + c) / 8] = make_uint4(ptx::pack_bf16x2(o[0], o[1]), ptx::pack_bf16x2(o[2], o[3]),
                                             ptx::pack_bf16x2(o[4], o[5]), ptx::pack_bf16x2(o[6], o[7]));
            }
          }
        }
      };
      if (hf) write_row(std::integral_constant<int, D>{}, kColDK, p.dk, n_tiles > 0 ? p.scale : 1.0f, false);
      else write_row(std::integral_constant<int, DV>{}, kColDV, p.dv, p.dout_scale, p.dv_accumulate != 0);
    }
    ptx::tc_fence_before();
    __syncthreads();
  } else {
    // ------------------------------------------- dQ accumulation (query rows)
    // Per tile: TMEM -> registers (then dQ's TMEM is free again), registers ->
    // the staging buffer (swizzled: row r's 16-byte chunk k at k ^ (r & 7)),
    // and one thread adds the staged tile to the fp32 accumulator with a bulk
    // tensor reduction (rows past Lq skipped by the map).  Whether to go on is
    // decided jointly by the four warps (barrier with an AND), so that every
    // warp takes the same named barriers.
    ptx::setmaxnreg_dec<kBwdDQRegs>();
    const int quad = warp & 3;
    const int r = quad * 32 + lane;          // query row of the tile
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const bool issuer = warp == 12 && lane == 0;
    constexpr uint32_t kBarDQ = 1, kDQThreads = 128;
    bool ok = true;
    for (int n = 0; n < n_tiles && ok; ++n) {
      const int h = hkv * group + n / nq, i0 = (it_lo + n % nq) * 128;
      const bool got = __all_sync(0xffffffffu, wait_bar(dq_full, n & 1u, ctl, 70));
      if (!ptx::named_bar_and(kBarDQ, kDQThreads, got)) { ok = false; break; }
      ptx::tc_fence_after();
      uint8_t* sb = smem + L::OFF_DQS;
      // the reduction that last read the staging buffer is done with it
      auto staging_free = [&]() {
        if (issuer) ptx::bulk_wait_group_read0();
        ptx::named_bar_sync(kBarDQ, kDQThreads);
      };
      // row r's 32 fp32 values into staging box sbx
      auto store_box = [&](const float* a, int sbx) {
        uint8_t* box = sb + sbx * (128 * 128);
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<float4*>(box + r * 128 + (((c >> 2) ^ (r & 7)) << 4)) =
              make_float4(a[c], a[c + 1], a[c + 2], a[c + 3]);
      };
      // staging boxes [0, nbx) -> channels 32 (bx0 + i) of the accumulator
      auto reduce_staged = [&](int bx0, int nbx) {
        ptx::fence_proxy_async_smem();
        ptx::named_bar_sync(kBarDQ, kDQThreads);
        if (issuer) {
          for (int i = 0; i < nbx; ++i)
            ptx::tma_reduce_add_3d(&tmDQ, sb + i * (128 * 128), 32 * (bx0 + i), i0, b * p.Hq + h);
          ptx::bulk_commit_group();
        }
      };
      if constexpr (D <= 64) {
        float a[D];
#pragma unroll
        for (int c = 0; c < D; c += 32) ptx::tmem_ld32f(tl + kColDQ + c, &a[c]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < D; c += 32) ptx::reg_fence32f(&a[c]);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(dq_free);
        staging_free();
#pragma unroll
        for (int bx = 0; bx < D / 32; ++bx) store_box(&a[32 * bx], bx);
        reduce_staged(0, D / 32);
      } else {
        // d = 128 through one staging box: channels 0-31 go out first, 32-127
        // wait in registers; dQ's TMEM (shared with dP^T) is released once
        // all are read
        float a0[32], a1[96];
        ptx::tmem_ld32f(tl + kColDQ, &a0[0]);
        ptx::tmem_ld_wait();
        ptx::reg_fence32f(&a0[0]);
        staging_free();
        store_box(a0, 0);
        reduce_staged(0, 1);
#pragma unroll
        for (int c = 0; c < 96; c += 32) ptx::tmem_ld32f(tl + kColDQ + 32 + c, &a1[c]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 96; c += 32) ptx::reg_fence32f(&a1[c]);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(dq_free);
#pragma unroll
        for (int bx = 1; bx < 4; ++bx) {
          staging_free();
          store_box(&a1[32 * (bx - 1)], 0);
          reduce_staged(bx, 1);
        }
      }
    }
    if (issuer) ptx::bulk_wait_group0();
    ptx::tc_fence_before();
    __syncthreads();
  }
}

// D_i = dout_scale * sum_c dO_ic O_ic, L2_i = LSE_i log2(e) (a row that saw
// no key: +inf, so that its P is 0), and the dQ accumulator zeroed; DV / 8
// lanes per row, 16 bytes of O and dO each, D / (DV / 8) accumulator values.
template <int D, int DV>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const __grid_constant__ BwdParams p) {
  constexpr int LPR = DV / 8;
  constexpr int ZPL = D / LPR;  // accumulator floats zeroed per lane (4 or 8)
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (256 / LPR) + threadIdx.x / LPR;
  const int sub = threadIdx.x % LPR;
  const bool valid = row < p.rows;
  const int64_t off = (valid ? row : 0) * DV + sub * 8;
  const uint4 ov = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.out) + off));
  const uint4 gv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.dout) + off));
  const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float2 of = __bfloat1622float2(o2[c]), gf = __bfloat1622float2(g2[c]);
    s = fmaf(of.x, gf.x, fmaf(of.y, gf.y, s));
  }
#pragma unroll
  for (int w = LPR / 2; w > 0; w >>= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
  if (!valid) return;
  float4* acc = reinterpret_cast<float4*>(p.dq_acc + row * D + sub * ZPL);
#pragma unroll
  for (int i = 0; i < ZPL / 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sub == 0) {
    p.dvec[row] = s * p.dout_scale;
    const float l = p.lse[row];
    p.l2[row] = l == -CUDART_INF_F ? CUDART_INF_F : l * kLog2e;
  }
}

// dQ = scale * accumulator, rounded to bf16; eight elements per thread.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const __grid_constant__ BwdParams p) {
  const int64_t e = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) * 8;
  if (e >= p.rows * D) return;
  const float4 a = *reinterpret_cast<const float4*>(p.dq_acc + e);
  const float4 c = *reinterpret_cast<const float4*>(p.dq_acc + e + 4);
  const float f = p.scale;
  *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dq) + e) =
      make_uint4(ptx::pack_bf16x2(a.x * f, a.y * f), ptx::pack_bf16x2(a.z * f, a.w * f),
                 ptx::pack_bf16x2(c.x * f, c.y * f), ptx::pack_bf16x2(c.z * f, c.w * f));
}

template <int D, int DV, int SCORE>
cudaError_t launch_bwd_ds(const CUtensorMap* maps, const BwdParams& p, cudaStream_t s) {
  auto kern = attn_bwd_kernel<D, DV, SCORE>;
  constexpr int smem = BwdLayout<D, DV>::SMEM;
  static const cudaError_t checked = [&]() {
    cudaFuncAttributes a{};
    cudaError_t e = cudaFuncGetAttributes(&a, kern);
    if (e != cudaSuccess) return e;
    if (a.numRegs != kBwdLaunchRegs) return cudaErrorInvalidDeviceFunction;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  }();
  if (checked != cudaSuccess) return checked;
  const int rgrid = static_cast<int>((p.rows + 256 / (DV / 8) - 1) / (256 / (DV / 8)));
  attn_bwd_pre_kernel<D, DV><<<rgrid, 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kern<<<p.B * p.Hkv * p.n_ktiles, kBwdThreads, smem, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int pgrid = static_cast<int>((p.rows * D / 8 + 255) / 256);
  attn_bwd_post_kernel<D><<<pgrid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

template <int D, int DV>
cudaError_t launch_bwd_d(int score_mod, const CUtensorMap* maps, const BwdParams& p, cudaStream_t s) {
  switch (score_mod) {
    case SCORE_NONE: return launch_bwd_ds<D, DV, SCORE_NONE>(maps, p, s);
    case SCORE_ALIBI: return launch_bwd_ds<D, DV, SCORE_ALIBI>(maps, p, s);
    default: return launch_bwd_ds<D, DV, SCORE_SOFTCAP>(maps, p, s);
  }
}

}  // namespace

cudaError_t launch_bwd(int d, int dv, int score_mod, const CUtensorMap* maps, const BwdParams& p, cudaStream_t s) {
  if (dv != d) return launch_bwd_d<64, 128>(score_mod, maps, p, s);
  switch (d) {
    case 32: return launch_bwd_d<32, 32>(score_mod, maps, p, s);
    case 64: return launch_bwd_d<64, 64>(score_mod, maps, p, s);
    default: return launch_bwd_d<128, 128>(score_mod, maps, p, s);
  }
}

}  // namespace fl
