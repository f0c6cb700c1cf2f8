// Fused single-pass attention forward for sm_103a (GB300).
//
// One persistent CTA per SM walks a static list of work units.  A unit is
// two 128-row query tiles ("slots") that share every key/value tile the
// load warp brings in; per key tile the work is
//
//   S_s  = Q_s K^T                       (tcgen05.mma, bf16 -> fp32 in TMEM)
//   P_s  = exp2(score(S_s) - m_s)         (softmax warps, registers)
//   O_s += P_s V                         (tcgen05.mma, A = P from TMEM)
//
// which is the fused softmax(QK^T)V the Flashlight pages describe
// (technical summary, gist.science, Methodology: "Structural Fusion with
// Dimension Demotion", "Semantic Fusion with Algebraic Transformation",
// "Tiling-Aware Dimension Elimination and Logical Grids").
//
// Warp roles (320 threads):
//   warp 0      one thread issues TMA loads: Q once per unit, K/V tiles into
//               an mbarrier-guarded ring of STAGES buffers
//   warp 1      allocates TMEM; one thread issues every tcgen05.mma
//   warps 2-5   softmax for slot 0, one thread per query row
//   warps 6-9   softmax for slot 1
// The two slots ping-pong: while the softmax warps of one slot work on S,
// the tensor core computes the other slot's S or P V.
//
// TMEM columns (512 allocated): S0 [0,128), S1 [128,256), O0 [256,256+DV),
// O1 [256+DV, 256+2DV).  P (bf16 pairs) overwrites the first 64 columns of S.
//
// The online softmax keeps (m, l) per row in the log2 domain.  The
// reference max m is only raised when a new tile's max exceeds it by more
// than 8 (a factor 256), so O is rescaled rarely; O and l always use the
// same m, so the final O / l is exact whatever m was used.
//
// Every mbarrier wait is bounded (KParams::timeout_ns).  When one runs out
// the block records FL_ERR_TIMEOUT in the status word, every role leaves
// its loop, in-flight copies and MMAs are drained with bounded waits, and
// TMEM is freed before the block exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "params.h"
#include "ptx.cuh"

namespace fl {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int DV, int KIND>
struct Layout {
  static_assert(D == 32 || D == 64 || D == 128, "head dim");
  static_assert(DV == 32 || DV == 64 || DV == 128, "value head dim");
  // TMA boxes are at most one swizzle span (128 bytes) wide.
  static constexpr int BOXW_D = D >= 64 ? 64 : D;
  static constexpr int NBOX_D = D / BOXW_D;
  static constexpr int ROWB_D = BOXW_D * 2;
  static constexpr int BOX_D_BYTES = kBlockN * ROWB_D;
  static constexpr int BOXW_V = DV >= 64 ? 64 : DV;
  static constexpr int NBOX_V = DV / BOXW_V;
  static constexpr int ROWB_V = BOXW_V * 2;
  static constexpr int BOX_V_BYTES = kBlockN * ROWB_V;
  static constexpr int Q_BYTES = kBlockM * D * 2;
  static constexpr int K_BYTES = kBlockN * D * 2;
  static constexpr int V_BYTES = kBlockN * DV * 2;
  static constexpr int NK = KIND == KIND_DIFF ? 2 : 1;
  static constexpr int STAGE_BYTES = NK * K_BYTES + V_BYTES;
  static constexpr int RING_BUDGET = 200 * 1024 - 2 * Q_BYTES;
  static constexpr int STAGES_FIT = RING_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static_assert(STAGES >= 2, "ring too small");
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * NK * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * V_BYTES;
  // barriers: q_full[2] q_empty[2] k_full[S] k_empty[S] v_full[S] v_empty[S]
  //           s_full[2] p_full[2] o_full[2] o_empty[2] drain[1] xch_full[1]
  static constexpr int NBARS = 14 + 4 * STAGES;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int OFF_XCH = OFF_MISC + 64;          // float [2][128]
  static constexpr int END = OFF_XCH + 2 * kBlockM * 4;
  // +1 KB to align the dynamic base to 1024; at least ~117 KB so that only
  // one block (which owns all 512 TMEM columns) is resident per SM.
  static constexpr int SMEM_BYTES = (END + 1024) > 120 * 1024 ? (END + 1024) : 120 * 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static constexpr uint32_t SWZ_D = ROWB_D == 128 ? 2u : (ROWB_D == 64 ? 4u : 6u);
  static constexpr uint32_t SWZ_V = ROWB_V == 128 ? 2u : (ROWB_V == 64 ? 4u : 6u);
};

struct Unit {
  int b;         // batch (flattened batch * N_seq for the Evoformer)
  int hkv;       // key/value head
  int hq[2];     // query head of each slot
  int row0[2];   // first query row of each slot
  int valid[2];  // slot's results are stored
  int kv_lo, kv_hi;  // inclusive key-tile range (walked from kv_hi down)
};

// Visible keys of query row i form one interval [lo, hi] for every mask kind.
__device__ __forceinline__ void row_bounds(const KParams& p, int b, int i, int& lo, int& hi) {
  switch (p.mask_kind) {
    case MASK_NONE: lo = 0; hi = p.Lk - 1; break;
    case MASK_CAUSAL: lo = 0; hi = i; break;
    case MASK_WINDOW: lo = i - p.window + 1; hi = i; break;
    case MASK_PREFIX: lo = 0; hi = i > p.prefix - 1 ? i : p.prefix - 1; break;
    default: {
      const int32_t* off = p.doc_offsets + static_cast<int64_t>(b) * (p.num_docs + 1);
      int a = 0, z = p.num_docs - 1;
      while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (__ldg(off + mid) <= i) a = mid; else z = mid - 1;
      }
      lo = __ldg(off + a);
      hi = p.doc_causal ? i : __ldg(off + a + 1) - 1;
    }
  }
  lo = lo < 0 ? 0 : lo;
  hi = hi > p.Lk - 1 ? p.Lk - 1 : hi;
}

__device__ __forceinline__ Unit decode_unit(const KParams& p, int u) {
  Unit U;
  if (p.slot_mode == SLOT_ROWS) {
    const int per = p.B * p.Hq;
    const int n_pairs = (p.n_qtiles + 1) >> 1;
    const int tp = n_pairs - 1 - u / per;  // heaviest (last rows) first
    const int rem = u % per;
    U.b = rem / p.Hq;
    const int h = rem % p.Hq;
    U.hq[0] = U.hq[1] = h;
    U.hkv = h / p.group;
    U.row0[0] = (2 * tp) * kBlockM;
    U.row0[1] = (2 * tp + 1) * kBlockM;
    U.valid[0] = 1;
    U.valid[1] = (2 * tp + 1) < p.n_qtiles;
  } else if (p.slot_mode == SLOT_HEADS) {
    const int per = p.B * p.Hkv * p.pairs_per_group;
    const int t = p.n_qtiles - 1 - u / per;
    int rem = u % per;
    U.b = rem / (p.Hkv * p.pairs_per_group);
    rem %= (p.Hkv * p.pairs_per_group);
    U.hkv = rem / p.pairs_per_group;
    const int pair = rem % p.pairs_per_group;
    U.hq[0] = U.hkv * p.group + 2 * pair;
    U.valid[0] = 1;
    U.valid[1] = (2 * pair + 1) < p.group;
    U.hq[1] = U.valid[1] ? U.hq[0] + 1 : U.hq[0];
    U.row0[0] = U.row0[1] = t * kBlockM;
  } else {  // SLOT_BRANCH
    const int per = p.B * p.Hq;
    const int t = p.n_qtiles - 1 - u / per;
    const int rem = u % per;
    U.b = rem / p.Hq;
    U.hq[0] = U.hq[1] = rem % p.Hq;
    U.hkv = U.hq[0];
    U.row0[0] = U.row0[1] = t * kBlockM;
    U.valid[0] = U.valid[1] = 1;
  }
  int lo_min = 0x7fffffff, hi_max = -1;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    if (U.row0[s] >= p.Lq) continue;
    const int r1 = min(U.row0[s] + kBlockM - 1, p.Lq - 1);
    int lo, hi, lo2, hi2;
    row_bounds(p, U.b, U.row0[s], lo, hi);
    row_bounds(p, U.b, r1, lo2, hi2);
    lo_min = min(lo_min, min(lo, lo2));
    hi_max = max(hi_max, max(hi, hi2));
  }
  if (hi_max < lo_min) { lo_min = 0; hi_max = 0; }  // keep >= 1 tile
  U.kv_lo = lo_min / kBlockN;
  U.kv_hi = hi_max / kBlockN;
  return U;
}

// ------------------------------------------------------------ bounded waits
struct Ctl {
  volatile uint32_t* abort;
  uint32_t* status;
  uint64_t timeout_ns;
};

static __device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, const Ctl& c, int where) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (ptx::globaltimer_ns() - t0 > c.timeout_ns) {
      *c.abort = 1u;
      atomicOr(c.status, 1u);
      atomicExch(c.status + 1, static_cast<uint32_t>(where));
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctl& c, int where) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, c, where);
}

// Drain wait used after an abort: ignores the abort flag, gives up after limit.
static __device__ __noinline__ void wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) return;
  }
}

// ------------------------------------------------------------------ kernel
template <int D, int DV, int KIND, int SCORE>
__global__ void __launch_bounds__(kThreads, 1)
    fused_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ0, const __grid_constant__ CUtensorMap tmK0,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ1,
                          const __grid_constant__ CUtensorMap tmK1, const __grid_constant__ KParams p) {
  using L = Layout<D, DV, KIND>;
  constexpr int S = L::STAGES;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 2;
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = bars + 4 + S;
  uint64_t* v_full = bars + 4 + 2 * S;
  uint64_t* v_empty = bars + 4 + 3 * S;
  uint64_t* s_full = bars + 4 + 4 * S;
  uint64_t* p_full = bars + 6 + 4 * S;
  uint64_t* o_full = bars + 8 + 4 * S;
  uint64_t* o_empty = bars + 10 + 4 * S;
  uint64_t* drain = bars + 12 + 4 * S;
  uint64_t* xch_full = bars + 13 + 4 * S;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  float* xch = reinterpret_cast<float*>(smem + L::OFF_XCH);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&q_full[0], 1); ptx::mbar_init(&q_full[1], 1);
    ptx::mbar_init(&q_empty[0], 1); ptx::mbar_init(&q_empty[1], 1);
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&k_full[s], 1); ptx::mbar_init(&k_empty[s], 1);
      ptx::mbar_init(&v_full[s], 1); ptx::mbar_init(&v_empty[s], 1);
    }
    ptx::mbar_init(&s_full[0], 1); ptx::mbar_init(&s_full[1], 1);
    ptx::mbar_init(&p_full[0], 4); ptx::mbar_init(&p_full[1], 4);
    ptx::mbar_init(&o_full[0], 1); ptx::mbar_init(&o_full[1], 1);
    ptx::mbar_init(&o_empty[0], 4); ptx::mbar_init(&o_empty[1], 4);
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(xch_full, 8);
    misc[1] = 0u;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&misc[0], 512);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmQ0); ptx::prefetch_tensormap(&tmK0); ptx::prefetch_tensormap(&tmV);
    if (KIND == KIND_DIFF) { ptx::prefetch_tensormap(&tmQ1); ptx::prefetch_tensormap(&tmK1); }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const Ctl ctl{reinterpret_cast<volatile uint32_t*>(&misc[1]), p.status, p.timeout_ns};
  const uint64_t drain_ns = 50ull * 1000ull * 1000ull;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA load
    if (lane == 0) {
      const uint64_t pol_stream = ptx::policy_evict_first();
      const uint64_t pol_reuse = ptx::policy_evict_last();
      uint32_t it = 0, uc = 0;
      uint32_t k_count = 0, v_count = 0;   // K / V tile loads issued so far (ring order)
      int64_t skipped = -1;                // ring index whose K load was skipped (debug)
      int q_iss[2] = {-1, -1};
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++uc) {
        const Unit U = decode_unit(p, u);
        bool ok = true;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (!wait_bar(&q_empty[s], (uc & 1u) ^ 1u, ctl, 1)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&q_full[s], L::Q_BYTES);
          const CUtensorMap* mq = (KIND == KIND_DIFF && s == 1) ? &tmQ1 : &tmQ0;
#pragma unroll
          for (int bx = 0; bx < L::NBOX_D; ++bx)
            ptx::tma_load_4d(smem + L::OFF_Q + s * L::Q_BYTES + bx * L::BOX_D_BYTES, mq, &q_full[s],
                             bx * L::BOXW_D, U.row0[s], U.hq[s], U.b, pol_stream);
          q_iss[s] = static_cast<int>(uc & 1u);
        }
        if (!ok) break;
        for (int t = U.kv_hi; t >= U.kv_lo; --t, ++it) {
          const int st = static_cast<int>(it % S);
          const uint32_t ph = (it / S) & 1u;
          if (!wait_bar(&k_empty[st], ph ^ 1u, ctl, 2)) { ok = false; break; }
          const bool skip = p.dbg_skip_tile >= 0 && blockIdx.x == 0 && uc == 0 && (U.kv_hi - t) == p.dbg_skip_tile;
          if (!skip) {
            ptx::mbar_arrive_expect_tx(&k_full[st], L::NK * L::K_BYTES);
#pragma unroll
            for (int kk = 0; kk < L::NK; ++kk) {
              const CUtensorMap* mk = kk == 0 ? &tmK0 : &tmK1;
#pragma unroll
              for (int bx = 0; bx < L::NBOX_D; ++bx)
                ptx::tma_load_4d(smem + L::OFF_K + (st * L::NK + kk) * L::K_BYTES + bx * L::BOX_D_BYTES, mk,
                                 &k_full[st], bx * L::BOXW_D, t * kBlockN, U.hkv, U.b, pol_reuse);
            }
          } else {
            skipped = it;
          }
          k_count = it + 1;
          if (!wait_bar(&v_empty[st], ph ^ 1u, ctl, 3)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&v_full[st], L::V_BYTES);
#pragma unroll
          for (int bx = 0; bx < L::NBOX_V; ++bx)
            ptx::tma_load_4d(smem + L::OFF_V + st * L::V_BYTES + bx * L::BOX_V_BYTES, &tmV, &v_full[st],
                             bx * L::BOXW_V, t * kBlockN, U.hkv, U.b, pol_reuse);
          v_count = it + 1;
        }
        if (!ok) break;
      }
      if (*ctl.abort) {
        // let every copy this thread started land before the block exits:
        // per ring slot, wait for the phase of its most recent load
        for (uint32_t back = 1; back <= static_cast<uint32_t>(S); ++back) {
          if (k_count >= back) {
            const uint32_t idx = k_count - back;
            if (static_cast<int64_t>(idx) != skipped) wait_drain(&k_full[idx % S], (idx / S) & 1u, drain_ns);
          }
          if (v_count >= back) {
            const uint32_t idx = v_count - back;
            wait_drain(&v_full[idx % S], (idx / S) & 1u, drain_ns);
          }
        }
        for (int s = 0; s < 2; ++s)
          if (q_iss[s] >= 0) wait_drain(&q_full[s], static_cast<uint32_t>(q_iss[s]), drain_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(kBlockM, kBlockN, false);
      constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(kBlockM, DV, true);
      uint32_t it = 0, uc = 0, pc0 = 0, pc1 = 0;
      const uint32_t q_base = ptx::smem_u32(smem + L::OFF_Q);
      const uint32_t k_base = ptx::smem_u32(smem + L::OFF_K);
      const uint32_t v_base = ptx::smem_u32(smem + L::OFF_V);

      auto issue_s = [&](int s, int st) {
        const uint32_t qa = q_base + s * L::Q_BYTES;
        const uint32_t ka = k_base + (st * L::NK + (L::NK == 2 ? s : 0)) * L::K_BYTES;
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb) {
          const uint32_t off = (kb * 16 / L::BOXW_D) * L::BOX_D_BYTES + (kb * 16 % L::BOXW_D) * 2;
          const uint64_t ad = ptx::smem_desc(qa + off, 16, 8 * L::ROWB_D, L::SWZ_D);
          const uint64_t bd = ptx::smem_desc(ka + off, 16, 8 * L::ROWB_D, L::SWZ_D);
          ptx::mma_ss(tmem + s * 128, ad, bd, IDESC_S, kb > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int s, int st, bool acc) {
        const uint32_t va = v_base + st * L::V_BYTES;
#pragma unroll
        for (int kb = 0; kb < kBlockN / 16; ++kb) {
          const uint64_t bd = ptx::smem_desc(va + kb * 16 * L::ROWB_V, L::BOX_V_BYTES, 8 * L::ROWB_V, L::SWZ_V);
          ptx::mma_ts(tmem + 256 + s * DV, tmem + s * 128 + kb * 8, bd, IDESC_O, (acc || kb > 0) ? 1u : 0u);
        }
      };

      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++uc) {
        const Unit U = decode_unit(p, u);
        const int n = U.kv_hi - U.kv_lo + 1;
        if (!wait_bar(&q_full[0], uc & 1u, ctl, 10) || !wait_bar(&q_full[1], uc & 1u, ctl, 10)) { ok = false; break; }
        {
          const int st = static_cast<int>(it % S);
          if (!wait_bar(&k_full[st], (it / S) & 1u, ctl, 11)) { ok = false; break; }
          ptx::tc_fence_after();
          issue_s(0, st);
          ptx::mma_commit(&s_full[0]);
          issue_s(1, st);
          ptx::mma_commit(&s_full[1]);
          ptx::mma_commit(&k_empty[st]);
        }
        for (int t = 0; t < n; ++t) {
          const uint32_t itc = it + t;
          const int st = static_cast<int>(itc % S);
          const bool more = t + 1 < n;
          const int stn = static_cast<int>((itc + 1) % S);
          const uint32_t phn = ((itc + 1) / S) & 1u;
          if (!wait_bar(&v_full[st], (itc / S) & 1u, ctl, 12)) { ok = false; break; }
          if (t == 0) {
            if (!wait_bar(&o_empty[0], (uc & 1u) ^ 1u, ctl, 13)) { ok = false; break; }
            if (KIND == KIND_DIFF && !wait_bar(&o_empty[1], (uc & 1u) ^ 1u, ctl, 13)) { ok = false; break; }
          }
          if (!wait_bar(&p_full[0], pc0 & 1u, ctl, 14)) { ok = false; break; }
          ++pc0;
          ptx::tc_fence_after();
          issue_pv(0, st, t > 0);
          if (more) {
            if (!wait_bar(&k_full[stn], phn, ctl, 15)) { ok = false; break; }
            ptx::tc_fence_after();
            issue_s(0, stn);
            ptx::mma_commit(&s_full[0]);
          } else {
            ptx::mma_commit(&o_full[0]);
          }
          if (t == 0 && KIND != KIND_DIFF) {
            if (!wait_bar(&o_empty[1], (uc & 1u) ^ 1u, ctl, 16)) { ok = false; break; }
          }
          if (!wait_bar(&p_full[1], pc1 & 1u, ctl, 17)) { ok = false; break; }
          ++pc1;
          ptx::tc_fence_after();
          issue_pv(1, st, t > 0);
          ptx::mma_commit(&v_empty[st]);
          if (more) {
            issue_s(1, stn);
            ptx::mma_commit(&s_full[1]);
            ptx::mma_commit(&k_empty[stn]);
          } else {
            ptx::mma_commit(&o_full[1]);
            ptx::mma_commit(&q_empty[0]);
            ptx::mma_commit(&q_empty[1]);
          }
        }
        it += n;
      }
      // every MMA this thread issued must finish before TMEM is released
      ptx::mma_commit(drain);
      wait_drain(drain, 0u, drain_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int s = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t tS = tl + s * 128;
    const uint32_t tO = tl + 256 + s * DV;
    const float scale_log2 = p.scale_log2;
    uint32_t scnt = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++uc) {
      const Unit U = decode_unit(p, u);
      const int n = U.kv_hi - U.kv_lo + 1;
      const int i = U.row0[s] + r;
      const int ic = i < p.Lq ? i : p.Lq - 1;
      int lo, hi;
      row_bounds(p, U.b, ic, lo, hi);
      float slope2 = 0.f;
      if (SCORE == SCORE_ALIBI) slope2 = __ldg(p.slopes + U.hq[s]) * kLog2e;
      const float* pb_row = nullptr;
      const float* mb_row = nullptr;
      if (KIND == KIND_EVO) {
        const int bb = U.b / p.n_seq;
        if (p.pair_bias) pb_row = p.pair_bias + (static_cast<int64_t>(bb * p.Hq + U.hq[s]) * p.Lq + ic) * p.Lk;
        if (p.mask_bias) mb_row = p.mask_bias + static_cast<int64_t>(U.b) * p.Lk;
      }
      float m = -CUDART_INF_F, l = 0.f;
      for (int t = 0; t < n; ++t, ++scnt) {
        const int j0 = (U.kv_hi - t) * kBlockN;
        if (!__all_sync(0xffffffffu, wait_bar(&s_full[s], scnt & 1u, ctl, 20 + s))) { ok = false; break; }
        ptx::tc_fence_after();
        float x[kBlockN];
        {
          uint32_t rr[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            ptx::tmem_ld32(tS + c * 32, rr);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(rr);
#pragma unroll
            for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(rr[e]);
          }
        }
        // score transform into the log2 domain
        if (SCORE == SCORE_NONE && KIND != KIND_EVO) {
#pragma unroll
          for (int c = 0; c < kBlockN; ++c) x[c] *= scale_log2;
        } else if (SCORE == SCORE_ALIBI) {
          const float base = slope2 * static_cast<float>(j0 - ic);
#pragma unroll
          for (int c = 0; c < kBlockN; ++c) x[c] = fmaf(x[c], scale_log2, fmaf(slope2, static_cast<float>(c), base));
        } else if (SCORE == SCORE_SOFTCAP) {
          // cap * tanh(s*scale/cap), tanh(y) = 1 - 2 / (1 + e^(2y))
          const float a = scale_log2 * 2.0f / p.softcap;   // 2 * y * log2(e) = s * a
          const float cap2 = p.softcap * kLog2e;
#pragma unroll
          for (int c = 0; c < kBlockN; ++c) {
            const float e = ptx::ex2(x[c] * a);
            const float th = fmaf(-2.0f, ptx::rcp(1.0f + e), 1.0f);
            x[c] = th * cap2;
          }
        }
        if (KIND == KIND_EVO) {
          const bool ragged = j0 + kBlockN > p.Lk;
#pragma unroll
          for (int c4 = 0; c4 < kBlockN / 4; ++c4) {
            float4 pb = make_float4(0.f, 0.f, 0.f, 0.f), mb = pb;
            const int j = j0 + 4 * c4;
            if (!ragged) {
              if (pb_row) pb = __ldg(reinterpret_cast<const float4*>(pb_row + j));
              if (mb_row) mb = __ldg(reinterpret_cast<const float4*>(mb_row + j));
            } else {
              if (pb_row) {
                pb.x = j + 0 < p.Lk ? __ldg(pb_row + j + 0) : 0.f; pb.y = j + 1 < p.Lk ? __ldg(pb_row + j + 1) : 0.f;
                pb.z = j + 2 < p.Lk ? __ldg(pb_row + j + 2) : 0.f; pb.w = j + 3 < p.Lk ? __ldg(pb_row + j + 3) : 0.f;
              }
              if (mb_row) {
                mb.x = j + 0 < p.Lk ? __ldg(mb_row + j + 0) : 0.f; mb.y = j + 1 < p.Lk ? __ldg(mb_row + j + 1) : 0.f;
                mb.z = j + 2 < p.Lk ? __ldg(mb_row + j + 2) : 0.f; mb.w = j + 3 < p.Lk ? __ldg(mb_row + j + 3) : 0.f;
              }
            }
            x[4 * c4 + 0] = fmaf(x[4 * c4 + 0], scale_log2, (pb.x + mb.x) * kLog2e);
            x[4 * c4 + 1] = fmaf(x[4 * c4 + 1], scale_log2, (pb.y + mb.y) * kLog2e);
            x[4 * c4 + 2] = fmaf(x[4 * c4 + 2], scale_log2, (pb.z + mb.z) * kLog2e);
            x[4 * c4 + 3] = fmaf(x[4 * c4 + 3], scale_log2, (pb.w + mb.w) * kLog2e);
          }
        }
        // mask (only when some row of this warp has a partially visible tile)
        if (__any_sync(0xffffffffu, (j0 < lo) || (j0 + kBlockN - 1 > hi))) {
          const int clo = lo - j0, chi = hi - j0;
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (c < clo || c > chi) x[c] = -CUDART_INF_F;
        }
        // row max
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = x[e];
#pragma unroll
        for (int c = 8; c < kBlockN; c += 8)
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], x[c + e]);
        const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_new = fmaxf(m, tmax);
        float alpha = 1.f;
        if (m_new > m + kRescaleThreshold || (m == -CUDART_INF_F && m_new != -CUDART_INF_F)) {
          alpha = (m == -CUDART_INF_F) ? 0.f : ptx::ex2(m - m_new);
          m = m_new;
        }
        l *= alpha;
        const float msub = (m == -CUDART_INF_F) ? 0.f : m;
        float ls[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ls[e] = 0.f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ptx::ex2(x[h * 32 + 2 * e] - msub);
            const float p1 = ptx::ex2(x[h * 32 + 2 * e + 1] - msub);
            ls[(2 * e) & 7] += p0;
            ls[(2 * e + 1) & 7] += p1;
            pk[e] = ptx::pack_bf16x2(p0, p1);
          }
          ptx::tmem_st16(tS + h * 16, pk);
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        // O rescale after the P stores so that x[] is dead (register pressure)
        if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < DV; c += 32) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + c, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st32(tO + c, o);
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&p_full[s]);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      if (!__all_sync(0xffffffffu, wait_bar(&o_full[s], uc & 1u, ctl, 30 + s))) { ok = false; break; }
      if (KIND == KIND_DIFF && !__all_sync(0xffffffffu, wait_bar(&o_full[s ^ 1], uc & 1u, ctl, 30 + s))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const float lse2 = (l > 0.f) ? (m + __log2f(l)) : -CUDART_INF_F;  // log2 domain
      if (KIND == KIND_DIFF) {
        // Each branch's softmax warps publish l for their rows, then each
        // slot produces half of the output channels of O1/l1 - lambda O2/l2.
        // xch is rewritten only in the next unit's epilogue, which needs
        // o_full of the next unit, hence the MMA warp's wait on both o_empty
        // barriers, which each slot arrives on only after its reads below.
        xch[s * kBlockM + r] = l;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(xch_full);
        ok = wait_bar(xch_full, uc & 1u, ctl, 32);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const float l0 = xch[r];
        const float l1 = xch[kBlockM + r];
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float inv1 = l1 > 0.f ? -p.lambda / l1 : 0.f;
        const uint32_t tO0 = tl + 256, tO1 = tl + 256 + DV;
        constexpr int HALF = DV / 2;
        uint32_t packed[HALF / 2];
#pragma unroll
        for (int c = 0; c < HALF; c += 32) {
          uint32_t a[32], bq[32];
          ptx::tmem_ld32(tO0 + s * HALF + c, a);
          ptx::tmem_ld32(tO1 + s * HALF + c, bq);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(a);
          ptx::reg_fence32(bq);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float y0 = fmaf(__uint_as_float(bq[2 * e]), inv1, __uint_as_float(a[2 * e]) * inv0);
            const float y1 = fmaf(__uint_as_float(bq[2 * e + 1]), inv1, __uint_as_float(a[2 * e + 1]) * inv0);
            packed[c / 2 + e] = ptx::pack_bf16x2(y0, y1);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&o_empty[s]);
        if (i < p.Lq) {
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + U.b * p.o_sb + U.hq[s] * p.o_sh +
                                static_cast<int64_t>(i) * p.o_sl + s * HALF;
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int e = 0; e < HALF / 8; ++e)
            dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
          if (p.lse)
            p.lse[static_cast<int64_t>(s) * p.B * p.Hq * p.Lq + (static_cast<int64_t>(U.b) * p.Hq + U.hq[s]) * p.Lq + i] =
                lse2 * kLn2;
        }
      } else {
        const bool store = i < p.Lq && U.valid[s];
        const int64_t orow_off = U.b * p.o_sb + U.hq[s] * p.o_sh + static_cast<int64_t>(i) * p.o_sl;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float gsig[KIND == KIND_EVO ? DV : 1];
        if (KIND == KIND_EVO) {
          // out = sigmoid(gate) * O / l, sigmoid(g) = 1 / (1 + 2^(-g log2 e))
          const uint4* g4 = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.gate) + orow_off);
#pragma unroll
          for (int e = 0; e < DV / 8; ++e) {
            const uint4 gv = store ? __ldg(g4 + e) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[w]));
              gsig[8 * e + 2 * w] = ptx::rcp(1.f + ptx::ex2(-gf.x * kLog2e)) * inv;
              gsig[8 * e + 2 * w + 1] = ptx::rcp(1.f + ptx::ex2(-gf.y * kLog2e)) * inv;
            }
          }
        }
        uint32_t packed[DV / 2];
#pragma unroll
        for (int c = 0; c < DV; c += 32) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + c, o);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(o);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float f0 = KIND == KIND_EVO ? gsig[(c + 2 * e) % (KIND == KIND_EVO ? DV : 1)] : inv;
            const float f1 = KIND == KIND_EVO ? gsig[(c + 2 * e + 1) % (KIND == KIND_EVO ? DV : 1)] : inv;
            packed[c / 2 + e] = ptx::pack_bf16x2(__uint_as_float(o[2 * e]) * f0, __uint_as_float(o[2 * e + 1]) * f1);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&o_empty[s]);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow_off);
#pragma unroll
          for (int e = 0; e < DV / 8; ++e)
            dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
          if (p.lse) p.lse[(static_cast<int64_t>(U.b) * p.Hq + U.hq[s]) * p.Lq + i] = lse2 * kLn2;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace fl
