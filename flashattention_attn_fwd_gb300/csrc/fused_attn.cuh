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
// Warp roles (352 threads):
//   warp 0      one thread issues TMA loads: Q once per unit (double-buffered,
//               so the next unit's Q arrives early), K/V tiles into an
//               mbarrier-guarded ring of STAGES buffers
//   warp 1      allocates TMEM; one thread issues slot 0's tcgen05.mma
//   warp 10     one thread issues slot 1's tcgen05.mma
//   warps 2-5   softmax for slot 0, one thread per query row
//   warps 6-9   softmax for slot 1
// While the softmax warps of one slot work on S, the tensor core computes
// the other slot's S or P V.
//
// TMEM columns (512 allocated): S0 [0,128), S1 [128,256).  For DV <= 64 the
// bf16 P of each slot has its own 64 columns (P0 [256,320), P1 [320,384))
// and O0, O1 follow; the next tile's S is then issued as soon as the softmax
// warps have pulled the current S into registers, so a slot's softmax never
// waits for its own P V.  For DV = 128 (no room left) P overwrites the first
// 64 columns of S, O0, O1 start at column 256, and the next S follows the
// P V in issue order.
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

// Optional per-phase clock64() stamps of block 0 (compile with -DFL_TRACE and
// set KParams::trace): role 0 = MMA thread, 1/2 = softmax slot 0/1 (lane 0 of
// its first warp), 3 = TMA thread; up to 64 tiles, 8 events each.
#ifdef FL_TRACE
#define FL_TR(role, idx, ev)                                                        \
  do {                                                                              \
    if (p.trace && blockIdx.x == 0 && (idx) < 64)                                   \
      p.trace[((role) * 64 + (idx)) * 8 + (ev)] = static_cast<unsigned long long>(clock64()); \
  } while (0)
#else
#define FL_TR(role, idx, ev) \
  do {                       \
  } while (0)
#endif

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// tanh(y) ~= y * P(y^2) on |y| <= kTanhPolyRange, P of degree 4 in y^2
// (coefficients from csrc/fit_tanh_poly.py: minimax relative error, float32
// max relative error 1.1e-7 on the range).
constexpr float kTanhPolyRange = 0.5f;
constexpr float kTanhC1 = -0.333330691f;
constexpr float kTanhC2 = 0.133247837f;
constexpr float kTanhC3 = -0.0529862903f;
constexpr float kTanhC4 = 0.0171353891f;

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
  // Q is double-buffered (the next unit's Q loads while this one runs) when
  // that still leaves room for two K/V stages.
  static constexpr int QBUF = (4 * Q_BYTES + 2 * STAGE_BYTES <= 200 * 1024) ? 2 : 1;
  static constexpr int RING_BUDGET = 200 * 1024 - 2 * QBUF * Q_BYTES;
  static constexpr int STAGES_FIT = RING_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static_assert(STAGES >= 2, "ring too small");
  static constexpr int OFF_Q = 0;                        // Q[buffer][slot]
  static constexpr int OFF_K = 2 * QBUF * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * NK * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * V_BYTES;
  // barriers: q_full[4] q_empty[4] kv_full[S] kv_empty[S] s_full[2] s_free[2]
  //           p_full[2] pv_done[2] o_empty[2] drain[2] xch_full[1] stagger[1]
  //           o_staged[2]
  static constexpr int NBARS = 24 + 2 * STAGES;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int OFF_XCH = OFF_MISC + 64;          // float [2][128]
  static constexpr int OFF_UNITS = OFF_XCH + 2 * kBlockM * 4;  // Unit[4]: decoded units, ring
  static constexpr int END = OFF_UNITS + 4 * 64;
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
static_assert(sizeof(Unit) <= 64, "unit ring entry");

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
                          const __grid_constant__ CUtensorMap tmK1, const __grid_constant__ CUtensorMap tmO,
                          const __grid_constant__ KParams p) {
  using L = Layout<D, DV, KIND>;
  constexpr int S = L::STAGES;
  // TMEM columns: S0 [0,128) S1 [128,256); with DV <= 64 a separate P region
  // P0 [256,320) P1 [320,384) and O0, O1 from 384; with DV = 128 P is
  // written over the first 64 columns of S and O0, O1 start at 256.
  constexpr bool kSepP = DV <= 64;
  constexpr uint32_t kColP = kSepP ? 256u : 0u;   // + 64 * slot (sep) or + 128 * slot (aliased)
  constexpr uint32_t kColO = kSepP ? 384u : 256u;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;               // [buffer * 2 + slot]
  uint64_t* q_empty = bars + 4;          // [buffer * 2 + slot]
  uint64_t* kv_full = bars + 8;          // [stage]
  uint64_t* kv_empty = bars + 8 + S;     // [stage]
  uint64_t* s_full = bars + 8 + 2 * S;   // [slot]
  uint64_t* s_free = bars + 10 + 2 * S;
  uint64_t* p_full = bars + 12 + 2 * S;
  uint64_t* pv_done = bars + 14 + 2 * S;
  uint64_t* o_empty = bars + 16 + 2 * S;
  uint64_t* drain = bars + 18 + 2 * S;
  uint64_t* xch_full = bars + 20 + 2 * S;
  uint64_t* stagger = bars + 21 + 2 * S;
  uint64_t* o_staged = bars + 22 + 2 * S;  // [slot]: output tile written to shared memory
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  float* xch = reinterpret_cast<float*>(smem + L::OFF_XCH);
  // The TMA thread decodes each unit once and publishes it here before
  // arriving on the unit's q_full barriers (release); the MMA and softmax
  // threads read it after waiting on q_full (acquire).  A ring of 4 suffices:
  // the TMA thread runs at most two units ahead (two Q buffers).
  Unit* units = reinterpret_cast<Unit*>(smem + L::OFF_UNITS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(&q_full[i], 1);
      ptx::mbar_init(&q_empty[i], 1);
    }
    for (int st = 0; st < S; ++st) {
      ptx::mbar_init(&kv_full[st], 1);
      ptx::mbar_init(&kv_empty[st], 2);  // released by both slots' MMA threads
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s_full[i], 1);
      ptx::mbar_init(&s_free[i], 4);
      ptx::mbar_init(&p_full[i], 4);
      ptx::mbar_init(&pv_done[i], 1);
      ptx::mbar_init(&o_empty[i], 4);
      ptx::mbar_init(&drain[i], 1);
    }
    ptx::mbar_init(xch_full, 8);
    ptx::mbar_init(stagger, 4);
    ptx::mbar_init(&o_staged[0], 4);
    ptx::mbar_init(&o_staged[1], 4);
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
    ptx::prefetch_tensormap(&tmO);
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
      uint32_t kv_count = 0;               // K/V stage loads issued so far (ring order)
      int64_t skipped = -1;                // ring index whose K load was skipped (debug)
      int q_iss[4] = {-1, -1, -1, -1};     // phase of the latest Q load per buffer
      constexpr uint32_t kStageTx = L::NK * L::K_BYTES + L::V_BYTES;
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++uc) {
        const Unit U = decode_unit(p, u);
        const uint32_t qb = uc % L::QBUF, qph = (uc / L::QBUF) & 1u;
        bool ok = true;
        units[uc & 3u] = U;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const int qi = static_cast<int>(qb) * 2 + s;
          if (!wait_bar(&q_empty[qi], qph ^ 1u, ctl, 1)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&q_full[qi], L::Q_BYTES);
          const CUtensorMap* mq = (KIND == KIND_DIFF && s == 1) ? &tmQ1 : &tmQ0;
#pragma unroll
          for (int bx = 0; bx < L::NBOX_D; ++bx)
            ptx::tma_load_4d(smem + L::OFF_Q + qi * L::Q_BYTES + bx * L::BOX_D_BYTES, mq, &q_full[qi],
                             bx * L::BOXW_D, U.row0[s], U.hq[s], U.b, pol_stream);
          q_iss[qi] = static_cast<int>(qph);
        }
        if (!ok) break;
        for (int t = U.kv_hi; t >= U.kv_lo; --t, ++it) {
          const int st = static_cast<int>(it % S);
          const uint32_t ph = (it / S) & 1u;
          if (!wait_bar(&kv_empty[st], ph ^ 1u, ctl, 2)) { ok = false; break; }
          const bool skip = p.dbg_skip_tile >= 0 && blockIdx.x == 0 && uc == 0 && (U.kv_hi - t) == p.dbg_skip_tile;
          ptx::mbar_arrive_expect_tx(&kv_full[st], kStageTx);
          if (!skip) {
#pragma unroll
            for (int kk = 0; kk < L::NK; ++kk) {
              const CUtensorMap* mk = kk == 0 ? &tmK0 : &tmK1;
#pragma unroll
              for (int bx = 0; bx < L::NBOX_D; ++bx)
                ptx::tma_load_4d(smem + L::OFF_K + (st * L::NK + kk) * L::K_BYTES + bx * L::BOX_D_BYTES, mk,
                                 &kv_full[st], bx * L::BOXW_D, t * kBlockN, U.hkv, U.b, pol_reuse);
            }
          } else {
            skipped = it;  // this stage's barrier never completes: the waits on it run out
          }
#pragma unroll
          for (int bx = 0; bx < L::NBOX_V; ++bx)
            ptx::tma_load_4d(smem + L::OFF_V + st * L::V_BYTES + bx * L::BOX_V_BYTES, &tmV, &kv_full[st],
                             bx * L::BOXW_V, t * kBlockN, U.hkv, U.b, pol_reuse);
          kv_count = it + 1;
        }
        if (!ok) break;
      }
      if (*ctl.abort) {
        // let every copy this thread started land before the block exits:
        // per ring slot and Q buffer, wait for the phase of its latest load
        for (uint32_t back = 1; back <= static_cast<uint32_t>(S); ++back) {
          if (kv_count >= back) {
            const uint32_t idx = kv_count - back;
            if (static_cast<int64_t>(idx) != skipped) wait_drain(&kv_full[idx % S], (idx / S) & 1u, drain_ns);
          }
        }
        for (int qi = 0; qi < 4; ++qi)
          if (q_iss[qi] >= 0) wait_drain(&q_full[qi], static_cast<uint32_t>(q_iss[qi]), drain_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 10) {
    // ------------------------------------------------------------ MMA issue
    // One thread per slot issues that slot's MMAs, so neither slot's hand-offs
    // wait behind the other's.  Per tile: the next S as soon as the softmax
    // warps have pulled the current S into registers (s_free) and its K tile
    // is in (kv_full); P V as soon as P is in TMEM (p_full).  With P written
    // over S (DV = 128) the next S follows the P V instead.
    // With separate P each slot gets its own issuing thread (warp 1: slot 0,
    // warp 10: slot 1); with P over S one thread (warp 1) alternates the
    // slots -- P V(0), S(0, next), P V(1), S(1, next) -- so the two softmax
    // warpgroups stay half a tile apart.
    const int s_lo = kSepP ? (warp == 1 ? 0 : 1) : 0;
    const int s_hi = kSepP ? s_lo : 1;
    if (lane == 0 && (kSepP || warp == 1)) {
      constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(kBlockM, kBlockN, false);
      constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(kBlockM, DV, true);
      uint32_t it = 0, uc = 0;
      uint32_t pc[2] = {0u, 0u}, sf[2] = {0u, 0u};
      const uint32_t q_base = ptx::smem_u32(smem + L::OFF_Q);
      const uint32_t k_base = ptx::smem_u32(smem + L::OFF_K);
      const uint32_t v_base = ptx::smem_u32(smem + L::OFF_V);

      // Descriptors are built once per call from the tile base; the k-step
      // offsets only add to the 14-bit start-address field (tile bases and
      // offsets stay below 256 KB, so the field never carries).
      auto issue_s = [&](int s, uint32_t qb, int st) -> bool {
        if (!wait_bar(&s_free[s], (sf[s] & 1u) ^ 1u, ctl, 18 + s)) return false;
        ptx::tc_fence_after();
        const uint32_t qa = q_base + (qb * 2 + s) * L::Q_BYTES;
        const uint32_t ka = k_base + (st * L::NK + (L::NK == 2 ? s : 0)) * L::K_BYTES;
        const uint64_t ad0 = ptx::smem_desc(qa, 16, 8 * L::ROWB_D, L::SWZ_D);
        const uint64_t bd0 = ptx::smem_desc(ka, 16, 8 * L::ROWB_D, L::SWZ_D);
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb) {
          const uint32_t off = ((kb * 16 / L::BOXW_D) * L::BOX_D_BYTES + (kb * 16 % L::BOXW_D) * 2) >> 4;
          ptx::mma_ss(tmem + s * 128, ad0 + off, bd0 + off, IDESC_S, kb > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&s_full[s]);
        ++sf[s];
        return true;
      };
      auto issue_pv = [&](int s, int st, bool acc) {
        const uint64_t bd0 = ptx::smem_desc(v_base + st * L::V_BYTES, L::BOX_V_BYTES, 8 * L::ROWB_V, L::SWZ_V);
        const uint32_t tP = tmem + (kSepP ? kColP + s * 64 : s * 128);
        const uint32_t tO = tmem + kColO + s * DV;
#pragma unroll
        for (int kb = 0; kb < kBlockN / 16; ++kb)
          ptx::mma_ts(tO, tP + kb * 8, bd0 + ((kb * 16 * L::ROWB_V) >> 4), IDESC_O, (acc || kb > 0) ? 1u : 0u);
      };

      // With two Q buffers the first S of the next unit is issued in place
      // of a "next tile" S during the last tile of the current unit.
      constexpr bool kCross = kSepP && L::QBUF == 2;
      auto wait_q = [&](uint32_t ucn) -> bool {
        for (int s = s_lo; s <= s_hi; ++s)
          if (!wait_bar(&q_full[(ucn % L::QBUF) * 2 + s], (ucn / L::QBUF) & 1u, ctl, 10)) return false;
        return true;
      };
      auto first_s = [&](uint32_t ucn, uint32_t itn) -> bool {
        const int st = static_cast<int>(itn % S);
        if (!wait_q(ucn) || !wait_bar(&kv_full[st], (itn / S) & 1u, ctl, 11)) return false;
        for (int s = s_lo; s <= s_hi; ++s)
          if (!issue_s(s, ucn % L::QBUF, st)) return false;
        return true;
      };
      bool ok = true;
      int u = blockIdx.x;
      if (u < p.num_units) ok = first_s(0u, 0u);
      while (u < p.num_units && ok) {
        if (!kCross && !wait_q(uc)) { ok = false; break; }  // (kCross: waited in first_s)
        const Unit U = units[uc & 3u];
        const int n = U.kv_hi - U.kv_lo + 1;
        const uint32_t qb = uc % L::QBUF;
        const bool next_unit = u + static_cast<int>(gridDim.x) < p.num_units;
        for (int t = 0; t < n && ok; ++t) {
          const uint32_t itc = it + t;
          const int st = static_cast<int>(itc % S);
          const bool more = t + 1 < n;
          const int stn = static_cast<int>((itc + 1) % S);
          const uint32_t phn = ((itc + 1) / S) & 1u;
          FL_TR(0, itc, 0);
          if (kSepP && more) {
            if (!wait_bar(&kv_full[stn], phn, ctl, 15)) { ok = false; break; }
            FL_TR(0, itc, 1);
            for (int s = s_lo; s <= s_hi && ok; ++s)
              if (!issue_s(s, qb, stn)) ok = false;
            if (!ok) break;
          } else if (kCross && !more && next_unit) {
            if (!first_s(uc + 1, itc + 1)) { ok = false; break; }
          }
          FL_TR(0, itc, 2);
          for (int s = s_lo; s <= s_hi; ++s) {
            if (t == 0) {
              if (!wait_bar(&o_empty[s], (uc & 1u) ^ 1u, ctl, 13)) { ok = false; break; }
              if (KIND == KIND_DIFF && !wait_bar(&o_empty[s ^ 1], (uc & 1u) ^ 1u, ctl, 13)) { ok = false; break; }
            }
            FL_TR(0, itc, 3);
            if (!wait_bar(&p_full[s], pc[s] & 1u, ctl, 14)) { ok = false; break; }
            FL_TR(0, itc, 4);
            ++pc[s];
            ptx::tc_fence_after();
            issue_pv(s, st, t > 0);
            ptx::mma_commit(&pv_done[s]);
            ptx::mma_commit(&kv_empty[st]);
            FL_TR(0, itc, 5);
            if (!kSepP && more) {
              if (s == s_lo && !wait_bar(&kv_full[stn], phn, ctl, 15)) { ok = false; break; }
              if (!issue_s(s, qb, stn)) { ok = false; break; }
            }
          }
        }
        it += n;
        ++uc;
        u += gridDim.x;
        if (ok && !kCross && u < p.num_units) ok = first_s(uc, it);
      }
      // every MMA this thread issued must finish before TMEM is released
      ptx::mma_commit(&drain[s_lo]);
      wait_drain(&drain[s_lo], 0u, drain_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int s = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t tS = tl + s * 128;
    const uint32_t tP = tl + (kSepP ? kColP + s * 64 : s * 128);
    const uint32_t tO = tl + kColO + s * DV;
    const float scale_log2 = p.scale_log2;
    uint32_t scnt = 0, uc = 0;
    uint32_t pc = 0;  // P tiles handed to the MMA warp so far (= P V launched for this slot)
    bool ok = true;

    // What the epilogue of a unit needs once its tile loop is over.
    struct Epi {
      int b, hq, row0, valid, i;
      uint32_t uc, pcl;  // unit counter; index of the unit's last P V completion
      float m, l;
    };
    // With two Q buffers the epilogue of a unit runs after the next unit's
    // first tile (its last P V has finished by then, and that tile's softmax
    // overlaps the wait), and the bulk store's hold on the staging buffer is
    // released at the next tile instead of being waited for.
    constexpr bool kDefer = L::QBUF == 2;
    const bool leader = lane == 0 && warp == 2 + 4 * s;
    int pending_qi = -1;  // leader: Q buffer whose bulk store may still be reading it
    bool have_prev = false;
    Epi prev{};
    auto release_pending = [&]() {
      if (leader && pending_qi >= 0) {
        ptx::bulk_wait_group_read0();
        ptx::mbar_arrive(&q_empty[pending_qi]);
        pending_qi = -1;
      }
    };
    auto epilogue = [&](const Epi& e) -> bool {
      const bool tre = lane == 0 && warp == 2;
      if (tre) FL_TR(3, e.uc, 0);
      // O is final once the unit's last P V is done
      if (!__all_sync(0xffffffffu, wait_bar(&pv_done[s], e.pcl & 1u, ctl, 30 + s))) return false;
      if (tre) FL_TR(3, e.uc, 1);
      if (KIND == KIND_DIFF && !__all_sync(0xffffffffu, wait_bar(&pv_done[s ^ 1], e.pcl & 1u, ctl, 30 + s)))
        return false;
      ptx::tc_fence_after();
      const float lse2 = (e.l > 0.f) ? (e.m + __log2f(e.l)) : -CUDART_INF_F;  // log2 domain
      // Each slot writes its output tile (all DV channels; differential
      // attention: its half of them) into its own Q buffer of that unit,
      // which the unit's last S has finished reading, in the TMA swizzle
      // layout; one thread then stores the tile with a bulk tensor copy, and
      // only after the copy has read the buffer is it handed back to the
      // load warp for a later unit's Q.
      constexpr int OUT_COLS = KIND == KIND_DIFF ? DV / 2 : DV;
      uint32_t packed[OUT_COLS / 2];
      int64_t lse_off;
      if (KIND == KIND_DIFF) {
        // Each branch's softmax warps publish l for their rows, then each
        // slot produces half of the output channels of O1/l1 - lambda O2/l2.
        // xch is rewritten only in the next unit's epilogue, which needs the
        // next unit's P V, hence the MMA warp's wait on both o_empty
        // barriers, which each slot arrives on only after its reads below.
        xch[s * kBlockM + r] = e.l;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(xch_full);
        if (!__all_sync(0xffffffffu, wait_bar(xch_full, e.uc & 1u, ctl, 32))) return false;
        const float l0 = xch[r];
        const float l1 = xch[kBlockM + r];
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float inv1 = l1 > 0.f ? -p.lambda / l1 : 0.f;
        const uint32_t tO0 = tl + kColO, tO1 = tl + kColO + DV;
#pragma unroll
        for (int c = 0; c < OUT_COLS; c += 32) {
          uint32_t a[32], bq[32];
          ptx::tmem_ld32(tO0 + s * OUT_COLS + c, a);
          ptx::tmem_ld32(tO1 + s * OUT_COLS + c, bq);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(a);
          ptx::reg_fence32(bq);
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float y0 = fmaf(__uint_as_float(bq[2 * q]), inv1, __uint_as_float(a[2 * q]) * inv0);
            const float y1 = fmaf(__uint_as_float(bq[2 * q + 1]), inv1, __uint_as_float(a[2 * q + 1]) * inv0);
            packed[c / 2 + q] = ptx::pack_bf16x2(y0, y1);
          }
        }
        lse_off = static_cast<int64_t>(s) * p.B * p.Hq * p.Lq + (static_cast<int64_t>(e.b) * p.Hq + e.hq) * p.Lq + e.i;
      } else {
        const int64_t orow_off = e.b * p.o_sb + e.hq * p.o_sh + static_cast<int64_t>(e.i) * p.o_sl;
        const float inv = e.l > 0.f ? 1.f / e.l : 0.f;
        float gsig[KIND == KIND_EVO ? DV : 1];
        if (KIND == KIND_EVO) {
          // out = sigmoid(gate) * O / l, sigmoid(g) = 1 / (1 + 2^(-g log2 e))
          const bool row_ok = e.i < p.Lq;
          const uint4* g4 = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.gate) + orow_off);
#pragma unroll
          for (int q = 0; q < DV / 8; ++q) {
            const uint4 gv = row_ok ? __ldg(g4 + q) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[w]));
              gsig[8 * q + 2 * w] = ptx::rcp(1.f + ptx::ex2(-gf.x * kLog2e)) * inv;
              gsig[8 * q + 2 * w + 1] = ptx::rcp(1.f + ptx::ex2(-gf.y * kLog2e)) * inv;
            }
          }
        }
        // O in chunks of up to 64 columns, all loads of a chunk before one wait
        constexpr int CH = DV <= 64 ? DV : 64;
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += CH) {
          uint32_t o[CH];
#pragma unroll
          for (int c = 0; c < CH; c += 32) ptx::tmem_ld32(tO + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(&o[c]));
          ptx::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < CH; c += 32) ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&o[c]));
#pragma unroll
          for (int q = 0; q < CH / 2; ++q) {
            const int cc = c0 + 2 * q;
            const float f0 = KIND == KIND_EVO ? gsig[cc % (KIND == KIND_EVO ? DV : 1)] : inv;
            const float f1 = KIND == KIND_EVO ? gsig[(cc + 1) % (KIND == KIND_EVO ? DV : 1)] : inv;
            packed[cc / 2] = ptx::pack_bf16x2(__uint_as_float(o[2 * q]) * f0, __uint_as_float(o[2 * q + 1]) * f1);
          }
        }
        lse_off = (static_cast<int64_t>(e.b) * p.Hq + e.hq) * p.Lq + e.i;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&o_empty[s]);  // O may be overwritten by the next unit
      if (tre) FL_TR(3, e.uc, 2);
      // row r of the tile: 16-byte chunks at the swizzled positions
      constexpr int ROWB = L::ROWB_V;                       // bytes per row of one box
      constexpr int NBOX = OUT_COLS * 2 / ROWB;
      constexpr uint32_t SWM = ROWB == 128 ? 7u : (ROWB == 64 ? 3u : 1u);
      const int qi = static_cast<int>(e.uc % L::QBUF) * 2 + s;
      uint8_t* stage = smem + L::OFF_Q + qi * L::Q_BYTES;
#pragma unroll
      for (int bx = 0; bx < NBOX; ++bx)
#pragma unroll
        for (int c = 0; c < ROWB / 16; ++c) {
          uint32_t off = static_cast<uint32_t>(r * ROWB + c * 16);
          off ^= ((off >> 7) & SWM) << 4;
          const int w = bx * (ROWB / 4) + 4 * c;
          *reinterpret_cast<uint4*>(stage + bx * kBlockM * ROWB + off) =
              make_uint4(packed[w], packed[w + 1], packed[w + 2], packed[w + 3]);
        }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&o_staged[s]);
      if (e.i < p.Lq && p.lse && e.valid) p.lse[lse_off] = lse2 * kLn2;
      if (leader) {
        const bool w_ok = wait_bar(&o_staged[s], e.uc & 1u, ctl, 34 + s);
        if (w_ok) {
          if (e.valid) {
#pragma unroll
            for (int bx = 0; bx < NBOX; ++bx)
              ptx::tma_store_4d(&tmO, stage + bx * kBlockM * ROWB,
                                (KIND == KIND_DIFF ? s * OUT_COLS : 0) + bx * (ROWB / 2), e.row0, e.hq, e.b);
            ptx::bulk_commit_group();
          }
          pending_qi = qi;
          if (!kDefer) release_pending();
        }
      }
      if (tre) FL_TR(3, e.uc, 3);
      return __all_sync(0xffffffffu, !*ctl.abort);
    };

    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++uc) {
      if (lane == 0 && warp == 2) FL_TR(3, 32 + uc, 0);
      if (!__all_sync(0xffffffffu, wait_bar(&q_full[(uc % L::QBUF) * 2 + s], (uc / L::QBUF) & 1u, ctl, 27))) {
        ok = false;
        break;
      }
      const Unit U = units[uc & 3u];
      if (lane == 0 && warp == 2) FL_TR(3, 32 + uc, 1);
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
      if (lane == 0 && warp == 2) FL_TR(3, 32 + uc, 2);
      if (kSepP && s == 1 && uc == 0 && !__all_sync(0xffffffffu, wait_bar(stagger, 0u, ctl, 26))) {
        ok = false;
        break;
      }
      for (int t = 0; t < n; ++t, ++scnt) {
        const int j0 = (U.kv_hi - t) * kBlockN;
        if (kDefer) release_pending();
        const bool tr = lane == 0 && (warp == 2 || warp == 6);
        if (tr) FL_TR(1 + s, scnt, 0);
        if (!__all_sync(0xffffffffu, wait_bar(&s_full[s], scnt & 1u, ctl, 20 + s))) { ok = false; break; }
        if (tr) FL_TR(1 + s, scnt, 1);
        ptx::tc_fence_after();
        // Plain scores stay raw until the exponent, where the scale is
        // folded into one FMA: p = 2^(s * scale_log2 - m).
        constexpr bool kRaw = SCORE == SCORE_NONE && KIND != KIND_EVO;
        float x[kBlockN];
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          ptx::tmem_ld32(tS + 0, r0);
          ptx::tmem_ld32(tS + 32, r1);
          ptx::tmem_ld32(tS + 64, r2);
          ptx::tmem_ld32(tS + 96, r3);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(r0);
          ptx::reg_fence32(r1);
          ptx::reg_fence32(r2);
          ptx::reg_fence32(r3);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(r0[e]);
            x[32 + e] = __uint_as_float(r1[e]);
            x[64 + e] = __uint_as_float(r2[e]);
            x[96 + e] = __uint_as_float(r3[e]);
          }
        }
        if (tr) FL_TR(1 + s, scnt, 2);
        // S is in registers: its TMEM columns may take the next tile's S
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s_free[s]);
        const float2 c1 = make_float2(scale_log2, scale_log2);
        // does any row of this warp see only part of this key tile?
        const bool need_mask = __any_sync(0xffffffffu, (j0 < lo) || (j0 + kBlockN - 1 > hi));
        float tmax_fast = 0.f;  // softcap: the tile max from the max raw score (tanh is monotonic)
        // score transform into the log2 domain
        if (SCORE == SCORE_ALIBI) {
          // x = s * scale_log2 + slope_log2 * (j - i)
          // bias of columns (c, c+1) kept in four running pairs, each
          // advanced by 8 columns: no per-column constants
          const float base = slope2 * static_cast<float>(j0 - ic);
          float2 bias[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            bias[k] = make_float2(fmaf(slope2, static_cast<float>(2 * k), base),
                                  fmaf(slope2, static_cast<float>(2 * k + 1), base));
          const float2 step = make_float2(8.f * slope2, 8.f * slope2);
#pragma unroll
          for (int c = 0; c < kBlockN; c += 2) {
            const int k = (c >> 1) & 3;
            const float2 r = ptx::fma2(make_float2(x[c], x[c + 1]), c1, bias[k]);
            bias[k] = ptx::add2(bias[k], step);
            x[c] = r.x;
            x[c + 1] = r.y;
          }
        } else if (SCORE == SCORE_SOFTCAP) {
          // t = cap * tanh(s * scale / cap), in log2 units x = cap*log2(e) * tanh(y).
          // When every |y| of the warp's rows is within the polynomial's
          // range, tanh runs on the FMA pipe; otherwise the exact form
          // tanh(y) = 1 - 2 / (1 + e^(2y)) on the MUFU pipe.
          float mx4[4], mn4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            mx4[e] = fmaxf(x[e], x[4 + e]);
            mn4[e] = fminf(x[e], x[4 + e]);
          }
#pragma unroll
          for (int c = 8; c < kBlockN; c += 8)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              mx4[e] = ptx::max3(mx4[e], x[c + e], x[c + 4 + e]);
              mn4[e] = ptx::min3(mn4[e], x[c + e], x[c + 4 + e]);
            }
          const float smax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
          const float smin = fminf(fminf(mn4[0], mn4[1]), fminf(mn4[2], mn4[3]));
          const float ya = scale_log2 / (kLog2e * p.softcap);   // y = s * ya
          const float kcap = p.softcap * kLog2e;
          if (__all_sync(0xffffffffu, fmaxf(smax, -smin) * ya <= kTanhPolyRange)) {
            const float2 ya2 = make_float2(ya, ya), k2 = make_float2(kcap, kcap);
            const float2 c4 = make_float2(kTanhC4, kTanhC4), c3 = make_float2(kTanhC3, kTanhC3);
            const float2 c2 = make_float2(kTanhC2, kTanhC2), c1v = make_float2(kTanhC1, kTanhC1);
            const float2 one = make_float2(1.f, 1.f);
#pragma unroll
            for (int c = 0; c < kBlockN; c += 2) {
              const float2 y = ptx::mul2(make_float2(x[c], x[c + 1]), ya2);
              const float2 z = ptx::mul2(y, y);
              float2 q = ptx::fma2(c4, z, c3);
              q = ptx::fma2(q, z, c2);
              q = ptx::fma2(q, z, c1v);
              q = ptx::fma2(q, z, one);
              const float2 r = ptx::mul2(ptx::mul2(y, k2), q);
              x[c] = r.x;
              x[c + 1] = r.y;
            }
            const float ym = smax * ya, zm = ym * ym;
            tmax_fast = kcap * ym * fmaf(fmaf(fmaf(fmaf(kTanhC4, zm, kTanhC3), zm, kTanhC2), zm, kTanhC1), zm, 1.f);
          } else {
            const float a = 2.0f * ya * kLog2e;   // 2 * y * log2(e) = s * a
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) {
              const float e = ptx::ex2(x[c] * a);
              x[c] = fmaf(-2.0f * kcap, ptx::rcp(1.0f + e), kcap);
            }
            tmax_fast = fmaf(-2.0f * kcap, ptx::rcp(1.0f + ptx::ex2(smax * a)), kcap);
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
            const float2 l2e = make_float2(kLog2e, kLog2e);
            const float2 r0 = ptx::fma2(make_float2(x[4 * c4], x[4 * c4 + 1]), c1,
                                        ptx::mul2(ptx::add2(make_float2(pb.x, pb.y), make_float2(mb.x, mb.y)), l2e));
            const float2 r1 = ptx::fma2(make_float2(x[4 * c4 + 2], x[4 * c4 + 3]), c1,
                                        ptx::mul2(ptx::add2(make_float2(pb.z, pb.w), make_float2(mb.z, mb.w)), l2e));
            x[4 * c4] = r0.x; x[4 * c4 + 1] = r0.y; x[4 * c4 + 2] = r1.x; x[4 * c4 + 3] = r1.y;
          }
        }
        // mask (only when some row of this warp has a partially visible tile)
        if (need_mask) {
          const int clo = lo - j0, chi = hi - j0;
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (c < clo || c > chi) x[c] = -CUDART_INF_F;
        }
        // row max (three-input max tree)
        float tmax;
        if (SCORE == SCORE_SOFTCAP && !need_mask) {
          tmax = tmax_fast;
        } else {
          float mx[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = fmaxf(x[e], x[8 + e]);
#pragma unroll
          for (int c = 16; c < kBlockN; c += 16)
#pragma unroll
            for (int e = 0; e < 8; ++e) mx[e] = ptx::max3(mx[e], x[c + e], x[c + 8 + e]);
          tmax = ptx::max3(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
          if (kRaw) tmax *= scale_log2;
        }
        // raise the reference max only when the tile's max exceeds it by more
        // than the threshold (or it is the first finite max of the row);
        // alpha = 2^(m_old - m_new) is 0 when m_old = -inf
        const float m_new = fmaxf(m, tmax);
        const bool raise = m_new > m + kRescaleThreshold || (m == -CUDART_INF_F && m_new != -CUDART_INF_F);
        const float alpha = raise ? ptx::ex2(m - m_new) : 1.f;
        m = raise ? m_new : m;
        l *= alpha;
        // stagger (once per block): slot 1 starts once slot 0 is past its
        // first row max, so the two slots' exponent phases (MUFU-bound)
        // alternate with their max phases instead of coinciding; each slot's
        // pipeline is independent afterwards, so the offset persists
        if (kSepP && s == 0 && scnt == 0) {
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(stagger);
        }
        if (tr) FL_TR(1 + s, scnt, 3);
        // the previous P V of this slot must be done before P (and O) change
        if (pc > 0 && !__all_sync(0xffffffffu, wait_bar(&pv_done[s], (pc - 1) & 1u, ctl, 24 + s))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (tr) FL_TR(1 + s, scnt, 4);
        const float msub = (m == -CUDART_INF_F) ? 0.f : m;
        const float2 negm = make_float2(-msub, -msub);
        float2 ls[2];
        ls[0] = ls[1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 xv = make_float2(x[h * 32 + 2 * e], x[h * 32 + 2 * e + 1]);
            const float2 arg = kRaw ? ptx::fma2(xv, c1, negm) : ptx::add2(xv, negm);
            const float2 pv = make_float2(ptx::ex2(arg.x), ptx::ex2(arg.y));
            ls[e & 1] = ptx::add2(ls[e & 1], pv);
            pk[e] = ptx::pack_bf16x2(pv.x, pv.y);
          }
          ptx::tmem_st16(tP + h * 16, pk);
        }
        const float2 lsum = ptx::add2(ls[0], ls[1]);
        l += lsum.x + lsum.y;
        if (tr) FL_TR(1 + s, scnt, 5);
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
        if (tr) FL_TR(1 + s, scnt, 6);
        ++pc;
        if (kDefer && t == 0 && have_prev) {
          have_prev = false;
          if (!epilogue(prev)) { ok = false; break; }
        }
      }
      if (!ok) break;
      if (lane == 0 && warp == 2) FL_TR(3, 32 + uc, 3);
      {
        const Epi cur{U.b, U.hq[s], U.row0[s], U.valid[s], i, uc, pc - 1, m, l};
        if (kDefer) {
          prev = cur;
          have_prev = true;
        } else if (!epilogue(cur)) {
          ok = false;
          break;
        }
      }
    }
    if (ok && have_prev) ok = epilogue(prev);
    if (leader && pending_qi >= 0) ptx::bulk_wait_group_read0();  // the buffer outlives no store
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace fl
