// Fused single-pass attention forward for sm_103a (GB300).
//
// One persistent CTA per SM walks a static list of work units.  A unit is
// two 128-row query tiles ("slots") that share the key/value tiles the load
// warp brings in; per key tile the work is
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
// Warp roles (384 threads, three warpgroups):
//   warp 0      one thread issues TMA loads: Q once per unit, K/V tiles (and
//               the Evoformer bias tiles) into an mbarrier-guarded ring
//   warp 1      allocates TMEM; one thread issues slot 0's tcgen05.mma
//               (with DV = 128: both slots' MMAs)
//   warp 2      one thread issues slot 1's tcgen05.mma (DV <= 64)
//   warps 4-7   softmax for slot 0, one thread per query row
//   warps 8-11  softmax for slot 1
// The control warpgroup gives registers to the softmax warpgroups
// (setmaxnreg), which hold a whole 128-score row per thread.
//
// TMEM columns (512 allocated): S0 [0,128), S1 [128,256).  For DV <= 64 the
// bf16 P of each slot has its own 64 columns (P0 [256,320), P1 [320,384))
// and O0, O1 follow; the next tile's S is then issued as soon as the softmax
// warps have pulled the current S into registers.  For DV = 128 P
// overwrites the first 64 columns of S and O0, O1 start at column 256.
//
// Each slot walks only the key tiles its own rows can see (per-slot ranges,
// DV <= 64); the load warp fetches the union and releases a stage on behalf
// of a slot that skips it.
//
// The online softmax keeps (m, l) per row in the log2 domain.  The
// reference max m is only raised when a new tile's max exceeds it by more
// than 8 (a factor 256), so O is rescaled rarely; O and l always use the
// same m, so the final O / l is exact whatever m was used.  Optionally
// (FL_EMU_*) a share of the exponentials is evaluated on the FMA pipe
// (Cody-Waite split plus a fitted cubic) instead of the MUFU unit; on sm_103a
// the MUFU unit keeps up with the tensor core at d = 64, so the share is 0 by
// default.
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
// set KParams::trace): role 0/1 = MMA thread of slot 0/1, 2/3 = softmax of
// slot 0/1 (lane 0 of its first warp), 4 = epilogue and unit events, 5 = TMA
// thread; up to 64 tiles, 8 events each.
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

// 2^f ~= E(f) on [0, 1), cubic with minimax relative error (fit_poly.py exp2
// 3: float32 max relative error 7.5e-5, below bf16's half ulp of 2^-9).
constexpr float kExp2E0 = 0.999925196f;
constexpr float kExp2E1 = 0.695833504f;
constexpr float kExp2E2 = 0.2260672f;
constexpr float kExp2E3 = 0.0780244842f;
// 1.5 * 2^23 + 127: x + kExp2Magic rounded down holds floor(x) + 127 in its
// low mantissa bits for -127 <= x < 128, which shifted left by 23 is the
// bit pattern of 2^floor(x).
constexpr float kExp2Magic = 12583039.0f;

// Pairs of columns (of 16 per 32-column chunk) whose exponentials run on the
// FMA pipe, by kernel kind and score modification.
#ifndef FL_EMU_PLAIN
#define FL_EMU_PLAIN 0
#endif
#ifndef FL_EMU_ALIBI
#define FL_EMU_ALIBI 0
#endif
#ifndef FL_EMU_SOFTCAP
#define FL_EMU_SOFTCAP 0
#endif
#ifndef FL_EMU_EVO
#define FL_EMU_EVO 0
#endif
template <int KIND, int SCORE>
struct EmuPairs {
  static constexpr int value = (KIND == KIND_EVO || KIND == KIND_EVO_COL) ? FL_EMU_EVO
                               : SCORE == SCORE_ALIBI                   ? FL_EMU_ALIBI
                               : SCORE == SCORE_SOFTCAP                 ? FL_EMU_SOFTCAP
                                                                        : FL_EMU_PLAIN;
  static_assert(value >= 0 && value <= 16, "share of FMA-pipe exponentials");
};

// In units where both slots walk the same key tiles, the two slots'
// exponent phases can take turns: a slot waits for the other slot's previous
// phase to end, so that each slot's loads, maxima and waits overlap the other
// slot's exponentials.  It only orders work: the wait gives up quietly after
// kTurnWaitNs.  Left alone, the slots' phases drift into lockstep within a
// few tiles and then contend for the MUFU unit; the turns pay off only where
// the transform phase is long (softcap), so they are on for softcap and,
// with FL_PINGPONG=1, for every score_mod.
#ifndef FL_PINGPONG
#define FL_PINGPONG 0
#endif
constexpr uint64_t kTurnWaitNs = 1500;

template <int D, int DV, int KIND, int SCORE = SCORE_NONE>
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
  static constexpr bool PAIR = KIND == KIND_EVO || KIND == KIND_EVO_COL;
  static constexpr int NK = (KIND == KIND_DIFF || PAIR) ? 2 : 1;  // K tiles per stage
  static constexpr int NV = PAIR ? 2 : 1;                          // V tiles per stage
  // Evoformer row-wise: the pair-bias tile [128 query rows][128 keys] fp32,
  // as four TMA boxes of 32 columns with the 128-byte swizzle.
  static constexpr int PB_BYTES = KIND == KIND_EVO ? kBlockM * kBlockN * 4 : 0;
  static constexpr int PB_BOX_BYTES = kBlockM * 128;
  // Evoformer: one 128-key row of the mask bias per slot.
  static constexpr int MB_BYTES = PAIR ? 2 * kBlockN * 4 : 0;
  static constexpr int STAGE_BYTES = NK * K_BYTES + NV * V_BYTES + PB_BYTES + MB_BYTES;
  // barriers, misc words, the differential-attention exchange, the unit ring
  static constexpr int UNIT_BYTES = 128;
  static constexpr int XCH_BYTES = KIND == KIND_DIFF ? 2 * kBlockM * 4 : 0;     // differential: row sums
  static constexpr int XM_BYTES = kRowSplit == 2 ? 12 * kBlockM * 4 : 0;         // two threads per row
  // ALiBi on the tensor core: one extra k-step of the S product, with a
  // constant key-index tile K_ext [128 keys][16] and per slot a one-row
  // tile Q_ext [8 rows][16] (read for all 128 rows) holding slope / scale
  // split into three bf16 parts; both K-major without swizzle.
  static constexpr bool EXT = KIND == KIND_ATTN && SCORE == SCORE_ALIBI;
  static constexpr int EXTK_BYTES = EXT ? kBlockN * 32 : 0;
  static constexpr int EXTQ_BYTES = EXT ? 4 * 256 : 0;  // [Q buffer][slot]
  static constexpr int FIXED_BYTES = 64 * 8 + 64 + XCH_BYTES + 4 * UNIT_BYTES + XM_BYTES + EXTK_BYTES + EXTQ_BYTES;
  static constexpr int BUDGET = 227 * 1024 - 1024 - FIXED_BYTES;
  // Q is double-buffered (the next unit's Q loads while this one runs) when
  // that still leaves room for two stages.
  static constexpr int QBUF = (4 * Q_BYTES + 2 * STAGE_BYTES <= BUDGET) ? 2 : 1;
  static constexpr int STAGES_FIT = (BUDGET - 2 * QBUF * Q_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static_assert(STAGES >= 2, "ring too small");
  static constexpr int OFF_Q = 0;                        // Q[buffer][slot]
  static constexpr int OFF_K = 2 * QBUF * Q_BYTES;       // K[stage][NK]
  static constexpr int OFF_V = OFF_K + STAGES * NK * K_BYTES;   // V[stage][NV]
  static constexpr int OFF_PB = OFF_V + STAGES * NV * V_BYTES;  // PB[stage]
  static constexpr int OFF_MB = OFF_PB + STAGES * PB_BYTES;     // MB[stage][slot]
  static constexpr int OFF_BAR = OFF_MB + STAGES * MB_BYTES;
  // barriers: q_full[4] q_empty[4] kv_full[S] kv_empty[S] s_full[2] s_free[2]
  //           p_full[2] pv_done[2] o_empty[2] drain[2] xch_full[1] stagger[1]
  //           o_staged[2] xm_bar[8] xl_bar[8] exp_turn[2] ks_full[1] p_hi[2]
  static constexpr int NBARS = 45 + 2 * STAGES;
  static_assert(NBARS <= 64, "barrier area");
  static constexpr int OFF_MISC = OFF_BAR + 64 * 8;
  static constexpr int OFF_XCH = OFF_MISC + 64;                // float [2][128]
  static constexpr int OFF_UNITS = OFF_XCH + XCH_BYTES;        // Unit[4]: decoded units, ring
  static constexpr int OFF_XMAX = OFF_UNITS + 4 * UNIT_BYTES;   // float [2 parities][2 slots][2 halves][128]
  static constexpr int OFF_XL = OFF_XMAX + 8 * kBlockM * 4;     // float [2 slots][2 halves][128]
  // Q_ext[buffer][slot] (256 bytes each), then K_ext; every address either
  // descriptor can form stays inside these 5 KB
  static constexpr int OFF_EXTQ = OFF_XMAX + XM_BYTES;
  static constexpr int OFF_EXTK = OFF_EXTQ + EXTQ_BYTES;
  static constexpr int END = OFF_EXTK + EXTK_BYTES;
  // +1 KB to align the dynamic base to 1024; at least ~117 KB so that only
  // one block (which owns all 512 TMEM columns) is resident per SM.
  static constexpr int SMEM_BYTES = (END + 1024) > 120 * 1024 ? (END + 1024) : 120 * 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static constexpr uint32_t SWZ_D = ROWB_D == 128 ? 2u : (ROWB_D == 64 ? 4u : 6u);
  static constexpr uint32_t SWZ_V = ROWB_V == 128 ? 2u : (ROWB_V == 64 ? 4u : 6u);
};

struct Unit {
  int b[2];          // batch coordinate of each slot (Evoformer row-wise: b * N_seq + s)
  int hq[2];         // query head of each slot
  int hkv[2];        // key/value head of each slot
  int row0[2];       // first query row of each slot
  int valid[2];      // slot's results are stored
  int mbrow[2];      // Evoformer: row of the mask-bias matrix
  int lo[2], hi[2];  // key tiles each slot walks (inclusive, walked from hi down)
  int kv_lo, kv_hi;  // union of the slots' ranges: the tiles the load warp fetches
  int pb_b, pb_h;    // Evoformer: pair-bias tile coordinates
  int ks;            // key-split unit: both slots hold the same query rows,
                     // slot 0 the upper and slot 1 the lower half of the key
                     // range; their tiles alternate in the ring
};
static_assert(sizeof(Unit) <= 128, "unit ring entry");

// Reads of the document offsets: through the read-only cache on the device,
// plainly on the host (the host-side schedule query gets host offsets).
__host__ __device__ __forceinline__ int32_t load_offset(const int32_t* x) {
#ifdef __CUDA_ARCH__
  return __ldg(x);
#else
  return *x;
#endif
}

// Visible keys of query row i form one interval [lo, hi] for every mask kind.
__host__ __device__ __forceinline__ void row_bounds(const KParams& p, int b, int i, int& lo, int& hi) {
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
        if (load_offset(off + mid) <= i) a = mid; else z = mid - 1;
      }
      lo = load_offset(off + a);
      hi = p.doc_causal ? i : load_offset(off + a + 1) - 1;
    }
  }
  lo = lo < 0 ? 0 : lo;
  hi = hi > p.Lk - 1 ? p.Lk - 1 : hi;
}

// Static schedule: unit indices of this CTA are first, first + step, ... < end.
struct Sched {
  int first, step, end;
};
__device__ __forceinline__ Sched make_sched(const KParams& p) {
  Sched s;
  if (p.chunked) {
    s.first = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.num_units / gridDim.x);
    s.end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.num_units / gridDim.x);
    s.step = 1;
  } else {
    s.first = blockIdx.x;
    s.end = p.num_units;
    s.step = gridDim.x;
  }
  return s;
}

// Ring position of slot s's first own tile within a unit, and the distance
// between its consecutive own tiles.
__host__ __device__ __forceinline__ int ring_first(const Unit& U, int s) { return U.ks ? s : U.kv_hi - U.hi[s]; }
__host__ __device__ __forceinline__ int ring_stride(const Unit& U) { return U.ks ? 2 : 1; }
// Key tile the load warp fetches at ring position i of a unit.
__host__ __device__ __forceinline__ int ring_tile(const Unit& U, int i) {
  return U.ks ? U.hi[i & 1] - (i >> 1) : U.kv_hi - i;
}

template <int KIND>
__host__ __device__ __forceinline__ Unit decode_base(const KParams& p, int u, bool per_slot) {
  Unit U;
  U.ks = 0;
  U.pb_b = 0;
  U.pb_h = 0;
  U.mbrow[0] = U.mbrow[1] = 0;
  if (KIND == KIND_EVO) {
    // (b, h, query tile, MSA-row pair) with the pair index fastest: a CTA's
    // consecutive units reuse the same pair-bias tiles
    const int n_pairs = (p.evo_n + 1) >> 1;
    const int sp = u % n_pairs;
    int r = u / n_pairs;
    const int qt = r % p.n_qtiles;
    r /= p.n_qtiles;
    const int h = r % p.evo_h;
    const int b = r / p.evo_h;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int idx = 2 * sp + s;
      U.valid[s] = idx < p.evo_n;
      const int row = b * p.evo_n + (U.valid[s] ? idx : 2 * sp);
      U.b[s] = row;
      U.mbrow[s] = row;
      U.hq[s] = U.hkv[s] = h;
      U.row0[s] = qt * kBlockM;
    }
    U.pb_b = b;
    U.pb_h = h;
  } else if (KIND == KIND_EVO_COL) {
    // (b, h, residue pair, query tile over the MSA rows)
    const int n_pairs = (p.evo_n + 1) >> 1;
    const int qt = u % p.n_qtiles;
    int r = u / p.n_qtiles;
    const int rp = r % n_pairs;
    r /= n_pairs;
    const int h = r % p.evo_h;
    const int b = r / p.evo_h;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int res = 2 * rp + s;
      U.valid[s] = res < p.evo_n;
      const int rr = U.valid[s] ? res : 2 * rp;
      U.b[s] = b;
      U.hq[s] = U.hkv[s] = h * p.evo_n + rr;
      U.mbrow[s] = b * p.evo_n + rr;
      U.row0[s] = qt * kBlockM;
    }
  } else if (p.slot_mode == SLOT_ROWS) {
    const int per = p.B * p.Hq;
    const int n_pairs = (p.n_qtiles + 1) >> 1;
    const int tp = n_pairs - 1 - u / per;  // heaviest (last rows) first
    const int rem = u % per;
    const int b = rem / p.Hq;
    const int h = rem % p.Hq;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      U.b[s] = b;
      U.hq[s] = h;
      U.hkv[s] = h / p.group;
      U.row0[s] = (2 * tp + s) * kBlockM;
    }
    U.valid[0] = 1;
    U.valid[1] = (2 * tp + 1) < p.n_qtiles;
  } else if (p.slot_mode == SLOT_HEADS) {
    const int per = p.B * p.Hkv * p.pairs_per_group;
    const int t = p.n_qtiles - 1 - u / per;
    int rem = u % per;
    const int b = rem / (p.Hkv * p.pairs_per_group);
    rem %= (p.Hkv * p.pairs_per_group);
    const int hkv = rem / p.pairs_per_group;
    const int pair = rem % p.pairs_per_group;
    U.valid[0] = 1;
    U.valid[1] = (2 * pair + 1) < p.group;
    U.hq[0] = hkv * p.group + 2 * pair;
    U.hq[1] = U.valid[1] ? U.hq[0] + 1 : U.hq[0];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      U.b[s] = b;
      U.hkv[s] = hkv;
      U.row0[s] = t * kBlockM;
    }
  } else {  // SLOT_BRANCH
    const int per = p.B * p.Hq;
    const int t = p.n_qtiles - 1 - u / per;
    const int rem = u % per;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      U.b[s] = rem / p.Hq;
      U.hq[s] = U.hkv[s] = rem % p.Hq;
      U.row0[s] = t * kBlockM;
      U.valid[s] = 1;
    }
  }
  int lo_min = 0x7fffffff, hi_max = -1;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    U.lo[s] = 0;
    U.hi[s] = -1;
    if (!U.valid[s] || U.row0[s] >= p.Lq) continue;
    const int r1 = min(U.row0[s] + kBlockM - 1, p.Lq - 1);
    int lo, hi, lo2, hi2;
    row_bounds(p, U.b[s], U.row0[s], lo, hi);
    row_bounds(p, U.b[s], r1, lo2, hi2);
    lo = min(lo, lo2);
    hi = max(hi, hi2);
    if (hi < lo) { lo = 0; hi = 0; }  // keep >= 1 tile
    U.lo[s] = lo / kBlockN;
    U.hi[s] = hi / kBlockN;
    lo_min = min(lo_min, U.lo[s]);
    hi_max = max(hi_max, U.hi[s]);
  }
  if (hi_max < 0) { lo_min = 0; hi_max = 0; }
  U.kv_lo = lo_min;
  U.kv_hi = hi_max;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    // a slot with no rows of its own runs one tile (its results are dropped);
    // without per-slot ranges both slots walk the union
    if (!per_slot) {
      U.lo[s] = lo_min;
      U.hi[s] = hi_max;
    } else if (U.hi[s] < U.lo[s]) {
      U.lo[s] = U.hi[s] = hi_max;
    }
  }
  return U;
}

// Work unit u.  A key-split unit (the last ks_count units) takes one query
// tile of a base unit and hands each slot half of that tile's key range:
// slot 0 the upper ceil(n/2) tiles, slot 1 the lower floor(n/2); the
// epilogue merges the two partial (m, l, O) of every row.  A tile with a
// single key tile (or a padding tile) is not split: it runs as a unit whose
// second slot is a dropped copy of the first.
template <int KIND>
__host__ __device__ __forceinline__ Unit decode_unit(const KParams& p, int u, bool per_slot) {
  const int ks_first = p.num_units - p.ks_count;
  if (KIND != KIND_ATTN || !per_slot || u < ks_first) return decode_base<KIND>(p, u, per_slot);
  const int j = u - ks_first;
  Unit U = decode_base<KIND>(p, ks_first + (j >> 1), per_slot);
  const bool s1 = (j & 1) != 0;
  // selects rather than a runtime index: U stays in registers
  const bool real = (s1 ? U.valid[1] : U.valid[0]) && (s1 ? U.row0[1] : U.row0[0]) < p.Lq &&
                    !(p.slot_mode == SLOT_HEADS && s1 && U.hq[1] == U.hq[0]);
  const int lo = s1 ? U.lo[1] : U.lo[0], hi = s1 ? U.hi[1] : U.hi[0];
  U.b[0] = U.b[1] = s1 ? U.b[1] : U.b[0];
  U.hq[0] = U.hq[1] = s1 ? U.hq[1] : U.hq[0];
  U.hkv[0] = U.hkv[1] = s1 ? U.hkv[1] : U.hkv[0];
  U.row0[0] = U.row0[1] = s1 ? U.row0[1] : U.row0[0];
  U.valid[0] = real;
  U.valid[1] = 0;
  U.kv_lo = lo;
  U.kv_hi = hi;
  const int n = hi - lo + 1;
  if (real && n >= 2) {
    const int n0 = (n + 1) >> 1;
    U.ks = 1;
    U.lo[0] = hi - n0 + 1;
    U.hi[0] = hi;
    U.lo[1] = lo;
    U.hi[1] = lo + (n - n0) - 1;
  } else {
    U.ks = 0;
    U.lo[0] = U.lo[1] = lo;
    U.hi[0] = U.hi[1] = hi;
  }
  return U;
}

// ------------------------------------------------------------ bounded waits
struct Ctl {
  volatile uint32_t* abort;
  uint32_t* status;
  uint64_t timeout_ns;
};

#ifndef FL_SPIN_TEST
#define FL_SPIN_TEST 0
#endif
static __device__ __forceinline__ bool wait_slow(uint64_t* bar, uint32_t parity, const Ctl& c, int where) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#if FL_SPIN_TEST
    if (ptx::mbar_test_wait(bar, parity)) return true;
#else
    if (ptx::mbar_try_wait(bar, parity)) return true;
#endif
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
#if FL_SPIN_TEST
  if (ptx::mbar_test_wait(bar, parity)) return true;
#else
  if (ptx::mbar_try_wait(bar, parity)) return true;
#endif
  return wait_slow(bar, parity, c, where);
}

// Wait that gives up quietly after `limit_ns` (used for scheduling hints,
// where proceeding early is always correct): true if the phase completed.
static __device__ __forceinline__ bool wait_soft(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Drain wait used after an abort: ignores the abort flag, gives up after limit.
static __device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) return;
  }
}

// ------------------------------------------------------------ exponentials
// 2^a on the FMA pipe for a <= 128: a = j + f with j = floor(a) (round-down
// add of a magic constant), 2^f from the fitted cubic, 2^j by building the
// exponent bits; a below -127 is clamped (2^-127 is 0 after the scaling).
__device__ __forceinline__ float2 exp2_fma(float2 a) {
  a.x = fmaxf(a.x, -127.0f);
  a.y = fmaxf(a.y, -127.0f);
  const float2 mg = make_float2(kExp2Magic, kExp2Magic);
  const float2 t = ptx::add2_rm(a, mg);
  const float2 f = ptx::sub2(a, ptx::sub2(t, mg));
  float2 e = ptx::fma2(make_float2(kExp2E3, kExp2E3), f, make_float2(kExp2E2, kExp2E2));
  e = ptx::fma2(e, f, make_float2(kExp2E1, kExp2E1));
  e = ptx::fma2(e, f, make_float2(kExp2E0, kExp2E0));
  const float2 sc = make_float2(__uint_as_float(__float_as_uint(t.x) << 23), __uint_as_float(__float_as_uint(t.y) << 23));
  return ptx::mul2(e, sc);
}

// ------------------------------------------------------------------ kernel
template <int D, int DV, int KIND, int SCORE>
__global__ void __launch_bounds__(kThreads, 1)
    fused_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ0, const __grid_constant__ CUtensorMap tmK0,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ1,
                          const __grid_constant__ CUtensorMap tmK1, const __grid_constant__ CUtensorMap tmO,
                          const __grid_constant__ CUtensorMap tmPB, const __grid_constant__ CUtensorMap tmMB,
                          const __grid_constant__ KParams p) {
  using L = Layout<D, DV, KIND, SCORE>;
  constexpr int S = L::STAGES;
  constexpr bool kEvo = KIND == KIND_EVO || KIND == KIND_EVO_COL;
  // TMEM columns: S0 [0,128) S1 [128,256); with DV <= 64 a separate P region
  // P0 [256,320) P1 [320,384) and O0, O1 from 384; with DV = 128 P is
  // written over the first 64 columns of S and O0, O1 start at 256.
  constexpr bool kSepP = DV <= 64;
  // ALiBi's bias enters S through one extra k-step (see Layout::EXT)
  constexpr bool kAlibiExt = L::EXT;
  // P handed to the tensor core in two halves of 64 keys: the first half's
  // P V runs while the softmax warps compute the second half's exponentials
  constexpr bool kSplitP = kSepP && kRowSplit == 1;
  constexpr uint32_t kColP = kSepP ? 256u : 0u;   // + 64 * slot (sep) or + 128 * slot (aliased)
  constexpr uint32_t kColO = kSepP ? 384u : 256u;
  // per-slot key ranges need one MMA thread per slot
  constexpr bool kPerSlot = kSepP;

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
  uint64_t* xm_bar = bars + 24 + 2 * S;    // [slot * 4 + quad]: half-row maxima exchanged
  uint64_t* xl_bar = bars + 32 + 2 * S;    // [slot * 4 + quad]: half-row sums exchanged
  uint64_t* exp_turn = bars + 40 + 2 * S;  // [slot]: the other slot's exponent phase is over
  uint64_t* ks_full = bars + 42 + 2 * S;   // key-split unit: slot 1's (m, l) published
  uint64_t* p_hi = bars + 43 + 2 * S;      // [slot]: P of the tile's upper 64 keys in TMEM (kSplitP)
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  float* xch = reinterpret_cast<float*>(smem + L::OFF_XCH);
  // The TMA thread decodes each unit once and publishes it here before
  // arriving on the unit's q_full barriers (release); the MMA and softmax
  // threads read it after waiting on q_full (acquire).  A ring of 4 suffices:
  // the TMA thread runs at most two units ahead (two Q buffers).
  auto unit_at = [&](uint32_t ucn) -> Unit& {
    return *reinterpret_cast<Unit*>(smem + L::OFF_UNITS + (ucn & 3u) * L::UNIT_BYTES);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Sched sch = make_sched(p);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(&q_full[i], 1);
      ptx::mbar_init(&q_empty[i], 1);
    }
    for (int st = 0; st < S; ++st) {
      ptx::mbar_init(&kv_full[st], 1);
      ptx::mbar_init(&kv_empty[st], 2);  // one arrival per slot
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s_full[i], 1);
      ptx::mbar_init(&s_free[i], kSoftmaxWarps / 2);
      ptx::mbar_init(&p_full[i], kSoftmaxWarps / 2);
      ptx::mbar_init(&pv_done[i], 1);
      ptx::mbar_init(&o_empty[i], kSoftmaxWarps / 2);
      ptx::mbar_init(&drain[i], 1);
    }
    ptx::mbar_init(xch_full, kSoftmaxWarps);
    ptx::mbar_init(stagger, kSoftmaxWarps / 2);
    ptx::mbar_init(&o_staged[0], kSoftmaxWarps / 2);
    ptx::mbar_init(&o_staged[1], kSoftmaxWarps / 2);
    for (int i = 0; i < 8; ++i) {
      ptx::mbar_init(&xm_bar[i], 2);
      ptx::mbar_init(&xl_bar[i], 2);
    }
    ptx::mbar_init(&exp_turn[0], kSoftmaxWarps / 2);
    ptx::mbar_init(&exp_turn[1], kSoftmaxWarps / 2);
    ptx::mbar_init(ks_full, kSoftmaxWarps / 2);
    ptx::mbar_init(&p_hi[0], kSoftmaxWarps / 2);
    ptx::mbar_init(&p_hi[1], kSoftmaxWarps / 2);
    misc[1] = 0u;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&misc[0], 512);
    ptx::tmem_relinquish();
  }
  if (kAlibiExt && threadIdx.x < kBlockN) {
    // K_ext row c: channels 0..2 hold the key index c within its tile (exact
    // in bf16), the rest zero; 8-row core matrices of 16-byte rows, the two
    // channel halves 128 bytes apart, row groups 256 bytes apart
    const int c = threadIdx.x;
    uint8_t* row = smem + L::OFF_EXTK + (c >> 3) * 256 + (c & 7) * 16;
    const float fc = static_cast<float>(c);
    *reinterpret_cast<uint4*>(row) = make_uint4(ptx::pack_bf16x2(fc, fc), ptx::pack_bf16x2(fc, 0.f), 0u, 0u);
    *reinterpret_cast<uint4*>(row + 128) = make_uint4(0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmQ0); ptx::prefetch_tensormap(&tmK0); ptx::prefetch_tensormap(&tmV);
    ptx::prefetch_tensormap(&tmO);
    if (KIND == KIND_DIFF) { ptx::prefetch_tensormap(&tmQ1); ptx::prefetch_tensormap(&tmK1); }
    if (KIND == KIND_EVO && p.has_pb) ptx::prefetch_tensormap(&tmPB);
    if (kEvo && p.has_mb) ptx::prefetch_tensormap(&tmMB);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const Ctl ctl{reinterpret_cast<volatile uint32_t*>(&misc[1]), p.status, p.timeout_ns};
  const uint64_t drain_ns = 50ull * 1000ull * 1000ull;

  if (warp < 4) {
  ptx::setmaxnreg_dec<kCtlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA load
    if (lane == 0) {
      const uint64_t pol_stream = ptx::policy_evict_first();
      const uint64_t pol_reuse = ptx::policy_evict_last();
      uint32_t it = 0, uc = 0;
      uint32_t kv_count = 0;               // K/V stage loads issued so far (ring order)
      int64_t skipped = -1;                // ring index whose K load was skipped (debug)
      int q_iss[4] = {-1, -1, -1, -1};     // phase of the latest Q load per buffer
      // Evoformer: which pair-bias tile each stage holds (b, h, query tile, key tile)
      int* pb_tag = reinterpret_cast<int*>(misc + 8);
      for (int st = 0; st < S; ++st) pb_tag[st] = -1;
      constexpr uint32_t kStageTx = L::NK * L::K_BYTES + L::NV * L::V_BYTES;
      for (int u = sch.first; u < sch.end; u += sch.step, ++uc) {
        unit_at(uc) = decode_unit<KIND>(p, u, kPerSlot);
        const Unit& U = unit_at(uc);  // fields are read back from shared memory
        const uint32_t qb = uc % L::QBUF, qph = (uc / L::QBUF) & 1u;
        bool ok = true;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const int qi = static_cast<int>(qb) * 2 + s;
          if (!wait_bar(&q_empty[qi], qph ^ 1u, ctl, 1)) { ok = false; break; }
          if (kAlibiExt) {
            // Q_ext of this slot: a = slope / scale as three bf16 parts
            // (a = h1 + h2 + h3 to within 2^-24 relative), the same in all 8
            // rows of the core matrix that every row group reads
            const float a = __ldg(p.slopes + U.hq[s]) / p.scale;
            const float h1 = __bfloat162float(__float2bfloat16_rn(a));
            const float h2 = __bfloat162float(__float2bfloat16_rn(a - h1));
            const float h3 = __bfloat162float(__float2bfloat16_rn(a - h1 - h2));
            const uint4 w = make_uint4(ptx::pack_bf16x2(h1, h2), ptx::pack_bf16x2(h3, 0.f), 0u, 0u);
            uint8_t* qe = smem + L::OFF_EXTQ + qi * 256;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              *reinterpret_cast<uint4*>(qe + 16 * i) = w;
              *reinterpret_cast<uint4*>(qe + 128 + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
            }
            ptx::fence_proxy_async_smem();
          }
          ptx::mbar_arrive_expect_tx(&q_full[qi], L::Q_BYTES);
          const CUtensorMap* mq = (KIND == KIND_DIFF && s == 1) ? &tmQ1 : &tmQ0;
#pragma unroll
          for (int bx = 0; bx < L::NBOX_D; ++bx)
            ptx::tma_load_4d(smem + L::OFF_Q + qi * L::Q_BYTES + bx * L::BOX_D_BYTES, mq, &q_full[qi],
                             bx * L::BOXW_D, U.row0[s], U.hq[s], U.b[s], pol_stream);
          q_iss[qi] = static_cast<int>(qph);
        }
        if (!ok) break;
        const int n_ring = U.kv_hi - U.kv_lo + 1;
        for (int i = 0; i < n_ring; ++i, ++it) {
          const int t = ring_tile(U, i);
          const int st = static_cast<int>(it % S);
          const uint32_t ph = (it / S) & 1u;
          FL_TR(5, it, 0);
          if (!wait_bar(&kv_empty[st], ph ^ 1u, ctl, 2)) { ok = false; break; }
          FL_TR(5, it, 1);
          const bool skip = p.dbg_skip_tile >= 0 && blockIdx.x == 0 && uc == 0 && i == p.dbg_skip_tile;
          int tag = -1;
          bool load_pb = false;
          if (KIND == KIND_EVO && p.has_pb) {
            tag = ((U.pb_b * p.evo_h + U.pb_h) * p.n_qtiles + U.row0[0] / kBlockM) * p.n_qtiles + t;
            load_pb = pb_tag[st] != tag;
          }
          const uint32_t tx = kStageTx + (load_pb ? static_cast<uint32_t>(L::PB_BYTES) : 0u) +
                              ((L::MB_BYTES > 0 && p.has_mb) ? static_cast<uint32_t>(L::MB_BYTES) : 0u);
          ptx::mbar_arrive_expect_tx(&kv_full[st], tx);
          if (!skip) {
#pragma unroll
            for (int kk = 0; kk < L::NK; ++kk) {
              const CUtensorMap* mk = (KIND == KIND_DIFF && kk == 1) ? &tmK1 : &tmK0;
#pragma unroll
              for (int bx = 0; bx < L::NBOX_D; ++bx)
                ptx::tma_load_4d(smem + L::OFF_K + (st * L::NK + kk) * L::K_BYTES + bx * L::BOX_D_BYTES, mk,
                                 &kv_full[st], bx * L::BOXW_D, t * kBlockN, U.hkv[kk], U.b[kk], pol_reuse);
            }
          } else {
            skipped = it;  // this stage's barrier never completes: the waits on it run out
          }
#pragma unroll
          for (int vv = 0; vv < L::NV; ++vv)
#pragma unroll
            for (int bx = 0; bx < L::NBOX_V; ++bx)
              ptx::tma_load_4d(smem + L::OFF_V + (st * L::NV + vv) * L::V_BYTES + bx * L::BOX_V_BYTES, &tmV,
                               &kv_full[st], bx * L::BOXW_V, t * kBlockN, U.hkv[vv], U.b[vv], pol_reuse);
          if (KIND == KIND_EVO && load_pb) {
#pragma unroll
            for (int bx = 0; bx < 4; ++bx)
              ptx::tma_load_4d(smem + L::OFF_PB + st * L::PB_BYTES + bx * L::PB_BOX_BYTES, &tmPB, &kv_full[st],
                               t * kBlockN + 32 * bx, U.row0[0], U.pb_h, U.pb_b, pol_reuse);
            pb_tag[st] = tag;
          }
          if (L::MB_BYTES > 0 && p.has_mb) {
#pragma unroll
            for (int s = 0; s < 2; ++s)
              ptx::tma_load_2d(smem + L::OFF_MB + st * L::MB_BYTES + s * kBlockN * 4, &tmMB, &kv_full[st],
                               t * kBlockN, U.mbrow[s], pol_reuse);
          }
          // release the stage on behalf of a slot that does not use this tile
#pragma unroll
          for (int s = 0; s < 2; ++s)
            if (U.ks ? s != (i & 1) : (t < U.lo[s] || t > U.hi[s])) ptx::mbar_arrive(&kv_empty[st]);
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
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(kBlockM, kBlockN, false);
    constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(kBlockM, DV, true);
    const uint32_t q_base = ptx::smem_u32(smem + L::OFF_Q);
    const uint32_t k_base = ptx::smem_u32(smem + L::OFF_K);
    const uint32_t v_base = ptx::smem_u32(smem + L::OFF_V);
    const uint32_t qext_base = ptx::smem_u32(smem + L::OFF_EXTQ);
    const uint32_t kext_base = ptx::smem_u32(smem + L::OFF_EXTK);
    uint32_t sf[2] = {0u, 0u};

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
      if (kAlibiExt) {
        // + (slope / scale) * (key index in the tile), no swizzle, K-major:
        // core matrices 128 bytes apart along k; Q_ext's row groups all
        // alias one core matrix (stride 0), K_ext's are 256 bytes apart
        const uint64_t qe = ptx::smem_desc(qext_base + (qb * 2 + s) * 256, 128, 0, 0u);
        const uint64_t ke = ptx::smem_desc(kext_base, 128, 256, 0u);
        ptx::mma_ss(tmem + s * 128, qe, ke, IDESC_S, 1u);
      }
      ptx::mma_commit(&s_full[s]);
      ++sf[s];
      return true;
    };
    auto issue_pv = [&](int s, int st, bool acc, int kb0 = 0, int kb1 = kBlockN / 16) {
      const uint32_t va = v_base + (st * L::NV + (L::NV == 2 ? s : 0)) * L::V_BYTES;
      const uint64_t bd0 = ptx::smem_desc(va, L::BOX_V_BYTES, 8 * L::ROWB_V, L::SWZ_V);
      const uint32_t tP = tmem + (kSepP ? kColP + s * 64 : s * 128);
      const uint32_t tO = tmem + kColO + s * DV;
#pragma unroll
      for (int kb = kb0; kb < kb1; ++kb)
        ptx::mma_ts(tO, tP + kb * 8, bd0 + ((kb * 16 * L::ROWB_V) >> 4), IDESC_O, (acc || kb > 0) ? 1u : 0u);
    };
    auto wait_q = [&](uint32_t ucn, int s) -> bool {
      return wait_bar(&q_full[(ucn % L::QBUF) * 2 + s], (ucn / L::QBUF) & 1u, ctl, 10);
    };

    if (kSepP && lane == 0) {
      // One thread per slot (warp 1: slot 0, warp 2: slot 1).  Per own tile:
      // the next S as soon as the softmax warps have pulled the current S
      // into registers (s_free) and its K tile is in (kv_full); P V as soon
      // as P is in TMEM (p_full).  The first S of the next unit is issued
      // during the last tile of the current one (two Q buffers) when the
      // ring distance allows it.
      const int s = warp - 1;
      constexpr bool kCross = L::QBUF == 2;
      uint32_t it = 0, uc = 0, pc = 0;
      bool ok = true;
      int u = sch.first;
      auto first_idx = [&](const Unit& V, uint32_t base) -> uint32_t {
        return base + static_cast<uint32_t>(ring_first(V, s));
      };
      auto first_s = [&](uint32_t ucn, uint32_t idx) -> bool {
        if (!wait_bar(&kv_full[idx % S], (idx / S) & 1u, ctl, 11)) return false;
        return issue_s(s, ucn % L::QBUF, static_cast<int>(idx % S));
      };
      bool s_issued = false;  // first S of the current unit already issued
      while (ok && u < sch.end) {
        if (!wait_q(uc, s)) { ok = false; break; }
        const Unit& Us = unit_at(uc);
        const int n = Us.kv_hi - Us.kv_lo + 1;
        const int ns = Us.hi[s] - Us.lo[s] + 1;
        const uint32_t idx0 = first_idx(Us, it);
        if (!s_issued && !first_s(uc, idx0)) { ok = false; break; }
        s_issued = false;
        const uint32_t qb = uc % L::QBUF;
        const int un = u + sch.step;
        const uint32_t stride = static_cast<uint32_t>(ring_stride(Us));
        for (int k = 0; k < ns && ok; ++k) {
          const uint32_t idx = idx0 + k * stride;
          const uint32_t idn = idx + stride;
          const int st = static_cast<int>(idx % S);
          FL_TR(s, idx, 0);
          if (k + 1 < ns) {
            if (!wait_bar(&kv_full[idn % S], (idn / S) & 1u, ctl, 15)) { ok = false; break; }
            if (!issue_s(s, qb, static_cast<int>(idn % S))) { ok = false; break; }
          }
          FL_TR(s, idx, 2);
          if (k == 0 && !wait_bar(&o_empty[s], (uc & 1u) ^ 1u, ctl, 13)) { ok = false; break; }
          const uint32_t pph = pc & 1u;
          if (!wait_bar(&p_full[s], pph, ctl, 14)) { ok = false; break; }
          FL_TR(s, idx, 4);
          ++pc;
          ptx::tc_fence_after();
          if (kSplitP) {
            issue_pv(s, st, k > 0, 0, kBlockN / 32);
            if (!wait_bar(&p_hi[s], pph, ctl, 16)) { ok = false; break; }
            ptx::tc_fence_after();
            issue_pv(s, st, true, kBlockN / 32, kBlockN / 16);
          } else {
            issue_pv(s, st, k > 0);
          }
          ptx::mma_commit(&pv_done[s]);
          ptx::mma_commit(&kv_empty[st]);
          if (k + 1 == ns && kCross && un < sch.end) {
            // next unit's first own tile, if its ring index is less than S
            // ahead of this one (issued after the last P V, which the next
            // unit's epilogue waits for)
            if (!wait_q(uc + 1, s)) { ok = false; break; }
            const uint32_t idxn = first_idx(unit_at(uc + 1), it + n);
            if (idxn - idx < static_cast<uint32_t>(S)) {
              if (!first_s(uc + 1, idxn)) { ok = false; break; }
              s_issued = true;
            }
          }
        }
        it += n;
        ++uc;
        u = un;
      }
      // every MMA this thread issued must finish before TMEM is released
      ptx::mma_commit(&drain[s]);
      wait_drain(&drain[s], 0u, drain_ns);
    } else if (!kSepP && warp == 1 && lane == 0) {
      // P written over S (DV = 128): one thread alternates the slots --
      // P V(0), S(0, next), P V(1), S(1, next) -- so the two softmax
      // warpgroups stay half a tile apart; both slots walk every tile.
      uint32_t it = 0, uc = 0;
      uint32_t pc[2] = {0u, 0u};
      auto first_s = [&](uint32_t ucn, uint32_t itn) -> bool {
        const int st = static_cast<int>(itn % S);
        if (!wait_q(ucn, 0) || !wait_q(ucn, 1) || !wait_bar(&kv_full[st], (itn / S) & 1u, ctl, 11)) return false;
        return issue_s(0, ucn % L::QBUF, st) && issue_s(1, ucn % L::QBUF, st);
      };
      bool ok = true;
      int u = sch.first;
      if (u < sch.end) ok = first_s(0u, 0u);
      while (u < sch.end && ok) {
        const int n = unit_at(uc).kv_hi - unit_at(uc).kv_lo + 1;
        const uint32_t qb = uc % L::QBUF;
        for (int t = 0; t < n && ok; ++t) {
          const uint32_t itc = it + t;
          const int st = static_cast<int>(itc % S);
          const bool more = t + 1 < n;
          const int stn = static_cast<int>((itc + 1) % S);
          const uint32_t phn = ((itc + 1) / S) & 1u;
          for (int s = 0; s < 2; ++s) {
            if (t == 0) {
              if (!wait_bar(&o_empty[s], (uc & 1u) ^ 1u, ctl, 13)) { ok = false; break; }
              if (KIND == KIND_DIFF && !wait_bar(&o_empty[s ^ 1], (uc & 1u) ^ 1u, ctl, 13)) { ok = false; break; }
            }
            if (!wait_bar(&p_full[s], pc[s] & 1u, ctl, 14)) { ok = false; break; }
            ++pc[s];
            ptx::tc_fence_after();
            issue_pv(s, st, t > 0);
            ptx::mma_commit(&pv_done[s]);
            ptx::mma_commit(&kv_empty[st]);
            if (more) {
              if (s == 0 && !wait_bar(&kv_full[stn], phn, ctl, 15)) { ok = false; break; }
              if (!issue_s(s, qb, stn)) { ok = false; break; }
            }
          }
        }
        it += n;
        ++uc;
        u += sch.step;
        if (ok && u < sch.end) ok = first_s(uc, it);
      }
      ptx::mma_commit(&drain[0]);
      wait_drain(&drain[0], 0u, drain_ns);
    }
    __syncwarp();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  } else {
    // ------------------------------------------------------------ softmax
    // 4 * kRowSplit warps per slot: the warp with lane quarter `quad` and
    // part `half` holds kHalfCols scores of 32 rows.  With two threads per
    // row (kRowSplit = 2) the two threads of a row exchange
    // their half-row maxima through shared memory once per tile and their
    // partial sums once per unit (an mbarrier per pair of warps, so that
    // every wait stays bounded).
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    const int sw = warp - 4;                 // softmax warp
    const int s = sw / (4 * kRowSplit);      // slot
    const int quad = sw & 3;                 // TMEM lane quarter (= warp % 4)
    const int half = (sw >> 2) & (kRowSplit - 1);  // part of the row (two threads per row)
    const int r = quad * 32 + lane;
    const int c_off = half * kHalfCols;      // first score column of this thread
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t tS = tl + s * 128 + c_off;
    const uint32_t tP = tl + (kSepP ? kColP + s * 64 : s * 128) + half * (kHalfCols / 2);
    constexpr int OUT_COLS = KIND == KIND_DIFF ? DV / 2 : DV;  // output columns of one slot
    constexpr int OUT_H = OUT_COLS / kRowSplit;                // ... of one thread
    const uint32_t tO = tl + kColO + s * DV;
    float* xmax = reinterpret_cast<float*>(smem + L::OFF_XMAX);   // [parity][slot][half][row]
    float* xl = reinterpret_cast<float*>(smem + L::OFF_XL);       // [slot][half][row]
    const float scale_log2 = p.scale_log2;
    // Scores stay in the units of the transform until the exponent: raw S
    // (plain scores, and ALiBi, whose column term comes with S: the scale is
    // folded into the exponent's FMA), natural units (Evoformer: scale q.k +
    // biases), log2 units otherwise (softcap).
    constexpr bool kRaw = SCORE == SCORE_NONE && !kEvo;
    const float xmul = (kRaw || kAlibiExt) ? scale_log2 : (kEvo ? kLog2e : 1.0f);
    constexpr int kEmu = EmuPairs<KIND, SCORE>::value;
    uint32_t scnt = 0, uc = 0, it = 0;
    uint32_t kscnt = 0;  // slot 0: key-split merges done so far
    uint32_t pc = 0;  // P tiles handed to the MMA warp so far (= P V launched for this slot)
    constexpr bool kPingPong = kPerSlot && (FL_PINGPONG || SCORE == SCORE_SOFTCAP);
    uint32_t tcnt = 0;  // exponent phases taken in turns so far
    bool ok = true;

    // What the epilogue of a unit needs once its tile loop is over (the
    // unit's own fields are read again from the ring, which keeps them until
    // the load warp is two units further on).
    struct Epi {
      uint32_t uc, pcl;  // unit counter; index of the unit's last P V completion
      float m, l;
      int ns;            // this slot's tiles in the unit
    };
    // With two Q buffers the epilogue of a unit runs when the next unit
    // starts (its last P V completes meanwhile, and the next unit's first S
    // is already issued), and the bulk store's hold on the staging buffer is
    // released at the next tile instead of being waited for.
    constexpr bool kDefer = L::QBUF == 2;
    // Output tile of one slot: staged in the slot's Q buffer and stored by
    // TMA when it fits (DV <= D, or half the channels for differential
    // attention), else written by each thread straight to global memory.
    // Evoformer row-wise (one Q buffer) stores directly instead, so that
    // its Q buffer is free as soon as the unit's last S is done and the next
    // unit's Q loads while this one finishes.
    constexpr bool kTmaOut = KIND != KIND_EVO && OUT_COLS * 2 * kBlockM <= L::Q_BYTES;
    constexpr bool kEarlyQ = !kTmaOut && KIND == KIND_EVO;
    // key-split units (attention only; the host enables them only where
    // key_split_ok holds)
    constexpr bool kKs = KIND == KIND_ATTN && key_split_ok(D, DV);
    static_assert(!kKs || (kPerSlot && kTmaOut && kRowSplit == 1 && S >= 3),
                  "key split needs per-slot MMA, staged output and three ring stages");
    const bool leader = lane == 0 && sw == 4 * kRowSplit * s;
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
      const bool tre = lane == 0 && sw == 0;
      if (tre) FL_TR(4, e.uc, 0);
      const Unit& Ue = unit_at(e.uc);
      const int e_b = Ue.b[s], e_hq = Ue.hq[s], e_row0 = Ue.row0[s], e_valid = Ue.valid[s];
      const int e_i = e_row0 + r;
      // the row's sum: this thread's part plus its partner's
      float lrow = e.l;
      if (kRowSplit == 2) {
        xl[(s * 2 + half) * kBlockM + r] = e.l;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&xl_bar[s * 4 + quad]);
        if (!__all_sync(0xffffffffu, wait_bar(&xl_bar[s * 4 + quad], e.uc & 1u, ctl, 37))) return false;
        lrow += xl[(s * 2 + (half ^ 1)) * kBlockM + r];
      }
      // O is final once the unit's last P V is done
      if (!__all_sync(0xffffffffu, wait_bar(&pv_done[s], e.pcl & 1u, ctl, 30 + s))) return false;
      if (KIND == KIND_DIFF && !__all_sync(0xffffffffu, wait_bar(&pv_done[s ^ 1], e.pcl & 1u, ctl, 30 + s)))
        return false;
      ptx::tc_fence_after();
      // log2 domain
      const float lse2 = (lrow > 0.f) ? (e.m + __log2f(lrow)) : -CUDART_INF_F;
      uint32_t packed[OUT_H / 2];
      int64_t lse_off;
      const int64_t orow_off = e_b * p.o_sb + e_hq * p.o_sh + static_cast<int64_t>(e_i) * p.o_sl;
      if (KIND == KIND_DIFF) {
        // Each branch's softmax warps publish l for their rows, then each
        // slot produces half of the output channels of O1/l1 - lambda O2/l2
        // (each thread a quarter).  xch is rewritten only in the next unit's
        // epilogue, which needs the next unit's P V, hence the MMA warp's
        // wait on both o_empty barriers, which each slot arrives on only
        // after its reads below.
        if (half == 0) xch[s * kBlockM + r] = lrow;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(xch_full);
        if (!__all_sync(0xffffffffu, wait_bar(xch_full, e.uc & 1u, ctl, 32))) return false;
        const float l0 = xch[r];
        const float l1 = xch[kBlockM + r];
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float inv1 = l1 > 0.f ? -p.lambda / l1 : 0.f;
        const int col0 = s * OUT_COLS + half * OUT_H;
        const uint32_t tO0 = tl + kColO + col0, tO1 = tl + kColO + DV + col0;
#pragma unroll
        for (int c = 0; c < OUT_H; c += 32) {
          uint32_t a[32], bq[32];
          ptx::tmem_ld32(tO0 + c, a);
          ptx::tmem_ld32(tO1 + c, bq);
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
        lse_off = static_cast<int64_t>(s) * p.B * p.Hq * p.Lq + (static_cast<int64_t>(e_b) * p.Hq + e_hq) * p.Lq + e_i;
      } else {
        const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
        float gsig[kEvo ? OUT_H : 1];
        if (kEvo) {
          // out = sigmoid(gate) * O / l, sigmoid(g) = (1 + tanh(g / 2)) / 2 (one MUFU op)
          const bool row_ok = e_i < p.Lq && e_valid;
          const uint4* g4 = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.gate) + orow_off +
                                                           half * OUT_H);
#pragma unroll
          for (int q = 0; q < OUT_H / 8; ++q) {
            const uint4 gv = row_ok ? __ldg(g4 + q) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[w]));
              gsig[8 * q + 2 * w] = fmaf(0.5f, ptx::tanh_approx(0.5f * gf.x), 0.5f) * inv;
              gsig[8 * q + 2 * w + 1] = fmaf(0.5f, ptx::tanh_approx(0.5f * gf.y), 0.5f) * inv;
            }
          }
        }
        // this thread's O columns in chunks of up to 64, 16 or 32 columns per
        // load, all loads of a chunk before one wait
        constexpr int CH = OUT_H <= 64 ? OUT_H : 64;
        constexpr int CW = CH >= 32 ? 32 : 16;
#pragma unroll
        for (int c0 = 0; c0 < OUT_H; c0 += CH) {
          uint32_t o[CH];
#pragma unroll
          for (int c = 0; c < CH; c += CW) {
            if (CW == 32) ptx::tmem_ld32(tO + half * OUT_H + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(&o[c]));
            else ptx::tmem_ld16(tO + half * OUT_H + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(&o[c]));
          }
          ptx::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < CH; c += CW) {
            if (CW == 32) ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&o[c]));
            else ptx::reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(&o[c]));
          }
#pragma unroll
          for (int q = 0; q < CH / 2; ++q) {
            const int cc = c0 + 2 * q;
            const float f0 = kEvo ? gsig[cc % (kEvo ? OUT_H : 1)] : inv;
            const float f1 = kEvo ? gsig[(cc + 1) % (kEvo ? OUT_H : 1)] : inv;
            packed[cc / 2] = ptx::pack_bf16x2(__uint_as_float(o[2 * q]) * f0, __uint_as_float(o[2 * q + 1]) * f1);
          }
        }
        lse_off = (static_cast<int64_t>(e_b) * p.Hq + e_hq) * p.Lq + e_i;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&o_empty[s]);  // O may be overwritten by the next unit
      if (tre) FL_TR(4, e.uc, 2);
      if (half == 0 && e_i < p.Lq && p.lse && e_valid) p.lse[lse_off] = lse2 * kLn2;
      const int qi = static_cast<int>(e.uc % L::QBUF) * 2 + s;
      if (kTmaOut) {
        // this thread's part of row r: 16-byte chunks at the swizzled positions
        constexpr int ROWB = L::ROWB_V;                       // bytes per row of one box
        constexpr int NBOX = OUT_COLS * 2 / ROWB;
        constexpr int BOXC = ROWB / 2;                        // columns per box
        constexpr uint32_t SWM = ROWB == 128 ? 7u : (ROWB == 64 ? 3u : 1u);
        uint8_t* stage = smem + L::OFF_Q + qi * L::Q_BYTES;
#pragma unroll
        for (int q = 0; q < OUT_H / 8; ++q) {
          const int col = half * OUT_H + 8 * q;
          uint32_t off = static_cast<uint32_t>(r * ROWB + (col % BOXC) * 2);
          off ^= ((off >> 7) & SWM) << 4;
          *reinterpret_cast<uint4*>(stage + (col / BOXC) * kBlockM * ROWB + off) =
              make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&o_staged[s]);
        if (leader) {
          const bool w_ok = wait_bar(&o_staged[s], e.uc & 1u, ctl, 34 + s);
          if (w_ok) {
            if (e_valid) {
#pragma unroll
              for (int bx = 0; bx < NBOX; ++bx)
                ptx::tma_store_4d(&tmO, stage + bx * kBlockM * ROWB,
                                  (KIND == KIND_DIFF ? s * OUT_COLS : 0) + bx * BOXC, e_row0, e_hq, e_b);
              ptx::bulk_commit_group();
            }
            pending_qi = qi;
            if (!kDefer) release_pending();
          }
        }
      } else {
        // direct 16-byte stores of this thread's part of its row
        if (e_i < p.Lq && e_valid) {
          uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow_off + half * OUT_H);
#pragma unroll
          for (int c = 0; c < OUT_H / 8; ++c)
            orow[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        }
        // this unit's Q buffer is free once both halves of every row are past
        // their last use of it (the last S was done before the last P V);
        // released in the tile loop already when the slot had tiles
        if (leader && (!kEarlyQ || e.ns == 0)) ptx::mbar_arrive(&q_empty[qi]);
      }
      if (tre) FL_TR(4, e.uc, 3);
      return __all_sync(0xffffffffu, !*ctl.abort);
    };

    // Epilogue of a key-split unit, run right after the unit's last tile
    // (never deferred; only tail units are split).  Slot 1 hands its row
    // (m, l) to slot 0 through its own Q buffer (idle: its last S is done)
    // and leaves O1 in TMEM; slot 0 rescales both halves to the larger
    // reference max, merges them, stores the tile, and releases slot 1's O
    // columns and Q buffer.
    auto epilogue_ks = [&](const Epi& e) -> bool {
      const Unit& Ue = unit_at(e.uc);
      if (!__all_sync(0xffffffffu, wait_bar(&pv_done[s], e.pcl & 1u, ctl, 30 + s))) return false;
      ptx::tc_fence_after();
      const int qi = static_cast<int>(e.uc % L::QBUF) * 2;  // slot 0's Q buffer; slot 1's is qi + 1
      float* xq = reinterpret_cast<float*>(smem + L::OFF_Q + (qi + 1) * L::Q_BYTES);
      if (s == 1) {
        xq[r] = e.m;
        xq[kBlockM + r] = e.l;
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&o_staged[1]);  // one phase per unit, as in the other units
          ptx::mbar_arrive(ks_full);
        }
        return __all_sync(0xffffffffu, !*ctl.abort);
      }
      if (!__all_sync(0xffffffffu, wait_bar(ks_full, kscnt & 1u, ctl, 38))) return false;
      ++kscnt;
      ptx::tc_fence_after();
      const float m1 = xq[r], l1 = xq[kBlockM + r];
      const float mrow = fmaxf(e.m, m1);
      const float w0 = e.m == -CUDART_INF_F ? 0.f : ptx::ex2(e.m - mrow);
      const float w1 = m1 == -CUDART_INF_F ? 0.f : ptx::ex2(m1 - mrow);
      const float lrow = e.l * w0 + l1 * w1;
      const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
      const float k0 = w0 * inv, k1 = w1 * inv;
      // O = (O0 w0 + O1 w1) / l, O1 in the columns after O0
      uint32_t packed[DV / 2];
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        uint32_t a[32], b1[32];
        ptx::tmem_ld32(tO + c0, a);
        ptx::tmem_ld32(tO + DV + c0, b1);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(a);
        ptx::reg_fence32(b1);
#pragma unroll
        for (int q = 0; q < 16; ++q)
          packed[c0 / 2 + q] =
              ptx::pack_bf16x2(fmaf(__uint_as_float(b1[2 * q]), k1, __uint_as_float(a[2 * q]) * k0),
                               fmaf(__uint_as_float(b1[2 * q + 1]), k1, __uint_as_float(a[2 * q + 1]) * k0));
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&o_empty[0]);
        ptx::mbar_arrive(&o_empty[1]);
      }
      const int e_i = Ue.row0[0] + r;
      if (e_i < p.Lq && p.lse && Ue.valid[0])
        p.lse[(static_cast<int64_t>(Ue.b[0]) * p.Hq + Ue.hq[0]) * p.Lq + e_i] =
            (lrow > 0.f ? mrow + __log2f(lrow) : -CUDART_INF_F) * kLn2;
      // the tile through slot 0's staging buffer, as in the epilogue above
      constexpr int ROWB = L::ROWB_V;
      constexpr int BOXC = ROWB / 2;
      constexpr uint32_t SWM = ROWB == 128 ? 7u : (ROWB == 64 ? 3u : 1u);
      uint8_t* stage = smem + L::OFF_Q + qi * L::Q_BYTES;
#pragma unroll
      for (int q = 0; q < DV / 8; ++q) {
        const int col = 8 * q;
        uint32_t off = static_cast<uint32_t>(r * ROWB + (col % BOXC) * 2);
        off ^= ((off >> 7) & SWM) << 4;
        *reinterpret_cast<uint4*>(stage + (col / BOXC) * kBlockM * ROWB + off) =
            make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&o_staged[0]);
      if (leader && wait_bar(&o_staged[0], e.uc & 1u, ctl, 34)) {
        if (Ue.valid[0]) {
#pragma unroll
          for (int bx = 0; bx < DV / BOXC; ++bx)
            ptx::tma_store_4d(&tmO, stage + bx * kBlockM * ROWB, bx * BOXC, Ue.row0[0], Ue.hq[0], Ue.b[0]);
          ptx::bulk_commit_group();
        }
        pending_qi = qi;
        // every warp of slot 0 has read (m, l) from slot 1's Q buffer
        ptx::mbar_arrive(&q_empty[qi + 1]);
        if (!kDefer) release_pending();
      }
      return __all_sync(0xffffffffu, !*ctl.abort);
    };

    for (int u = sch.first; u < sch.end && ok; u += sch.step, ++uc) {
      if (lane == 0 && sw == 0) FL_TR(4, 32 + uc, 0);
      // the previous unit's output store must have read its staging buffer
      // before the load warp can reuse that buffer for this unit's Q
      if (kDefer) release_pending();
      if (!__all_sync(0xffffffffu, wait_bar(&q_full[(uc % L::QBUF) * 2 + s], (uc / L::QBUF) & 1u, ctl, 27))) {
        ok = false;
        break;
      }
      // this slot's fields of the unit, read straight from shared memory
      const Unit& Us = unit_at(uc);
      const int u_hi = Us.hi[s], u_b = Us.b[s], u_hq = Us.hq[s], u_row0 = Us.row0[s];
      const int ns = u_hi - Us.lo[s] + 1;
      const bool turns = kPingPong && Us.lo[0] == Us.lo[1] && Us.hi[0] == Us.hi[1];
      const int n = Us.kv_hi - Us.kv_lo + 1;
      // ring index of this slot's first tile (only the Evoformer kinds read
      // the ring from here; their units are never key-split: stride 1)
      const uint32_t idx0 = it + static_cast<uint32_t>(ring_first(Us, s));
      const int i = u_row0 + r;
      const int ic = i < p.Lq ? i : p.Lq - 1;
      int lo, hi;
      row_bounds(p, u_b, ic, lo, hi);
      float slope2 = 0.f;
      if (SCORE == SCORE_ALIBI) slope2 = __ldg(p.slopes + u_hq) * kLog2e;
      float m = -CUDART_INF_F, l = 0.f;
      if (kPerSlot && s == 1 && uc == 0 && !__all_sync(0xffffffffu, wait_bar(stagger, 0u, ctl, 26))) {
        ok = false;
        break;
      }
      // the previous unit's epilogue: outside the tile loop, which stays small
      // (its last P V is done or nearly so; this unit's first S is already
      // in flight)
      if (kDefer && have_prev) {
        have_prev = false;
        if (!epilogue(prev)) {
          ok = false;
          break;
        }
      }
      for (int k = 0; k < ns; ++k, ++scnt) {
        const int t = u_hi - k;
        const int j0 = t * kBlockN + c_off;   // key of this thread's first column
        const uint32_t idx = idx0 + k;
        if (kDefer) release_pending();
        const bool tr = lane == 0 && (sw == 0 || sw == 4 * kRowSplit);
        if (tr) FL_TR(2 + s, scnt, 0);
        if (!__all_sync(0xffffffffu, wait_bar(&s_full[s], scnt & 1u, ctl, 20 + s))) { ok = false; break; }
        // the unit's last S has read this slot's Q: release the buffer
        if (kEarlyQ && k == ns - 1 && leader) ptx::mbar_arrive(&q_empty[(uc % L::QBUF) * 2 + s]);
        if (kEvo && !__all_sync(0xffffffffu, wait_bar(&kv_full[idx % S], (idx / S) & 1u, ctl, 21))) {
          ok = false;
          break;
        }
        if (tr) FL_TR(2 + s, scnt, 1);
        ptx::tc_fence_after();
        float x[kHalfCols];
        constexpr int NBLK = kHalfCols / 32;
        ptx::tmem_ld32f(tS + 0, &x[0]);
        ptx::tmem_ld_wait();
        ptx::reg_fence32f(&x[0]);
#pragma unroll
        for (int b = 1; b < NBLK; ++b) ptx::tmem_ld32f(tS + 32 * b, &x[32 * b]);
        const float2 c1 = make_float2(p.scale, p.scale);
        const uint8_t* pb_st = smem + L::OFF_PB + (idx % S) * L::PB_BYTES;
        const float* mb_st = reinterpret_cast<const float*>(smem + L::OFF_MB + (idx % S) * L::MB_BYTES) + s * kBlockN;
        float cmax[NBLK];
        // one vote per tile decides whether any block needs the mask
        const bool tile_part = __any_sync(0xffffffffu, (j0 < lo) || (j0 + kHalfCols - 1 > hi));
        // Softcap on a tile no row of the warp masks: the whole row first,
        // one range vote, then the polynomial on every score without
        // branches; it increases on its range, so the transformed row max is
        // the polynomial of the raw max.
        bool loads_done = false, row_done = false;  // row_done: the whole row is transformed
        if (SCORE == SCORE_SOFTCAP && !tile_part) {
          ptx::tmem_ld_wait();
#pragma unroll
          for (int b = 1; b < NBLK; ++b) ptx::reg_fence32f(&x[32 * b]);
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&s_free[s]);
          loads_done = true;
          float hi4[4], lo4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi4[e] = fmaxf(x[e], x[4 + e]);
            lo4[e] = fminf(x[e], x[4 + e]);
          }
#pragma unroll
          for (int c = 8; c < kHalfCols; c += 8)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              hi4[e] = ptx::max3(hi4[e], x[c + e], x[c + 4 + e]);
              lo4[e] = ptx::min3(lo4[e], x[c + e], x[c + 4 + e]);
            }
          const float shi = fmaxf(fmaxf(hi4[0], hi4[1]), fmaxf(hi4[2], hi4[3]));
          const float slo = fminf(fminf(lo4[0], lo4[1]), fminf(lo4[2], lo4[3]));
          row_done = __all_sync(0xffffffffu, shi <= p.sc_smax && slo >= -p.sc_smax);
          if (row_done) {
            const float2 sq0 = make_float2(p.sc_q[0], p.sc_q[0]), sq1 = make_float2(p.sc_q[1], p.sc_q[1]);
            const float2 sq2 = make_float2(p.sc_q[2], p.sc_q[2]), sq3 = make_float2(p.sc_q[3], p.sc_q[3]);
#pragma unroll
            for (int c = 0; c < kHalfCols; c += 2) {
              const float2 sv = make_float2(x[c], x[c + 1]);
              const float2 z = ptx::mul2(sv, sv);
              float2 q = ptx::fma2(sq3, z, sq2);
              q = ptx::fma2(q, z, sq1);
              q = ptx::fma2(q, z, sq0);
              const float2 v = ptx::mul2(sv, q);
              x[c] = v.x;
              x[c + 1] = v.y;
            }
            const float z = shi * shi;
            const float tm = shi * fmaf(fmaf(fmaf(p.sc_q[3], z, p.sc_q[2]), z, p.sc_q[1]), z, p.sc_q[0]);
#pragma unroll
            for (int b = 0; b < NBLK; ++b) cmax[b] = tm;
          }
        }
        // ALiBi (its bias already in S) and plain scores on such a tile: the
        // same whole-row form (one max tree instead of four blocks)
        if ((SCORE == SCORE_ALIBI || kRaw) && !tile_part) {
          ptx::tmem_ld_wait();
#pragma unroll
          for (int b = 1; b < NBLK; ++b) ptx::reg_fence32f(&x[32 * b]);
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&s_free[s]);
          loads_done = true;
          float mx[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) mx[e] = fmaxf(x[e], x[4 + e]);
#pragma unroll
          for (int c = 8; c < kHalfCols; c += 8)
#pragma unroll
            for (int e = 0; e < 4; ++e) mx[e] = ptx::max3(mx[e], x[c + e], x[c + 4 + e]);
          const float tm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
#pragma unroll
          for (int b = 0; b < NBLK; ++b) cmax[b] = tm;
          row_done = true;
        }
        // Score transform and max, 32 columns at a time: the first block
        // while the others are still being read from TMEM.
#pragma unroll
        for (int hf = 0; hf < NBLK && !row_done; ++hf) {
          const int c0 = hf * 32;
          if (hf == 1 && !loads_done) {
            ptx::tmem_ld_wait();
#pragma unroll
            for (int b = 1; b < NBLK; ++b) ptx::reg_fence32f(&x[32 * b]);
            // S is in registers: its TMEM columns may take the next tile's S
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s_free[s]);
          }
          if (SCORE == SCORE_SOFTCAP) {
            // x = cap*log2(e) * tanh(s * scale / cap): an odd polynomial in
            // s on the FMA pipe when every |s| of the warp's block is within
            // its range, else the exact form 1 - 2 / (1 + e^(2y)).
            float am[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) am[e] = fmaxf(fabsf(x[c0 + e]), fabsf(x[c0 + 4 + e]));
#pragma unroll
            for (int c = c0 + 8; c < c0 + 32; c += 8)
#pragma unroll
              for (int e = 0; e < 4; ++e) am[e] = ptx::max3(am[e], fabsf(x[c + e]), fabsf(x[c + 4 + e]));
            const float amax = fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3]));
            if (__all_sync(0xffffffffu, amax <= p.sc_smax)) {
              // x = s * (q0 + q1 s^2 + q2 s^4 + q3 s^6)
              const float2 sq0 = make_float2(p.sc_q[0], p.sc_q[0]), sq1 = make_float2(p.sc_q[1], p.sc_q[1]);
              const float2 sq2 = make_float2(p.sc_q[2], p.sc_q[2]), sq3 = make_float2(p.sc_q[3], p.sc_q[3]);
#pragma unroll
              for (int c = c0; c < c0 + 32; c += 2) {
                const float2 sv = make_float2(x[c], x[c + 1]);
                const float2 z = ptx::mul2(sv, sv);
                float2 q = ptx::fma2(sq3, z, sq2);
                q = ptx::fma2(q, z, sq1);
                q = ptx::fma2(q, z, sq0);
                const float2 v = ptx::mul2(sv, q);
                x[c] = v.x;
                x[c + 1] = v.y;
              }
            } else {
              const float kcap = p.softcap * kLog2e;
              const float a2 = 2.0f * scale_log2 / p.softcap;  // 2 y log2(e) = s * a2
#pragma unroll
              for (int c = c0; c < c0 + 32; ++c) {
                const float ez = ptx::ex2(x[c] * a2);
                x[c] = fmaf(-2.0f * kcap, ptx::rcp(1.0f + ez), kcap);
              }
            }
          }
          if (kEvo) {
            // natural units: x = scale * s + pair_bias + mask_bias; the pair
            // bias tile is swizzled (16-byte chunk q of row r at q ^ (r & 7))
            const bool hpb = KIND == KIND_EVO && p.has_pb;
            const bool hmb = p.has_mb;
#pragma unroll
            for (int c = c0; c < c0 + 32; c += 4) {
              float4 pb = make_float4(0.f, 0.f, 0.f, 0.f), mb = pb;
              const int cc = c_off + c;  // column within the 128-key tile
              if (hpb) {
                const int bx = cc >> 5, cq = (cc & 31) >> 2;
                pb = ptx::lds128(pb_st + bx * L::PB_BOX_BYTES + r * 128 + ((cq ^ (r & 7)) << 4));
              }
              if (hmb) mb = ptx::lds128(mb_st + cc);
              float2 v0 = ptx::fma2(make_float2(x[c], x[c + 1]), c1, make_float2(pb.x, pb.y));
              float2 v1 = ptx::fma2(make_float2(x[c + 2], x[c + 3]), c1, make_float2(pb.z, pb.w));
              v0 = ptx::add2(v0, make_float2(mb.x, mb.y));
              v1 = ptx::add2(v1, make_float2(mb.z, mb.w));
              x[c] = v0.x; x[c + 1] = v0.y; x[c + 2] = v1.x; x[c + 3] = v1.y;
            }
          }
          // mask (only when some row of this warp sees part of this block)
          if (tile_part && __any_sync(0xffffffffu, (j0 + c0 < lo) || (j0 + c0 + 31 > hi))) {
            const int clo = lo - j0, chi = hi - j0;
#pragma unroll
            for (int c = c0; c < c0 + 32; ++c)
              if (c < clo || c > chi) x[c] = -CUDART_INF_F;
          }
          // block max (three-input max tree)
          float mx[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) mx[e] = fmaxf(x[c0 + e], x[c0 + 4 + e]);
#pragma unroll
          for (int c = c0 + 8; c < c0 + 32; c += 8)
#pragma unroll
            for (int e = 0; e < 4; ++e) mx[e] = ptx::max3(mx[e], x[c + e], x[c + 4 + e]);
          cmax[hf] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        }
        // the row max: this thread's columns (and its partner's)
        float rmax = cmax[0];
#pragma unroll
        for (int b = 1; b < NBLK; ++b) rmax = fmaxf(rmax, cmax[b]);
        if (kRowSplit == 2) {
          const int par = static_cast<int>(scnt & 1u);
          xmax[((par * 2 + s) * 2 + half) * kBlockM + r] = rmax;
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&xm_bar[s * 4 + quad]);
          if (!__all_sync(0xffffffffu, wait_bar(&xm_bar[s * 4 + quad], scnt & 1u, ctl, 36))) { ok = false; break; }
          rmax = fmaxf(rmax, xmax[((par * 2 + s) * 2 + (half ^ 1)) * kBlockM + r]);
        }
        if (tr) FL_TR(2 + s, scnt, 2);
        // ALiBi: the row's term slope * (j0 - i) of this tile, in log2 units
        const float dlt = kAlibiExt ? slope2 * static_cast<float>(j0 - ic) : 0.f;
        const float tmax = rmax * xmul + dlt;
        // raise the reference max only when the tile's max exceeds it by more
        // than the threshold (or it is the first finite max of the row);
        // alpha = 2^(m_old - m_new) is 0 when m_old = -inf
        const float m_new = fmaxf(m, tmax);
        const bool raise = m_new > m + kRescaleThreshold || (m == -CUDART_INF_F && m_new != -CUDART_INF_F);
        float alpha = 1.f;
        if (__any_sync(0xffffffffu, raise)) {
          alpha = raise ? ptx::ex2(m - m_new) : 1.f;
          m = raise ? m_new : m;
          l *= alpha;
        }
        // stagger (once per block): slot 1 starts once slot 0 is past its
        // first row max, so the two slots' exponent phases alternate with
        // their max phases instead of coinciding
        if (kPerSlot && s == 0 && scnt == 0) {
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(stagger);
        }
        if (tr) FL_TR(2 + s, scnt, 3);
        if (turns) {
          // slot 0's k-th phase follows slot 1's (k-1)-th, slot 1's k-th
          // follows slot 0's k-th
          const uint32_t par = s == 0 ? ((tcnt & 1u) ^ 1u) : (tcnt & 1u);
          wait_soft(&exp_turn[s], par, kTurnWaitNs);
          __syncwarp();
        }
        // exponentials and the row sum; P is packed to bf16 pairs in
        // registers while this slot's previous P V may still be reading P
        const float msub = (m == -CUDART_INF_F) ? 0.f : m;
        const float2 negm = make_float2(dlt - msub, dlt - msub);
        const float2 xm2 = make_float2(xmul, xmul);
        float2 ls[2];
        ls[0] = ls[1] = make_float2(0.f, 0.f);
        uint32_t pk[kHalfCols / 2];
        // exponentials of 32-column block h: P packed to bf16 pairs, row sum
        auto expb = [&](int h) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 xv = make_float2(x[h * 32 + 2 * e], x[h * 32 + 2 * e + 1]);
            const float2 arg = ptx::fma2(xv, xm2, negm);
            float2 pv;
            if (e < kEmu) {
              pv = exp2_fma(arg);
            } else {
              pv = make_float2(ptx::ex2(arg.x), ptx::ex2(arg.y));
            }
            ls[e & 1] = ptx::add2(ls[e & 1], pv);
            pk[h * 16 + e] = ptx::pack_bf16x2(pv.x, pv.y);
          }
        };
        // blocks before the P hand-over (all of them unless P goes in halves)
        constexpr int NB1 = kSplitP ? NBLK / 2 : NBLK;
#pragma unroll
        for (int h = 0; h < NB1; ++h) expb(h);
        if (!kSplitP) {
          if (turns) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&exp_turn[s ^ 1]);
            ++tcnt;
          }
          const float2 lsum = ptx::add2(ls[0], ls[1]);
          l += lsum.x + lsum.y;
        }
        if (tr) FL_TR(2 + s, scnt, 4);
        // the previous P V of this slot must be done before P (and O) change
        if (pc > 0 && !__all_sync(0xffffffffu, wait_bar(&pv_done[s], (pc - 1) & 1u, ctl, 24 + s))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int h = 0; h < NB1; ++h)
          ptx::tmem_st16(tP + h * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[h * 16]));
        if (tr) FL_TR(2 + s, scnt, 5);
        // O rescale (this thread's half of the columns) after the P stores
        // so that x[] is dead (register pressure)
        if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          constexpr int RW = DV / kRowSplit >= 32 ? 32 : 16;
#pragma unroll
          for (int c = 0; c < DV / kRowSplit; c += RW) {
            uint32_t o[32];
            const uint32_t ta = tO + half * (DV / kRowSplit) + c;
            if (RW == 32) {
              ptx::tmem_ld32(ta, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
            } else {
              ptx::tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
            }
            ptx::tmem_ld_wait();
            if (RW == 32) ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&o[0]));
            else ptx::reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(&o[0]));
#pragma unroll
            for (int e = 0; e < RW; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            if (RW == 32) ptx::tmem_st32(ta, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
            else ptx::tmem_st16(ta, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&p_full[s]);
        if (kSplitP) {
          // the upper 64 keys while the tensor core takes the lower ones
#pragma unroll
          for (int h = NB1; h < NBLK; ++h) expb(h);
          if (turns) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&exp_turn[s ^ 1]);
            ++tcnt;
          }
          const float2 lsum = ptx::add2(ls[0], ls[1]);
          l += lsum.x + lsum.y;
#pragma unroll
          for (int h = NB1; h < NBLK; ++h)
            ptx::tmem_st16(tP + h * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[h * 16]));
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&p_hi[s]);
        }
        if (tr) FL_TR(2 + s, scnt, 6);
        ++pc;
      }
      if (!ok) break;
      it += n;
      if (lane == 0 && sw == 0) FL_TR(4, 32 + uc, 3);
      {
        const Epi cur{uc, pc - 1, m, l, ns};
        if (kKs && Us.ks) {
          if (!epilogue_ks(cur)) {
            ok = false;
            break;
          }
        } else if (kDefer) {
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
    ptx::tc_fence_before();
    __syncthreads();
  }
}

}  // namespace fl
