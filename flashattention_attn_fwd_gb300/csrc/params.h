// Kernel-side problem description shared by the host launcher and the
// device code.  Plain data only.
#pragma once

#include <cstdint>

namespace fl {

// KIND_ATTN    : softmax(score_mod(scale QK^T) + mask) V, MHA / GQA
// KIND_DIFF    : differential attention (two Q/K branches, one V)
// KIND_EVO     : Evoformer MSA row-wise gated attention (pair bias shared by
//                the MSA rows, residue mask bias, sigmoid gate)
// KIND_EVO_COL : Evoformer MSA column-wise gated attention (attention over
//                the MSA rows of each residue column, mask bias, gate)
enum Kind : int { KIND_ATTN = 0, KIND_DIFF = 1, KIND_EVO = 2, KIND_EVO_COL = 3 };
enum ScoreMod : int { SCORE_NONE = 0, SCORE_ALIBI = 1, SCORE_SOFTCAP = 2 };
enum MaskKind : int { MASK_NONE = 0, MASK_CAUSAL = 1, MASK_WINDOW = 2, MASK_PREFIX = 3, MASK_DOC = 4 };

// How the two query tiles ("slots") of one work unit are chosen.
//   SLOT_ROWS   : query row tiles 2t and 2t+1 of one head (MHA)
//   SLOT_HEADS  : the same row tile of two query heads of one GQA group
//   SLOT_BRANCH : the same rows of the two branches of differential attention
//   SLOT_PAIR   : the same rows of two independent problems with their own
//                 K/V (Evoformer: two MSA rows, or two residue columns)
enum SlotMode : int { SLOT_ROWS = 0, SLOT_HEADS = 1, SLOT_BRANCH = 2, SLOT_PAIR = 3 };

constexpr int kBlockM = 128;  // query rows per slot (one TMEM lane per row)
constexpr int kBlockN = 128;  // keys per key/value tile
// Softmax threads per query row (1: each thread holds a whole 128-score row;
// 2: two threads per row, each with half of it, exchanging their maxima).
#ifndef FL_ROW_SPLIT
#define FL_ROW_SPLIT 1
#endif
constexpr int kRowSplit = FL_ROW_SPLIT;
static_assert(kRowSplit == 1 || kRowSplit == 2, "threads per row");
constexpr int kHalfCols = kBlockN / kRowSplit;  // scores of one row held by one softmax thread
// Warpgroup 0 = warp 0 TMA, warps 1 / 2 MMA issue, warp 3 idle; then the
// softmax warpgroups of slot 0 and of slot 1 (4 * kRowSplit warps each).
constexpr int kSoftmaxWarps = 8 * kRowSplit;
constexpr int kThreads = 128 + 32 * kSoftmaxWarps;
// Registers per thread: at launch (65536 / kThreads rounded down to a
// multiple of 8), then after setmaxnreg for the control warpgroup and the
// softmax warpgroups; their total stays within the launch's.
constexpr int kLaunchRegs = kRowSplit == 1 ? 168 : 96;
constexpr int kCtlRegs = kRowSplit == 1 ? 56 : 32;
constexpr int kSoftmaxRegs = kRowSplit == 1 ? 224 : 112;
static_assert(128 * kCtlRegs + 32 * kSoftmaxWarps * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split");

// Key-split units (two slots on the same query rows, halves of the key
// range) need one MMA thread per slot (DV <= 64), the output tile staged in
// a Q buffer (DV <= D), one softmax thread per row, and a ring of at least
// three stages (a slot's next own tile is two ring positions ahead of the
// one it still holds), which D <= 64 leaves room for.
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr bool key_split_ok(int d, int dv) { return dv <= d && d <= 64 && kRowSplit == 1; }

struct KParams {
  // problem (Evoformer row-wise: B is B * N_seq, Hq == Hkv == H;
  // column-wise: Hq == Hkv == H * N_res, rows are MSA rows)
  int B, Hq, Hkv, Lq, Lk;
  int group;            // Hq / Hkv
  int n_qtiles;         // ceil(Lq / 128)
  int slot_mode;
  int pairs_per_group;  // SLOT_HEADS: ceil(group / 2)
  int num_units;
  int chunked;          // 1: each CTA takes a contiguous range of units
  // The last ks_count units are key-split units (attention, DV <= 64): unit
  // num_units - ks_count + j takes query tile (j & 1) of base unit
  // num_units - ks_count + (j >> 1) and walks its key range in two halves,
  // one per slot, merged in the epilogue.  0: none.
  int ks_count;
  float scale_log2;     // scale * log2(e)
  float scale;          // scale (natural units; Evoformer)

  // mask
  int mask_kind, doc_causal, window, prefix;
  const int32_t* doc_offsets;
  int num_docs;

  // score mod
  const float* slopes;  // ALiBi slopes, natural units
  float softcap;
  // softcap on the FMA pipe: x = s * (q0 + q1 s^2 + q2 s^4 + q3 s^6) (log2
  // units) while |s| <= sc_smax
  float sc_q[4];
  float sc_smax;

  // outputs; out strides in elements for (b, h, l), channel stride 1
  void* out;
  int64_t o_sb, o_sh, o_sl;
  float* lse;           // [B, Hq, Lq]; differential: [2, B, H, L]

  // differential attention
  float lambda;

  // Evoformer
  int evo_b;            // batch of the Evoformer call
  int evo_h;            // heads H
  int evo_n;            // the paired axis: N_seq (row-wise) or N_res (column-wise)
  int has_pb, has_mb;
  const void* gate;     // same layout as out

  // control
  uint32_t* status;     // device status word (bit 0: timeout), [1]: where
  uint64_t timeout_ns;
  int dbg_skip_tile;    // < 0: off
  // Phase timestamps of block 0 (builds with -DFL_TRACE only): [role 6][tile 64][event 8]
  unsigned long long* trace;
};

}  // namespace fl
