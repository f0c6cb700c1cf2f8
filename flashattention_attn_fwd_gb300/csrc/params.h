// Kernel-side problem description shared by the host launcher and the
// device code.  Plain data only.
#pragma once

#include <cstdint>

namespace fl {

enum Kind : int { KIND_ATTN = 0, KIND_DIFF = 1, KIND_EVO = 2 };
enum ScoreMod : int { SCORE_NONE = 0, SCORE_ALIBI = 1, SCORE_SOFTCAP = 2 };
enum MaskKind : int { MASK_NONE = 0, MASK_CAUSAL = 1, MASK_WINDOW = 2, MASK_PREFIX = 3, MASK_DOC = 4 };

// How the two query tiles ("slots") of one work unit are chosen.
//   SLOT_ROWS   : query row tiles 2t and 2t+1 of one head (MHA, Evoformer)
//   SLOT_HEADS  : the same row tile of two query heads of one GQA group
//   SLOT_BRANCH : the same rows of the two branches of differential attention
enum SlotMode : int { SLOT_ROWS = 0, SLOT_HEADS = 1, SLOT_BRANCH = 2 };

constexpr int kBlockM = 128;  // query rows per slot (one TMEM lane per row)
constexpr int kBlockN = 128;  // keys per key/value tile
// warp 0: TMA; warps 1 and 10: MMA issue for slot 0 / slot 1; warps 2-9:
// softmax (4 warps per slot)
constexpr int kThreads = 352;

struct KParams {
  // problem (for the Evoformer, B is B * N_seq and Hq == Hkv == H)
  int B, Hq, Hkv, Lq, Lk;
  int group;            // Hq / Hkv
  int n_qtiles;         // ceil(Lq / 128)
  int slot_mode;
  int pairs_per_group;  // SLOT_HEADS: ceil(group / 2)
  int num_units;
  float scale_log2;     // scale * log2(e)

  // mask
  int mask_kind, doc_causal, window, prefix;
  const int32_t* doc_offsets;
  int num_docs;

  // score mod
  const float* slopes;  // ALiBi slopes, natural units
  float softcap;

  // outputs; out strides in elements for (b, h, l), channel stride 1
  void* out;
  int64_t o_sb, o_sh, o_sl;
  float* lse;           // [B, Hq, Lq]; differential: [2, B, H, L]

  // differential attention
  float lambda;

  // Evoformer
  const float* pair_bias;   // [Bb, H, Nr, Nr]
  const float* mask_bias;   // [Bb * N_seq, Nr]
  const void* gate;         // same layout as out
  int n_seq;

  // control
  uint32_t* status;         // device status word (bit 0: timeout), [1]: where
  uint64_t timeout_ns;
  int dbg_skip_tile;        // < 0: off
  // Phase timestamps of block 0 (builds with -DFL_TRACE only): [role 4][tile 64][event 8]
  unsigned long long* trace;
};

}  // namespace fl
