/*
 * flattn -- fused attention forward for attention variants, sm_103a (GB300).
 *
 * One pass computes   out = softmax(score_mod(scale * Q K^T) + mask/bias) V
 * with an online softmax, the way the Flashlight pages describe the fused
 * kernel their compiler emits:
 *   - Flashlight technical summary (gist.science), Methodology, "Structural
 *     Fusion with Dimension Demotion" (QK^T fused with the row max),
 *     "Semantic Fusion with Algebraic Transformation" (online softmax with a
 *     running max and sum, rescaled by e^(x-y) = e^x / e^y), "Tiling-Aware
 *     Dimension Elimination and Logical Grids" (contiguous tiles, softmax(QK^T)V
 *     in one kernel); Key Contributions, "Kernel-Level Fusion".
 *   - Variant list: Flashlight wiki summary (papers.lqhl.me), 实验与结果
 *     (Vanilla, ALiBi, Softcap, Causal, Sliding Window, PrefixLM, Document
 *     Mask; MHA/GQA), and 问题与动机 / Results (differential attention,
 *     Evoformer row-wise gated self-attention).  The pages give no formula for
 *     any variant; the definitions below are this library's readings.
 *
 * Conventions shared by every entry point
 *   - Tensors are bf16 (q, k, v, gate, out) or fp32 (biases, lse), live in
 *     device memory owned by the caller, and have the head dimension
 *     contiguous.  Pointers and every non-unit stride (in bytes) must be
 *     multiples of 16 bytes (the TMA rule); otherwise FL_ERR_ALIGNMENT.
 *   - Calls are asynchronous on the given stream (NULL = legacy default
 *     stream).  Argument errors are returned before anything is launched.
 *   - Errors detected on the device (a pipeline wait that exceeded its time
 *     limit) are recorded in a per-device status word; fl_sync_status()
 *     synchronises the stream and returns and clears it.
 *   - The library allocates, once per device and on the first call that
 *     needs it, a small status word; it allocates nothing else.
 *   - lse (log-sum-exp of the final scores, natural log, fp32) may be NULL.
 *   - Query rows with no visible key produce out = 0 and lse = -inf.
 */
#ifndef FLATTN_H_
#define FLATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FL_ABI_VERSION 1

#if defined(__GNUC__)
#define FL_API __attribute__((visibility("default")))
#else
#define FL_API
#endif

typedef enum {
  FL_OK = 0,
  FL_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, bad variant field      */
  FL_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head dim 96)    */
  FL_ERR_ALIGNMENT = 3,     /* pointer or stride not 16-byte aligned           */
  FL_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed             */
  FL_ERR_TIMEOUT = 5,       /* a device-side pipeline wait hit its time limit  */
  FL_ERR_DEVICE_BOUNDS = 6  /* reserved: a device-side bounds check tripped    */
} fl_status;

typedef enum {
  FL_MASK_NONE = 0,           /* every key visible                              */
  FL_MASK_CAUSAL = 1,         /* key j visible to query i iff j <= i            */
  FL_MASK_SLIDING_WINDOW = 2, /* iff i - window < j <= i (window keys, self incl.) */
  FL_MASK_PREFIX_LM = 3,      /* iff j <= i or j < prefix_len                   */
  FL_MASK_DOCUMENT = 4        /* iff doc(i) == doc(j) [and j <= i if doc_causal] */
} fl_mask_kind;

typedef enum {
  FL_SCORE_NONE = 0,    /* t = s                                   */
  FL_SCORE_ALIBI = 1,   /* t = s + alibi_slopes[h] * (j - i)       */
  FL_SCORE_SOFTCAP = 2  /* t = softcap * tanh(s / softcap)         */
} fl_score_mod;

/* Debug switches (fl_attn_desc.debug_flags). */
#define FL_DEBUG_SKIP_KV_LOAD 0x1u /* block 0 never loads key tile `debug_arg`
                                      of its first work unit: its pipeline
                                      wait runs out and the call reports
                                      FL_ERR_TIMEOUT (tests the bounded waits) */
#define FL_DEBUG_KEY_SPLIT 0x2u    /* fl_attn_fwd with dv <= d <= 64: every
                                      work unit is split along the key axis
                                      (normally only the units of a last,
                                      partial wave over the SMs are), so that
                                      small problems exercise the split and
                                      its merge */

/*
 * Problem descriptor for fl_attn_fwd / fl_diffattn_fwd.
 *   q   [B, Hq,  Lq, d]     k [B, Hkv, Lk, d]     v [B, Hkv, Lk, dv]
 *   out [B, Hq,  Lq, dv]    lse [B, Hq, Lq] (contiguous)
 * Strides are in elements, ordered (b, h, l, c); the c stride is 1.  A
 * zero stride array means contiguous.  s = scale * q.k (scale <= 0 selects
 * 1/sqrt(d)); GQA maps query head h to key/value head h / (Hq / Hkv).
 */
typedef struct fl_attn_desc {
  int32_t B, Hq, Hkv, Lq, Lk, d, dv;
  float scale;
  int32_t mask_kind;        /* fl_mask_kind; masks other than NONE need Lq == Lk */
  int32_t doc_causal;       /* DOCUMENT only: also require j <= i              */
  int32_t window;           /* SLIDING_WINDOW: >= 1                            */
  int32_t prefix_len;       /* PREFIX_LM: >= 0                                 */
  int32_t score_mod;        /* fl_score_mod                                    */
  float softcap;            /* SOFTCAP: > 0                                    */
  const float* alibi_slopes;   /* ALIBI: device fp32 [Hq]                      */
  const int32_t* doc_offsets;  /* DOCUMENT: device int32 [B, num_docs + 1],
                                  offsets[b][0] = 0, strictly increasing,
                                  offsets[b][num_docs] = Lq                    */
  int32_t num_docs;
  int64_t q_strides[4], k_strides[4], v_strides[4], o_strides[4];
  void* stream;             /* cudaStream_t                                    */
  uint32_t debug_flags;     /* FL_DEBUG_*; 0 in normal use                     */
  int32_t debug_arg;
  uint32_t wait_limit_ms;   /* device wait limit; 0 = default (2000 ms)        */
  int32_t reserved[7];
} fl_attn_desc;

/* Fill *desc with zeros and the defaults (mask NONE, score NONE, scale 1/sqrt(d)). */
FL_API void fl_attn_desc_init(fl_attn_desc* desc);

/*
 * Fused attention forward, variants V1-V8: vanilla MHA, GQA, ALiBi, tanh
 * softcap, causal, sliding window, prefix-LM, document mask (score_mod and
 * mask compose).  Supported: d and dv each in {32, 64, 128} (dv may differ
 * from d), Hq % Hkv == 0, any Lq, Lk >= 1 (ragged tails are masked inside
 * the kernel).  Fully masked key tiles are skipped from the descriptor alone
 * (no block mask is built).
 */
FL_API fl_status fl_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      const fl_attn_desc* desc);

/*
 * Block-sparse schedule of fl_attn_fwd for `desc`, without running it (the
 * Flashlight wiki summary's open question 设计取舍 / 局限与 Future Work: whether
 * block_mask sparsity can be handled by analysing the mask at compile time
 * instead of building a block mask at run time).  The kernel derives, from
 * the descriptor alone, the key tiles each 128-row query tile visits; this
 * call walks the same schedule on the host and reports
 *   tiles[0]  (query tile, key tile) pairs computed for rows that exist,
 *   tiles[1]  the same including the padding slot of an odd tile count,
 *   tiles[2]  the dense count B * Hq * ceil(Lq/128) * ceil(Lk/128).
 * With FL_DEBUG_KEY_SPLIT in desc->debug_flags the walk is that of the
 * forced key split (tiles[0] is unchanged by the split).
 * doc_offsets_host: host copy of the document offsets (DOCUMENT only).
 * Pointers in desc other than doc offsets are not read.
 */
FL_API fl_status fl_attn_schedule(const fl_attn_desc* desc, const int32_t* doc_offsets_host, int64_t* tiles);

/*
 * Differential attention (the Flashlight pages, Problem Statement and Results,
 * name it; definition is this library's reading):
 *   out = softmax(scale Q1 K1^T) V - lambda * softmax(scale Q2 K2^T) V
 * q1, k1, q2, k2 [B, H, L, d] (d = 64), v [B, H, L, dv] (dv = 128),
 * out [B, H, L, dv]; lse (may be NULL) is [2, B, H, L]: branch 1 then branch 2.
 * desc: Hq == Hkv == H, Lq == Lk == L, d, dv, scale, mask_kind NONE or CAUSAL;
 * strides must be zero (contiguous).  lambda must be finite.
 */
FL_API fl_status fl_diffattn_fwd(const void* q1, const void* k1, const void* q2, const void* k2,
                          const void* v, void* out, float* lse, float lambda,
                          const fl_attn_desc* desc);

/*
 * AlphaFold Evoformer MSA row-wise gated self-attention (the Flashlight wiki
 * summary, 设计取舍, notes its extra broadcast bias dimension; technical
 * summary, Results, names the row-wise form):
 *   t[i,j] = scale q_i.k_j + pair_bias[b,h,i,j] + mask_bias[b,s,j]
 *   out    = sigmoid(gate) * softmax_j(t) V
 * q, k, v, gate, out : bf16 [B, N_seq, H, N_res, d] contiguous, d = 32
 *                      (AlphaFold's per-head width)
 * pair_bias          : fp32 [B, H, N_res, N_res] (shared by all N_seq rows), or NULL
 * mask_bias          : fp32 [B, N_seq, N_res] (e.g. 0 / -1e9), or NULL
 * lse                : fp32 [B, N_seq, H, N_res], or NULL
 * With a bias, N_res must be a multiple of 4 (16-byte bias rows), else
 * FL_ERR_UNSUPPORTED.  scale <= 0 selects 1/sqrt(d).
 */
FL_API fl_status fl_evoformer_gated_attn_fwd(const void* q, const void* k, const void* v,
                                      const float* pair_bias, const float* mask_bias,
                                      const void* gate, void* out, float* lse, int32_t B,
                                      int32_t N_seq, int32_t N_res, int32_t H, int32_t d,
                                      float scale, void* stream);

/*
 * AlphaFold Evoformer MSA column-wise gated self-attention (the Flashlight
 * technical summary, Results, names the column-wise form beside the
 * row-wise one): for every residue column r, attention over the MSA rows,
 *   t[s,s'] = scale q[b,s,h,r].k[b,s',h,r] + mask_bias[b,r,s']
 *   out[b,s,h,r] = sigmoid(gate[b,s,h,r]) * sum_s' softmax_s'(t[s,.]) v[b,s',h,r]
 * q, k, v, gate, out : bf16 [B, N_seq, H, N_res, d] contiguous (the same
 *                      layout as the row-wise call), d in {32, 64}
 * mask_bias          : fp32 [B, N_res, N_seq] (the MSA mask of each residue
 *                      column as an additive 0 / -1e9 bias), or NULL; N_seq
 *                      must then be a multiple of 4
 * lse                : fp32 [B, H, N_res, N_seq], or NULL
 * No pair bias enters the column-wise form.  scale <= 0 selects 1/sqrt(d).
 */
FL_API fl_status fl_evoformer_col_gated_attn_fwd(const void* q, const void* k, const void* v,
                                          const float* mask_bias, const void* gate, void* out,
                                          float* lse, int32_t B, int32_t N_seq, int32_t N_res,
                                          int32_t H, int32_t d, float scale, void* stream);

/*
 * Decode-phase attention over a key/value cache (the Flashlight wiki
 * summary's critical analysis, 批判性分析, names the serving path's decode
 * phase; the technical summary's online softmax is applied per key split):
 * Lq new query rows per sequence against the first kv_len[b] cached keys.
 * Query row i of sequence b sits at position p = kv_len[b] - Lq + i; key j
 * is visible when j < kv_len[b] and, with mask_kind CAUSAL, j <= p.  ALiBi
 * adds alibi_slopes[h] * (j - p); softcap as in fl_attn_fwd.
 *   q, out            : bf16 [B, Hq, Lq, d] contiguous
 *   k_cache, v_cache  : bf16 [B, Hkv, Lk, d] contiguous (desc->Lk = cache capacity)
 *   lse               : fp32 [B, Hq, Lq] or NULL
 *   kv_len            : device int32 [B] (values clamped to [0, Lk]), or NULL for Lk
 *   workspace         : caller-owned device buffer of at least
 *                       fl_attn_decode_workspace_size(desc) bytes (16-byte
 *                       aligned; may be NULL when that size is 0)
 * desc: d == dv in {64, 128}; (Hq / Hkv) * Lq <= 64; Lq <= Lk; mask NONE or
 * CAUSAL; strides zero.  The key axis is split over CTAs so that the grid
 * covers the GPU; each split's normalised partial output and log-sum-exp go
 * to the workspace and a second kernel merges them.  Rows that see no key
 * get out = 0 and lse = -inf.
 */
FL_API fl_status fl_attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache, void* out,
                                    float* lse, const int32_t* kv_len, void* workspace,
                                    size_t workspace_bytes, const fl_attn_desc* desc);

/* Workspace bytes fl_attn_decode_fwd needs for `desc` on the current device
   (0 when the key axis is not split, or on an invalid descriptor). */
FL_API size_t fl_attn_decode_workspace_size(const fl_attn_desc* desc);

/*
 * Backward pass of fl_attn_fwd (the Flashlight wiki summary lists the
 * training backward under 局限与 Future Work; the definition is the plain
 * derivative of the forward): given dout = dL/dout, returns
 *   dv = P^T dout,  dq = scale dS K,  dk = scale dS^T q,
 *   dS = P * (dout v^T - rowsum(dout * out)) * dT/dS
 * with P recomputed from the forward's lse (dT/dS = 1 - tanh(s/cap)^2 for
 * softcap, else 1); GQA sums dk, dv over each group's query heads.
 *   q, out, dout, dq : bf16 [B, Hq, Lq, d] contiguous
 *   k, v, dk, dv     : bf16 [B, Hkv, Lk, d] contiguous
 *   lse              : fp32 [B, Hq, Lq], the forward's (natural log)
 *   workspace        : caller-owned device buffer of at least
 *                      fl_attn_bwd_workspace_size(desc) bytes (16-byte
 *                      aligned): an fp32 dq accumulator and two per-row vectors
 * desc: the forward's descriptor; d == dv in {32, 64, 128}, or d 64 with
 * dv 128 (v, dv: [B, Hkv, Lk, dv]; out, dout: [B, Hq, Lq, dv]); Lq a
 * multiple of 4, strides zero.  Masks, ALiBi and softcap as in fl_attn_fwd.
 */
FL_API fl_status fl_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                             const float* lse, void* dq, void* dk, void* dv, void* workspace,
                             size_t workspace_bytes, const fl_attn_desc* desc);

/* Workspace bytes fl_attn_bwd needs for `desc` (0 on an invalid descriptor). */
FL_API size_t fl_attn_bwd_workspace_size(const fl_attn_desc* desc);

/*
 * Backward of fl_diffattn_fwd (differential attention, Flashlight technical
 * summary, Results: differential attention among the variants; the training
 * backward is future work in the wiki summary, 局限与 Future Work).  With
 * out = O1 - lambda O2, O_i = softmax(scale Q_i K_i^T [+ causal mask]) V, and
 * dout = dL/dout, returns the plain derivatives
 *   dq_i, dk_i : those of attention branch i for the output gradient dout
 *                (i = 1) or -lambda dout (i = 2)
 *   dv         : the sum of both branches' dV
 *   q1, k1, q2, k2, dq1, dk1, dq2, dk2 : bf16 [B, H, L, 64] contiguous
 *   v, dout, dv                        : bf16 [B, H, L, 128] contiguous
 *   workspace : caller-owned device buffer of at least
 *               fl_diffattn_bwd_workspace_size(desc) bytes (16-byte aligned);
 *               the call recomputes O1, O2 and their LSEs into it (the fused
 *               forward keeps only O1 - lambda O2)
 * desc: as for fl_diffattn_fwd (Hkv == Hq, Lk == Lq, d 64, dv 128, mask NONE
 * or CAUSAL, no score_mod, strides zero), and Lq a multiple of 4.  Errors as
 * fl_attn_bwd; asynchronous on desc->stream.
 */
FL_API fl_status fl_diffattn_bwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                                 const void* dout, float lambda, void* dq1, void* dk1, void* dq2, void* dk2,
                                 void* dv, void* workspace, size_t workspace_bytes, const fl_attn_desc* desc);

/* Workspace bytes fl_diffattn_bwd needs for `desc` (0 on an invalid descriptor). */
FL_API size_t fl_diffattn_bwd_workspace_size(const fl_attn_desc* desc);

/*
 * Allocation-free variant of fl_attn_fwd (no counterpart in the paper; it is
 * a property of this library's interface).  For callers that cannot let a
 * library call cudaMalloc: processes whose device memory all comes from
 * their own pre-reserved pool or arena, code that must not allocate while a
 * stream is captured into a CUDA graph, and callers with a hard memory
 * budget.  Same arguments, results and errors as fl_attn_fwd, but the
 * kernel's status words live in a 256-byte array compiled into the library
 * (present on every GPU that loads it, until the process exits) instead of
 * a cudaMalloc'd word, and nothing is allocated.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make that first call before any stream
 *     capture.
 *   - The scratch needed per call is 8 bytes whatever the problem size; a
 *     requirement above the array's 256 bytes would return
 *     FL_ERR_UNSUPPORTED.
 *   - All calls on a device share the array and it keeps what the last call
 *     wrote: a device-side timeout stays recorded until queried.  Calls that
 *     overlap on the GPU (different streams) race on it: a failure is
 *     reported to whichever query comes next.
 *   - Query mode: with q, k, v, out and lse all NULL the call synchronises
 *     desc->stream and returns (and clears) the recorded status: FL_OK or
 *     FL_ERR_TIMEOUT.  fl_sync_status does not see this path's status.
 */
FL_API fl_status fl_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                                     const fl_attn_desc* desc);

/* Synchronise `stream`, then return and clear the device status word of the
   current device (FL_OK, or FL_ERR_TIMEOUT if a kernel gave up waiting). */
FL_API fl_status fl_sync_status(void* stream);

/* What the last call on this thread that returned FL_ERR_CUDA failed on
   (the CUDA call or step and CUDA's message); "" if none has. */
FL_API const char* fl_last_error_detail(void);

/* Static description of a status code. */
FL_API const char* fl_status_string(fl_status status);

/* FL_ABI_VERSION of the loaded library. */
FL_API int32_t fl_abi_version(void);

/* sizeof(fl_attn_desc) as compiled into the library (binding layout check). */
FL_API int32_t fl_attn_desc_size(void);

#ifdef __cplusplus
}
#endif

#endif /* FLATTN_H_ */
