// C ABI of the fused attention library: argument validation, TMA tensor-map
// encoding, work-unit counting, launch, and the per-device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "flattn.h"
#include "kernels.h"
#include "params.h"

namespace {

using fl::KParams;

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 2000ull * 1000ull * 1000ull;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

struct DeviceState {
  int sm_count = 0;
  uint32_t* status = nullptr;  // [0]: error bits, [1]: where the wait gave up
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

fl_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_dev[dev];
  if (d.status == nullptr) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return FL_ERR_CUDA;
    uint32_t* st = nullptr;
    if (cudaMalloc(&st, 4 * sizeof(uint32_t)) != cudaSuccess) return FL_ERR_CUDA;
    if (cudaMemset(st, 0, 4 * sizeof(uint32_t)) != cudaSuccess) {
      cudaFree(st);
      return FL_ERR_CUDA;
    }
    d.sm_count = sms;
    d.status = st;
  }
  *out = &d;
  return FL_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 4-D bf16 tensor map over a [B, H, L, C] view (strides in elements; channel
// stride 1), boxes of box_c channels x 128 rows; swizzle = box_c * 2 bytes.
bool encode_bhlc(CUtensorMap* m, const void* base, int64_t C, int64_t L, int64_t H, int64_t B, int64_t sl,
                 int64_t sh, int64_t sb, int box_c) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sl * 2), static_cast<cuuint64_t>(sh * 2),
                           static_cast<cuuint64_t>(sb * 2)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_c), 128u, 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUtensorMapSwizzle sw = box_c * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : box_c * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct Strides {
  int64_t b, h, l;
};

// Resolve a (b, h, l, c) stride array; all-zero means contiguous [B,H,L,C].
bool resolve_strides(const int64_t s[4], int64_t H, int64_t L, int64_t C, Strides* out) {
  if (s[0] == 0 && s[1] == 0 && s[2] == 0 && s[3] == 0) {
    out->l = C;
    out->h = L * C;
    out->b = H * L * C;
    return true;
  }
  if (s[3] != 1 || s[0] <= 0 || s[1] <= 0 || s[2] <= 0) return false;
  out->b = s[0];
  out->h = s[1];
  out->l = s[2];
  return true;
}

bool strides_aligned(const Strides& s) { return (s.b * 2) % 16 == 0 && (s.h * 2) % 16 == 0 && (s.l * 2) % 16 == 0; }

int box_width(int c) { return c >= 64 ? 64 : c; }

uint64_t wait_ns(uint32_t ms) { return ms ? static_cast<uint64_t>(ms) * 1000ull * 1000ull : kDefaultWaitNs; }

}  // namespace

extern "C" {

void fl_attn_desc_init(fl_attn_desc* desc) {
  if (!desc) return;
  std::memset(desc, 0, sizeof(*desc));
  desc->mask_kind = FL_MASK_NONE;
  desc->score_mod = FL_SCORE_NONE;
  desc->scale = 0.f;
  desc->debug_arg = -1;
}

const char* fl_status_string(fl_status s) {
  switch (s) {
    case FL_OK: return "ok";
    case FL_ERR_INVALID_ARG: return "invalid argument";
    case FL_ERR_UNSUPPORTED: return "unsupported configuration";
    case FL_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case FL_ERR_CUDA: return "CUDA error";
    case FL_ERR_TIMEOUT: return "device pipeline wait timed out";
    case FL_ERR_DEVICE_BOUNDS: return "device bounds check failed";
  }
  return "unknown status";
}

int32_t fl_abi_version(void) { return FL_ABI_VERSION; }

int32_t fl_attn_desc_size(void) { return static_cast<int32_t>(sizeof(fl_attn_desc)); }

fl_status fl_sync_status(void* stream) {
  DeviceState* ds = nullptr;
  fl_status st = device_state(&ds);
  if (st != FL_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FL_ERR_CUDA;
  uint32_t h[2] = {0u, 0u};
  if (cudaMemcpy(h, ds->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FL_ERR_CUDA;
  if (h[0] == 0u) return FL_OK;
  if (cudaMemset(ds->status, 0, 2 * sizeof(uint32_t)) != cudaSuccess) return FL_ERR_CUDA;
  return (h[0] & 1u) ? FL_ERR_TIMEOUT : FL_ERR_DEVICE_BOUNDS;
}

fl_status fl_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      const fl_attn_desc* desc) {
  if (!desc || !q || !k || !v || !out) return FL_ERR_INVALID_ARG;
  const fl_attn_desc& d = *desc;
  if (d.B < 1 || d.Hq < 1 || d.Hkv < 1 || d.Lq < 1 || d.Lk < 1 || d.Hq % d.Hkv != 0) return FL_ERR_INVALID_ARG;
  if (!(d.d == 32 || d.d == 64 || d.d == 128)) return FL_ERR_UNSUPPORTED;
  if (d.dv != d.d) return FL_ERR_UNSUPPORTED;
  if (!std::isfinite(d.scale)) return FL_ERR_INVALID_ARG;
  if (d.mask_kind < FL_MASK_NONE || d.mask_kind > FL_MASK_DOCUMENT) return FL_ERR_INVALID_ARG;
  if (d.mask_kind != FL_MASK_NONE && d.Lq != d.Lk) return FL_ERR_UNSUPPORTED;
  if (d.mask_kind == FL_MASK_SLIDING_WINDOW && d.window < 1) return FL_ERR_INVALID_ARG;
  if (d.mask_kind == FL_MASK_PREFIX_LM && d.prefix_len < 0) return FL_ERR_INVALID_ARG;
  if (d.mask_kind == FL_MASK_DOCUMENT && (!d.doc_offsets || d.num_docs < 1 || d.num_docs > d.Lq))
    return FL_ERR_INVALID_ARG;
  if (d.score_mod < FL_SCORE_NONE || d.score_mod > FL_SCORE_SOFTCAP) return FL_ERR_INVALID_ARG;
  if (d.score_mod == FL_SCORE_ALIBI && !d.alibi_slopes) return FL_ERR_INVALID_ARG;
  if (d.score_mod == FL_SCORE_SOFTCAP && !(d.softcap > 0.f && std::isfinite(d.softcap))) return FL_ERR_INVALID_ARG;
  Strides sq, sk, sv, so;
  if (!resolve_strides(d.q_strides, d.Hq, d.Lq, d.d, &sq) || !resolve_strides(d.k_strides, d.Hkv, d.Lk, d.d, &sk) ||
      !resolve_strides(d.v_strides, d.Hkv, d.Lk, d.dv, &sv) || !resolve_strides(d.o_strides, d.Hq, d.Lq, d.dv, &so))
    return FL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !strides_aligned(sq) ||
      !strides_aligned(sk) || !strides_aligned(sv) || !strides_aligned(so))
    return FL_ERR_ALIGNMENT;
  if (d.mask_kind == FL_MASK_DOCUMENT && (reinterpret_cast<uintptr_t>(d.doc_offsets) & 3u)) return FL_ERR_ALIGNMENT;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FL_ERR_ALIGNMENT;

  DeviceState* ds = nullptr;
  fl_status st = device_state(&ds);
  if (st != FL_OK) return st;

  KParams p{};
  p.B = d.B; p.Hq = d.Hq; p.Hkv = d.Hkv; p.Lq = d.Lq; p.Lk = d.Lk;
  p.group = d.Hq / d.Hkv;
  p.n_qtiles = (d.Lq + fl::kBlockM - 1) / fl::kBlockM;
  const float scale = d.scale > 0.f ? d.scale : 1.0f / std::sqrt(static_cast<float>(d.d));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = d.mask_kind; p.doc_causal = d.doc_causal ? 1 : 0;
  p.window = d.window; p.prefix = d.prefix_len;
  p.doc_offsets = d.doc_offsets; p.num_docs = d.num_docs;
  p.slopes = d.alibi_slopes; p.softcap = d.softcap;
  p.out = out; p.o_sb = so.b; p.o_sh = so.h; p.o_sl = so.l;
  p.lse = lse;
  p.status = ds->status;
  p.timeout_ns = wait_ns(d.wait_limit_ms);
  p.dbg_skip_tile = (d.debug_flags & FL_DEBUG_SKIP_KV_LOAD) ? (d.debug_arg < 0 ? 0 : d.debug_arg) : -1;
#ifdef FL_TRACE
  if (const char* tp = std::getenv("FLATTN_TRACE_PTR"))
    p.trace = reinterpret_cast<unsigned long long*>(std::strtoull(tp, nullptr, 0));
#endif
  int64_t units;
  if (p.group == 1) {
    p.slot_mode = fl::SLOT_ROWS;
    units = static_cast<int64_t>(d.B) * d.Hq * ((p.n_qtiles + 1) / 2);
  } else {
    p.slot_mode = fl::SLOT_HEADS;
    p.pairs_per_group = (p.group + 1) / 2;
    units = static_cast<int64_t>(d.B) * d.Hkv * p.pairs_per_group * p.n_qtiles;
  }
  if (units > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(units);

  CUtensorMap maps[6];
  const int bq = box_width(d.d), bv = box_width(d.dv);
  if (!encode_bhlc(&maps[0], q, d.d, d.Lq, d.Hq, d.B, sq.l, sq.h, sq.b, bq) ||
      !encode_bhlc(&maps[1], k, d.d, d.Lk, d.Hkv, d.B, sk.l, sk.h, sk.b, bq) ||
      !encode_bhlc(&maps[2], v, d.dv, d.Lk, d.Hkv, d.B, sv.l, sv.h, sv.b, bv) ||
      !encode_bhlc(&maps[5], out, d.dv, d.Lq, d.Hq, d.B, so.l, so.h, so.b, bv))
    return FL_ERR_CUDA;
  maps[3] = maps[0];
  maps[4] = maps[1];

  const int grid = static_cast<int>(units < ds->sm_count ? units : ds->sm_count);
  cudaStream_t stream = static_cast<cudaStream_t>(d.stream);
  cudaError_t e;
  switch (d.d) {
    case 32: e = fl::launch_attn_d32(d.score_mod, maps, p, grid, stream); break;
    case 64: e = fl::launch_attn_d64(d.score_mod, maps, p, grid, stream); break;
    default: e = fl::launch_attn_d128(d.score_mod, maps, p, grid, stream); break;
  }
  return e == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

fl_status fl_diffattn_fwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v, void* out,
                          float* lse, float lambda, const fl_attn_desc* desc) {
  if (!desc || !q1 || !k1 || !q2 || !k2 || !v || !out) return FL_ERR_INVALID_ARG;
  const fl_attn_desc& d = *desc;
  if (d.B < 1 || d.Hq < 1 || d.Lq < 1 || d.Hkv != d.Hq || d.Lk != d.Lq) return FL_ERR_INVALID_ARG;
  if (!std::isfinite(lambda) || !std::isfinite(d.scale)) return FL_ERR_INVALID_ARG;
  if (d.d != 64 || d.dv != 128) return FL_ERR_UNSUPPORTED;
  if (d.mask_kind != FL_MASK_NONE && d.mask_kind != FL_MASK_CAUSAL) return FL_ERR_UNSUPPORTED;
  if (d.score_mod != FL_SCORE_NONE) return FL_ERR_UNSUPPORTED;
  for (int i = 0; i < 4; ++i)
    if (d.q_strides[i] || d.k_strides[i] || d.v_strides[i] || d.o_strides[i]) return FL_ERR_UNSUPPORTED;
  if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) || !aligned16(out))
    return FL_ERR_ALIGNMENT;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FL_ERR_ALIGNMENT;

  DeviceState* ds = nullptr;
  fl_status st = device_state(&ds);
  if (st != FL_OK) return st;

  const int H = d.Hq, L = d.Lq;
  KParams p{};
  p.B = d.B; p.Hq = H; p.Hkv = H; p.Lq = L; p.Lk = L; p.group = 1;
  p.n_qtiles = (L + fl::kBlockM - 1) / fl::kBlockM;
  const float scale = d.scale > 0.f ? d.scale : 0.125f;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = d.mask_kind;
  p.out = out; p.o_sl = 128; p.o_sh = static_cast<int64_t>(L) * 128; p.o_sb = static_cast<int64_t>(H) * L * 128;
  p.lse = lse;
  p.lambda = lambda;
  p.status = ds->status;
  p.timeout_ns = wait_ns(d.wait_limit_ms);
  p.dbg_skip_tile = (d.debug_flags & FL_DEBUG_SKIP_KV_LOAD) ? (d.debug_arg < 0 ? 0 : d.debug_arg) : -1;
  p.slot_mode = fl::SLOT_BRANCH;
  const int64_t units = static_cast<int64_t>(d.B) * H * p.n_qtiles;
  if (units > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(units);

  CUtensorMap maps[6];
  const int64_t sl = 64, sh = static_cast<int64_t>(L) * 64, sb = static_cast<int64_t>(H) * L * 64;
  if (!encode_bhlc(&maps[0], q1, 64, L, H, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[1], k1, 64, L, H, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[2], v, 128, L, H, d.B, 128, static_cast<int64_t>(L) * 128,
                   static_cast<int64_t>(H) * L * 128, 64) ||
      !encode_bhlc(&maps[3], q2, 64, L, H, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[4], k2, 64, L, H, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[5], out, 128, L, H, d.B, 128, static_cast<int64_t>(L) * 128,
                   static_cast<int64_t>(H) * L * 128, 64))
    return FL_ERR_CUDA;
  const int grid = static_cast<int>(units < ds->sm_count ? units : ds->sm_count);
  cudaError_t e = fl::launch_diff_d64(maps, p, grid, static_cast<cudaStream_t>(d.stream));
  return e == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

fl_status fl_evoformer_gated_attn_fwd(const void* q, const void* k, const void* v, const float* pair_bias,
                                      const float* mask_bias, const void* gate, void* out, float* lse, int32_t B,
                                      int32_t N_seq, int32_t N_res, int32_t H, int32_t d, float scale,
                                      void* stream) {
  if (!q || !k || !v || !gate || !out) return FL_ERR_INVALID_ARG;
  if (B < 1 || N_seq < 1 || N_res < 1 || H < 1 || !std::isfinite(scale)) return FL_ERR_INVALID_ARG;
  if (d != 32 && d != 64) return FL_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(gate) || !aligned16(out)) return FL_ERR_ALIGNMENT;
  if ((pair_bias && (reinterpret_cast<uintptr_t>(pair_bias) & 15u)) ||
      (mask_bias && (reinterpret_cast<uintptr_t>(mask_bias) & 15u)) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FL_ERR_ALIGNMENT;
  if ((pair_bias || mask_bias) && (N_res % 4) != 0) return FL_ERR_UNSUPPORTED;  // float4 bias rows

  DeviceState* ds = nullptr;
  fl_status st = device_state(&ds);
  if (st != FL_OK) return st;

  const int64_t Bf = static_cast<int64_t>(B) * N_seq;
  KParams p{};
  p.B = static_cast<int>(Bf); p.Hq = H; p.Hkv = H; p.Lq = N_res; p.Lk = N_res; p.group = 1;
  p.n_qtiles = (N_res + fl::kBlockM - 1) / fl::kBlockM;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d));
  p.scale_log2 = sc * 1.4426950408889634f;
  p.mask_kind = fl::MASK_NONE;
  p.out = out; p.o_sl = d; p.o_sh = static_cast<int64_t>(N_res) * d; p.o_sb = static_cast<int64_t>(H) * N_res * d;
  p.lse = lse;
  p.pair_bias = pair_bias; p.mask_bias = mask_bias; p.gate = gate; p.n_seq = N_seq;
  p.status = ds->status;
  p.timeout_ns = kDefaultWaitNs;
  p.dbg_skip_tile = -1;
  p.slot_mode = fl::SLOT_ROWS;
  const int64_t units = Bf * H * ((p.n_qtiles + 1) / 2);
  if (units > 0x7fffffff || Bf > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(units);

  CUtensorMap maps[6];
  const int bw = box_width(d);
  const int64_t sl = d, sh = static_cast<int64_t>(N_res) * d, sb = static_cast<int64_t>(H) * N_res * d;
  if (!encode_bhlc(&maps[0], q, d, N_res, H, Bf, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[1], k, d, N_res, H, Bf, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[2], v, d, N_res, H, Bf, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[5], out, d, N_res, H, Bf, sl, sh, sb, bw))
    return FL_ERR_CUDA;
  maps[3] = maps[0];
  maps[4] = maps[1];
  const int grid = static_cast<int>(units < ds->sm_count ? units : ds->sm_count);
  cudaError_t e = fl::launch_evo(d, maps, p, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

}  // extern "C"
