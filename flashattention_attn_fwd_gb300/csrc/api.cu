// C ABI of the fused attention library: argument validation, TMA tensor-map
// encoding, work-unit counting, launch, and the per-device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "bwd.h"
#include "decode.h"
#include "flattn.h"
#include "fused_attn.cuh"
#include "host.h"
#include "kernels.h"
#include "params.h"

namespace {

using fl::KParams;

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 2000ull * 1000ull * 1000ull;
constexpr double kLog2e = 1.4426950408889634;

// tanh(y) ~= y * (p0 + p1 y^2 + p2 y^4 + p3 y^6) for |y| <= kTanhRange, the
// minimax fit printed by csrc/fit_poly.py (defaults: float32 max relative
// error 6.2e-7).  The softcap kernels fold scale and cap into these.
constexpr double kTanhRange = 0.5;
constexpr float kTanhP[4] = {0.999999464f, -0.333263218f, 0.13190335f, -0.0444031134f};

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

// Detail of the last FL_ERR_CUDA on this thread (fl_last_error_detail).
thread_local char g_detail[192] = "";

fl_status cuda_fail(const char* where, cudaError_t e) {
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s", where, e == cudaSuccess ? "failed" : cudaGetErrorString(e));
  return FL_ERR_CUDA;
}

fl_status launched(const char* where, cudaError_t e) {
  return e == cudaSuccess ? FL_OK : cuda_fail(where, e);
}

struct DeviceState {
  int sm_count = 0;
  uint32_t* status = nullptr;  // [0]: error bits, [1]: where the wait gave up
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

fl_status device_state(DeviceState** out) {
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cuda_fail("cudaGetDevice", ge);
  // make the device's primary context current on this thread (a thread that
  // has made no runtime call yet, e.g. an autograd worker, has none, and the
  // tensor-map encoder is a driver call)
  const cudaError_t sd = cudaSetDevice(dev);
  if (sd != cudaSuccess) return cuda_fail("cudaSetDevice", sd);
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_dev[dev];
  if (d.status == nullptr) {
    int sms = 0;
    const cudaError_t ae = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (ae != cudaSuccess || sms <= 0) return cuda_fail("cudaDeviceGetAttribute", ae);
    uint32_t* st = nullptr;
    const cudaError_t me = cudaMalloc(&st, 4 * sizeof(uint32_t));
    if (me != cudaSuccess) return cuda_fail("cudaMalloc (status word)", me);
    const cudaError_t se = cudaMemset(st, 0, 4 * sizeof(uint32_t));
    if (se != cudaSuccess) {
      cudaFree(st);
      return cuda_fail("cudaMemset (status word)", se);
    }
    d.sm_count = sms;
    d.status = st;
  }
  *out = &d;
  return FL_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Tiled tensor map over `rank` dimensions (innermost first; strides in bytes
// for dimensions 1..rank-1), box `box`, the given swizzle.
bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
            const uint64_t* stride_bytes, const uint32_t* box, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1u;
    if (i + 1 < rank) s[i] = stride_bytes[i];
  }
  return enc(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, b, e,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D bf16 tensor map over a [B, H, L, C] view (strides in elements; channel
// stride 1), boxes of box_c channels x 128 rows; swizzle = box_c * 2 bytes.
bool encode_bhlc(CUtensorMap* m, const void* base, int64_t C, int64_t L, int64_t H, int64_t B, int64_t sl,
                 int64_t sh, int64_t sb, int box_c) {
  const uint64_t dims[4] = {static_cast<uint64_t>(C), static_cast<uint64_t>(L), static_cast<uint64_t>(H),
                            static_cast<uint64_t>(B)};
  const uint64_t str[3] = {static_cast<uint64_t>(sl * 2), static_cast<uint64_t>(sh * 2),
                           static_cast<uint64_t>(sb * 2)};
  const uint32_t box[4] = {static_cast<uint32_t>(box_c), 128u, 1u, 1u};
  const CUtensorMapSwizzle sw = box_c * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_c * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_32B;
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, str, box, sw);
}

// fp32 pair bias [B, H, N, N]: boxes of 32 columns x 128 rows, 128-byte swizzle.
bool encode_pair_bias(CUtensorMap* m, const float* pb, int64_t B, int64_t H, int64_t N) {
  const uint64_t dims[4] = {static_cast<uint64_t>(N), static_cast<uint64_t>(N), static_cast<uint64_t>(H),
                            static_cast<uint64_t>(B)};
  const uint64_t str[3] = {static_cast<uint64_t>(N * 4), static_cast<uint64_t>(N * N * 4),
                           static_cast<uint64_t>(H * N * N * 4)};
  const uint32_t box[4] = {32u, 128u, 1u, 1u};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pb, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// fp32 row-major matrix [rows, cols]: boxes of one 128-column row segment.
bool encode_rows_f32(CUtensorMap* m, const float* base, int64_t rows, int64_t cols) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t str[1] = {static_cast<uint64_t>(cols * 4)};
  const uint32_t box[2] = {128u, 1u};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
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

bool head_dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

// Softcap on the FMA pipe: cap*log2(e)*tanh(s*scale/cap) = s * Q(s^2) while
// |s * scale / cap| <= kTanhRange (the kernel checks the range per warp).
template <class Params>
void softcap_coefficients(Params& p, float scale, float cap) {
  const double ya = static_cast<double>(scale) / cap, k = static_cast<double>(cap) * kLog2e;
  double ypow = ya;
  for (int i = 0; i < 4; ++i) {
    p.sc_q[i] = static_cast<float>(k * kTanhP[i] * ypow);
    ypow *= ya * ya;
  }
  p.sc_smax = static_cast<float>(kTanhRange / ya);
}

cudaError_t launch_attn(int d, int dv, int score_mod, const CUtensorMap* maps, const KParams& p, int grid,
                        cudaStream_t s) {
#define FL_CASE(D, DV) \
  if (d == D && dv == DV) return fl::launch_attn_d##D##_dv##DV(score_mod, maps, p, grid, s);
  FL_CASE(32, 32) FL_CASE(32, 64) FL_CASE(32, 128)
  FL_CASE(64, 32) FL_CASE(64, 64) FL_CASE(64, 128)
  FL_CASE(128, 32) FL_CASE(128, 64) FL_CASE(128, 128)
#undef FL_CASE
  return cudaErrorInvalidValue;
}

// Kernel parameters of fl_attn_fwd for a validated descriptor (out strides
// `so`, status words `status`): problem, variant, schedule.
fl_status fill_attn_params(const fl_attn_desc& d, const Strides& so, uint32_t* status, KParams* p) {
  p->B = d.B; p->Hq = d.Hq; p->Hkv = d.Hkv; p->Lq = d.Lq; p->Lk = d.Lk;
  p->group = d.Hq / d.Hkv;
  p->n_qtiles = (d.Lq + fl::kBlockM - 1) / fl::kBlockM;
  const float scale = d.scale > 0.f ? d.scale : 1.0f / std::sqrt(static_cast<float>(d.d));
  p->scale = scale;
  p->scale_log2 = scale * static_cast<float>(kLog2e);
  p->mask_kind = d.mask_kind; p->doc_causal = d.doc_causal ? 1 : 0;
  p->window = d.window; p->prefix = d.prefix_len;
  p->doc_offsets = d.doc_offsets; p->num_docs = d.num_docs;
  p->slopes = d.alibi_slopes; p->softcap = d.softcap;
  if (d.score_mod == FL_SCORE_SOFTCAP) softcap_coefficients(*p, scale, d.softcap);
  p->o_sb = so.b; p->o_sh = so.h; p->o_sl = so.l;
  p->status = status;
  p->timeout_ns = wait_ns(d.wait_limit_ms);
  p->dbg_skip_tile = (d.debug_flags & FL_DEBUG_SKIP_KV_LOAD) ? (d.debug_arg < 0 ? 0 : d.debug_arg) : -1;
  int64_t units;
  if (p->group == 1) {
    p->slot_mode = fl::SLOT_ROWS;
    units = static_cast<int64_t>(d.B) * d.Hq * ((p->n_qtiles + 1) / 2);
  } else {
    p->slot_mode = fl::SLOT_HEADS;
    p->pairs_per_group = (p->group + 1) / 2;
    units = static_cast<int64_t>(d.B) * d.Hkv * p->pairs_per_group * p->n_qtiles;
  }
  if (units > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  p->num_units = static_cast<int>(units);
  return FL_OK;
}

// Key split of a last, partial wave.  Units are dealt to the persistent CTAs
// in turn, so with U units on W CTAs, R = U mod W of them run alone after
// the full waves while W - R CTAs idle.  When R <= W / 2 each of those R
// units becomes two key-split units (one per query tile, each walking its
// key range in two halves on the two slots): the last wave then takes half
// as long.  FL_DEBUG_KEY_SPLIT splits every unit.
void plan_key_split(const fl_attn_desc& d, int sm_count, KParams* p) {
  p->ks_count = 0;
  if (!fl::key_split_ok(d.d, d.dv)) return;
  const int units = p->num_units;
  if (d.debug_flags & FL_DEBUG_KEY_SPLIT) {
    if (units > 0x3fffffff) return;
    p->ks_count = 2 * units;
    p->num_units = 2 * units;
    return;
  }
  const int w = units < sm_count ? units : sm_count;
  if (w < 2 || units <= w) return;
  const int r = units % w;
  if (r == 0 || 2 * r > w) return;
  p->ks_count = 2 * r;
  p->num_units = units + r;
}

}  // namespace

namespace fl {

fl_status attn_fwd_check(const void* q, const void* k, const void* v, void* out, float* lse,
                         const fl_attn_desc* desc) {
  if (!desc || !q || !k || !v || !out) return FL_ERR_INVALID_ARG;
  const fl_attn_desc& d = *desc;
  if (d.B < 1 || d.Hq < 1 || d.Hkv < 1 || d.Lq < 1 || d.Lk < 1 || d.Hq % d.Hkv != 0) return FL_ERR_INVALID_ARG;
  if (!head_dim_ok(d.d) || !head_dim_ok(d.dv)) return FL_ERR_UNSUPPORTED;
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
  if (d.mask_kind == FL_MASK_DOCUMENT && !aligned4(d.doc_offsets)) return FL_ERR_ALIGNMENT;
  if (lse && !aligned4(lse)) return FL_ERR_ALIGNMENT;
  return FL_OK;
}

fl_status attn_fwd_launch(const void* q, const void* k, const void* v, void* out, float* lse,
                          const fl_attn_desc* desc, uint32_t* status, int sm_count) {
  const fl_status chk = attn_fwd_check(q, k, v, out, lse, desc);
  if (chk != FL_OK) return chk;
  const fl_attn_desc& d = *desc;
  Strides sq, sk, sv, so;
  resolve_strides(d.q_strides, d.Hq, d.Lq, d.d, &sq);
  resolve_strides(d.k_strides, d.Hkv, d.Lk, d.d, &sk);
  resolve_strides(d.v_strides, d.Hkv, d.Lk, d.dv, &sv);
  resolve_strides(d.o_strides, d.Hq, d.Lq, d.dv, &so);

  KParams p{};
  const fl_status fs = fill_attn_params(d, so, status, &p);
  if (fs != FL_OK) return fs;
  plan_key_split(d, sm_count, &p);
  p.out = out;
  p.lse = lse;
  const int64_t units = p.num_units;

  CUtensorMap maps[8];
  const int bq = box_width(d.d), bv = box_width(d.dv);
  if (!encode_bhlc(&maps[0], q, d.d, d.Lq, d.Hq, d.B, sq.l, sq.h, sq.b, bq) ||
      !encode_bhlc(&maps[1], k, d.d, d.Lk, d.Hkv, d.B, sk.l, sk.h, sk.b, bq) ||
      !encode_bhlc(&maps[2], v, d.dv, d.Lk, d.Hkv, d.B, sv.l, sv.h, sv.b, bv) ||
      !encode_bhlc(&maps[5], out, d.dv, d.Lq, d.Hq, d.B, so.l, so.h, so.b, bv))
    return cuda_fail("cuTensorMapEncodeTiled", cudaSuccess);
  maps[3] = maps[0];
  maps[4] = maps[1];
  maps[6] = maps[0];
  maps[7] = maps[0];

  const int grid = static_cast<int>(units < sm_count ? units : sm_count);
  return launched("attention kernel launch",
                  launch_attn(d.d, d.dv, d.score_mod, maps, p, grid, static_cast<cudaStream_t>(d.stream)));
}

}  // namespace fl

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

const char* fl_last_error_detail(void) { return g_detail; }

int32_t fl_attn_desc_size(void) { return static_cast<int32_t>(sizeof(fl_attn_desc)); }

fl_status fl_sync_status(void* stream) {
  DeviceState* ds = nullptr;
  fl_status st = device_state(&ds);
  if (st != FL_OK) return st;
  const cudaError_t se = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (se != cudaSuccess) return cuda_fail("cudaStreamSynchronize", se);
  uint32_t h[2] = {0u, 0u};
  const cudaError_t ce = cudaMemcpy(h, ds->status, sizeof(h), cudaMemcpyDeviceToHost);
  if (ce != cudaSuccess) return cuda_fail("cudaMemcpy (status word)", ce);
  if (h[0] == 0u) return FL_OK;
  const cudaError_t me = cudaMemset(ds->status, 0, 2 * sizeof(uint32_t));
  if (me != cudaSuccess) return cuda_fail("cudaMemset (status word)", me);
  return (h[0] & 1u) ? FL_ERR_TIMEOUT : FL_ERR_DEVICE_BOUNDS;
}

fl_status fl_attn_schedule(const fl_attn_desc* desc, const int32_t* doc_offsets_host, int64_t* tiles) {
  if (!desc || !tiles) return FL_ERR_INVALID_ARG;
  fl_attn_desc d = *desc;
  if (d.mask_kind == FL_MASK_DOCUMENT) {
    if (!doc_offsets_host) return FL_ERR_INVALID_ARG;
    d.doc_offsets = doc_offsets_host;
  }
  static const int64_t kFake = 0x10000;  // only validated, never dereferenced
  const void* f = reinterpret_cast<const void*>(kFake);
  if (d.score_mod == FL_SCORE_ALIBI && !d.alibi_slopes) d.alibi_slopes = static_cast<const float*>(f);
  const fl_status chk = fl::attn_fwd_check(f, f, f, const_cast<void*>(f), nullptr, &d);
  if (chk != FL_OK) return chk;
  Strides so;
  resolve_strides(d.o_strides, d.Hq, d.Lq, d.dv, &so);
  KParams p{};
  const fl_status fs = fill_attn_params(d, so, nullptr, &p);
  if (fs != FL_OK) return fs;
  // the last-wave split depends on the SM count and leaves the visited tiles
  // unchanged; the forced split (FL_DEBUG_KEY_SPLIT) is walked as launched
  if (d.debug_flags & FL_DEBUG_KEY_SPLIT) plan_key_split(d, 1, &p);
  const bool per_slot = d.dv <= 64;  // one MMA thread per slot: per-slot key ranges
  int64_t own = 0, all = 0;
  for (int u = 0; u < p.num_units; ++u) {
    const fl::Unit U = fl::decode_unit<fl::KIND_ATTN>(p, u, per_slot);
    for (int s = 0; s < 2; ++s) {
      const int64_t n = U.hi[s] - U.lo[s] + 1;
      all += n;
      // a key-split unit's second slot computes the lower half of the rows' keys
      if (U.ks || (U.valid[s] && U.row0[s] < p.Lq &&
                   !(p.slot_mode == fl::SLOT_HEADS && s == 1 && U.hq[1] == U.hq[0])))
        own += n;
    }
  }
  const int64_t nq = (d.Lq + 127) / 128, nk = (d.Lk + 127) / 128;
  tiles[0] = own;
  tiles[1] = all;
  tiles[2] = static_cast<int64_t>(d.B) * d.Hq * nq * nk;
  return FL_OK;
}

fl_status fl_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      const fl_attn_desc* desc) {
  const fl_status chk = fl::attn_fwd_check(q, k, v, out, lse, desc);
  if (chk != FL_OK) return chk;
  DeviceState* ds = nullptr;
  const fl_status st = device_state(&ds);
  if (st != FL_OK) return st;
  return fl::attn_fwd_launch(q, k, v, out, lse, desc, ds->status, ds->sm_count);
}

namespace {

fl_status decode_check(const void* q, const void* k, const void* v, void* out, float* lse, const int32_t* kv_len,
                       const fl_attn_desc* desc) {
  if (!desc || !q || !k || !v || !out) return FL_ERR_INVALID_ARG;
  const fl_attn_desc& d = *desc;
  if (d.B < 1 || d.Hq < 1 || d.Hkv < 1 || d.Lq < 1 || d.Lk < 1 || d.Hq % d.Hkv != 0 || d.Lq > d.Lk)
    return FL_ERR_INVALID_ARG;
  if (d.d != d.dv || (d.d != 64 && d.d != 128)) return FL_ERR_UNSUPPORTED;
  if ((d.Hq / d.Hkv) * d.Lq > fl::kDecodeMaxRows) return FL_ERR_UNSUPPORTED;
  if (!std::isfinite(d.scale)) return FL_ERR_INVALID_ARG;
  if (d.mask_kind != FL_MASK_NONE && d.mask_kind != FL_MASK_CAUSAL) return FL_ERR_UNSUPPORTED;
  if (d.score_mod < FL_SCORE_NONE || d.score_mod > FL_SCORE_SOFTCAP) return FL_ERR_INVALID_ARG;
  if (d.score_mod == FL_SCORE_ALIBI && !d.alibi_slopes) return FL_ERR_INVALID_ARG;
  if (d.score_mod == FL_SCORE_SOFTCAP && !(d.softcap > 0.f && std::isfinite(d.softcap))) return FL_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (d.q_strides[i] || d.k_strides[i] || d.v_strides[i] || d.o_strides[i]) return FL_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FL_ERR_ALIGNMENT;
  if ((lse && !aligned4(lse)) || (kv_len && !aligned4(kv_len))) return FL_ERR_ALIGNMENT;
  return FL_OK;
}

size_t decode_workspace(const fl_attn_desc& d, int sm_count, int* n_split, int* chunk) {
  fl::decode_split(d.B, d.Hkv, d.Lk, d.Hq / d.Hkv * d.Lq, sm_count, n_split, chunk);
  if (*n_split <= 1) return 0;
  const size_t rows = static_cast<size_t>(d.B) * d.Hq * d.Lq;
  return static_cast<size_t>(*n_split) * rows * (static_cast<size_t>(d.d) + 1) * sizeof(float);
}

}  // namespace

size_t fl_attn_bwd_workspace_size(const fl_attn_desc* desc) {
  if (!desc || desc->B < 1 || desc->Hq < 1 || desc->Lq < 1 || desc->d < 1) return 0;
  const size_t rows = static_cast<size_t>(desc->B) * desc->Hq * desc->Lq;
  return rows * (static_cast<size_t>(desc->d) + 2) * sizeof(float);
}

namespace {

// fl_attn_bwd for the gradients of dout_scale * dout, adding dV to dv's
// contents when dv_accumulate (the differential backward's second branch).
fl_status attn_bwd_run(const void* q, const void* k, const void* v, const void* out, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                       const fl_attn_desc* desc, float dout_scale, bool dv_accumulate) {
  if (!desc || !q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return FL_ERR_INVALID_ARG;
  const fl_attn_desc& d = *desc;
  if (d.B < 1 || d.Hq < 1 || d.Hkv < 1 || d.Lq < 1 || d.Lk < 1 || d.Hq % d.Hkv != 0) return FL_ERR_INVALID_ARG;
  const bool same = d.d == d.dv && (d.d == 32 || d.d == 64 || d.d == 128);
  if (!same && !(d.d == 64 && d.dv == 128)) return FL_ERR_UNSUPPORTED;
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
  for (int i = 0; i < 4; ++i)
    if (d.q_strides[i] || d.k_strides[i] || d.v_strides[i] || d.o_strides[i]) return FL_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, out, dout, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FL_ERR_ALIGNMENT;
  if (!aligned4(lse) || (d.mask_kind == FL_MASK_DOCUMENT && !aligned4(d.doc_offsets))) return FL_ERR_ALIGNMENT;
  if (d.Lq % 4 != 0) return FL_ERR_UNSUPPORTED;  // 16-byte rows of the per-query vectors (TMA)
  const size_t need = fl_attn_bwd_workspace_size(desc);
  if (!workspace || workspace_bytes < need) return FL_ERR_INVALID_ARG;

  DeviceState* ds = nullptr;
  const fl_status st = device_state(&ds);
  if (st != FL_OK) return st;
  fl::BwdParams p{};
  p.out = out; p.dout = dout; p.lse = lse; p.dq = dq; p.dk = dk; p.dv = dv;
  p.rows = static_cast<int64_t>(d.B) * d.Hq * d.Lq;
  p.dq_acc = static_cast<float*>(workspace);
  p.dvec = p.dq_acc + p.rows * d.d;
  p.l2 = p.dvec + p.rows;
  p.slopes = d.alibi_slopes; p.doc_offsets = d.doc_offsets;
  p.status = ds->status;
  p.timeout_ns = wait_ns(d.wait_limit_ms);
  p.B = d.B; p.Hq = d.Hq; p.Hkv = d.Hkv; p.Lq = d.Lq; p.Lk = d.Lk;
  p.n_ktiles = (d.Lk + 127) / 128;
  p.scale = d.scale > 0.f ? d.scale : 1.0f / std::sqrt(static_cast<float>(d.d));
  p.softcap = d.softcap;
  if (d.score_mod == FL_SCORE_SOFTCAP) softcap_coefficients(p, p.scale, d.softcap);
  p.dout_scale = dout_scale;
  p.dv_accumulate = dv_accumulate ? 1 : 0;
  p.mask_kind = d.mask_kind; p.doc_causal = d.doc_causal ? 1 : 0;
  p.window = d.window; p.prefix = d.prefix_len; p.num_docs = d.num_docs;
  if (static_cast<int64_t>(d.B) * d.Hkv * p.n_ktiles > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  CUtensorMap maps[7];
  const int bw = box_width(d.d), bwv = box_width(d.dv);
  const int64_t sl = d.d, slv = d.dv;
  // the fp32 dQ accumulator as [B * Hq][Lq][d], boxes of 32 channels x 128
  // rows (the target of the kernel's bulk reductions)
  const uint64_t qa_dims[3] = {static_cast<uint64_t>(d.d), static_cast<uint64_t>(d.Lq),
                               static_cast<uint64_t>(d.B) * d.Hq};
  const uint64_t qa_str[2] = {static_cast<uint64_t>(d.d) * 4, static_cast<uint64_t>(d.Lq) * d.d * 4};
  const uint32_t qa_box[3] = {32u, 128u, 1u};
  if (!encode_bhlc(&maps[0], q, d.d, d.Lq, d.Hq, d.B, sl, static_cast<int64_t>(d.Lq) * d.d,
                   static_cast<int64_t>(d.Hq) * d.Lq * d.d, bw) ||
      !encode_bhlc(&maps[1], k, d.d, d.Lk, d.Hkv, d.B, sl, static_cast<int64_t>(d.Lk) * d.d,
                   static_cast<int64_t>(d.Hkv) * d.Lk * d.d, bw) ||
      !encode_bhlc(&maps[2], v, d.dv, d.Lk, d.Hkv, d.B, slv, static_cast<int64_t>(d.Lk) * d.dv,
                   static_cast<int64_t>(d.Hkv) * d.Lk * d.dv, bwv) ||
      !encode_bhlc(&maps[3], dout, d.dv, d.Lq, d.Hq, d.B, slv, static_cast<int64_t>(d.Lq) * d.dv,
                   static_cast<int64_t>(d.Hq) * d.Lq * d.dv, bwv) ||
      !encode_rows_f32(&maps[4], p.l2, static_cast<int64_t>(d.B) * d.Hq, d.Lq) ||
      !encode_rows_f32(&maps[5], p.dvec, static_cast<int64_t>(d.B) * d.Hq, d.Lq) ||
      !encode(&maps[6], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.dq_acc, qa_dims, qa_str, qa_box,
              CU_TENSOR_MAP_SWIZZLE_128B))
    return cuda_fail("cuTensorMapEncodeTiled", cudaSuccess);
  return launched("backward kernel launch", fl::launch_bwd(d.d, d.dv, d.score_mod, maps, p, static_cast<cudaStream_t>(d.stream)));
}

}  // namespace

fl_status fl_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                      const fl_attn_desc* desc) {
  return attn_bwd_run(q, k, v, out, dout, lse, dq, dk, dv, workspace, workspace_bytes, desc, 1.0f, false);
}

size_t fl_diffattn_bwd_workspace_size(const fl_attn_desc* desc) {
  if (!desc || desc->B < 1 || desc->Hq < 1 || desc->Lq < 1) return 0;
  const size_t rows = static_cast<size_t>(desc->B) * desc->Hq * desc->Lq;
  // O1, O2 (bf16, dv = 128), the backward's workspace (d = 64), LSE1, LSE2
  return rows * (2 * 128 * 2 + (64 + 2) * 4 + 2 * 4);
}

fl_status fl_diffattn_bwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                          const void* dout, float lambda, void* dq1, void* dk1, void* dq2, void* dk2, void* dv,
                          void* workspace, size_t workspace_bytes, const fl_attn_desc* desc) {
  if (!desc || !q1 || !k1 || !q2 || !k2 || !v || !dout || !dq1 || !dk1 || !dq2 || !dk2 || !dv)
    return FL_ERR_INVALID_ARG;
  const fl_attn_desc& d = *desc;
  if (d.B < 1 || d.Hq < 1 || d.Lq < 1 || d.Hkv != d.Hq || d.Lk != d.Lq) return FL_ERR_INVALID_ARG;
  if (!std::isfinite(lambda) || !std::isfinite(d.scale)) return FL_ERR_INVALID_ARG;
  if (d.d != 64 || d.dv != 128) return FL_ERR_UNSUPPORTED;
  if (d.mask_kind != FL_MASK_NONE && d.mask_kind != FL_MASK_CAUSAL) return FL_ERR_UNSUPPORTED;
  if (d.score_mod != FL_SCORE_NONE) return FL_ERR_UNSUPPORTED;
  for (int i = 0; i < 4; ++i)
    if (d.q_strides[i] || d.k_strides[i] || d.v_strides[i] || d.o_strides[i]) return FL_ERR_UNSUPPORTED;
  const void* ptrs[] = {q1, k1, q2, k2, v, dout, dq1, dk1, dq2, dk2, dv, workspace};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FL_ERR_ALIGNMENT;
  if (d.Lq % 4 != 0) return FL_ERR_UNSUPPORTED;  // as fl_attn_bwd
  const size_t need = fl_diffattn_bwd_workspace_size(desc);
  if (!workspace || workspace_bytes < need) return FL_ERR_INVALID_ARG;

  // each branch is softmax attention (d 64, dv 128) over the shared V; the
  // fused forward keeps only O1 - lambda O2, so O1, O2 and their LSEs are
  // recomputed into the workspace: [O1 | O2 | backward workspace | LSE1 | LSE2]
  fl_attn_desc a = d;
  a.scale = d.scale > 0.f ? d.scale : 0.125f;
  const size_t rows = static_cast<size_t>(d.B) * d.Hq * d.Lq;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* o1 = ws;
  void* o2 = ws + rows * 256;
  void* bws = ws + rows * 512;
  const size_t bws_bytes = rows * (64 + 2) * 4;
  float* lse1 = reinterpret_cast<float*>(ws + rows * 512 + bws_bytes);
  float* lse2 = lse1 + rows;
  fl_status st = fl_attn_fwd(q1, k1, v, o1, lse1, &a);
  if (st == FL_OK) st = fl_attn_fwd(q2, k2, v, o2, lse2, &a);
  // d/dO1 = dout, d/dO2 = -lambda dout; dV sums both branches
  if (st == FL_OK) st = attn_bwd_run(q1, k1, v, o1, dout, lse1, dq1, dk1, dv, bws, bws_bytes, &a, 1.0f, false);
  if (st == FL_OK) st = attn_bwd_run(q2, k2, v, o2, dout, lse2, dq2, dk2, dv, bws, bws_bytes, &a, -lambda, true);
  return st;
}

size_t fl_attn_decode_workspace_size(const fl_attn_desc* desc) {
  if (!desc || desc->B < 1 || desc->Hkv < 1 || desc->Lk < 1) return 0;
  DeviceState* ds = nullptr;
  if (device_state(&ds) != FL_OK) return 0;
  int ns = 1, chunk = 0;
  return decode_workspace(*desc, ds->sm_count, &ns, &chunk);
}

fl_status fl_attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
                             const int32_t* kv_len, void* workspace, size_t workspace_bytes,
                             const fl_attn_desc* desc) {
  const fl_status chk = decode_check(q, k_cache, v_cache, out, lse, kv_len, desc);
  if (chk != FL_OK) return chk;
  const fl_attn_desc& d = *desc;
  DeviceState* ds = nullptr;
  const fl_status st = device_state(&ds);
  if (st != FL_OK) return st;
  fl::DecodeParams p{};
  const size_t need = decode_workspace(d, ds->sm_count, &p.n_split, &p.chunk);
  if (need > 0 && (!workspace || workspace_bytes < need)) return FL_ERR_INVALID_ARG;
  if (need > 0 && !aligned16(workspace)) return FL_ERR_ALIGNMENT;
  p.q = q; p.out = out; p.lse = lse; p.kv_len = kv_len; p.slopes = d.alibi_slopes;
  p.B = d.B; p.Hq = d.Hq; p.Hkv = d.Hkv; p.Lq = d.Lq; p.Lmax = d.Lk;
  p.rows = static_cast<int64_t>(d.B) * d.Hq * d.Lq;
  if (need > 0) {
    p.opart = static_cast<float*>(workspace);
    p.lpart = p.opart + static_cast<int64_t>(p.n_split) * p.rows * d.d;
  }
  p.scale = d.scale > 0.f ? d.scale : 1.0f / std::sqrt(static_cast<float>(d.d));
  p.softcap = d.softcap;
  p.score_mod = d.score_mod;
  p.causal = d.mask_kind == FL_MASK_CAUSAL;
  p.status = ds->status;
  p.timeout_ns = wait_ns(d.wait_limit_ms);
  if (static_cast<int64_t>(d.B) * d.Hkv * p.n_split > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  CUtensorMap maps[2];
  const int64_t sl = d.d, sh = static_cast<int64_t>(d.Lk) * d.d, sb = static_cast<int64_t>(d.Hkv) * d.Lk * d.d;
  if (!encode_bhlc(&maps[0], k_cache, d.d, d.Lk, d.Hkv, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[1], v_cache, d.d, d.Lk, d.Hkv, d.B, sl, sh, sb, 64))
    return cuda_fail("cuTensorMapEncodeTiled", cudaSuccess);
  return launched("decode kernel launch", fl::launch_decode(d.d, maps, p, static_cast<cudaStream_t>(d.stream)));
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
  if (lse && !aligned4(lse)) return FL_ERR_ALIGNMENT;

  DeviceState* ds = nullptr;
  fl_status st = device_state(&ds);
  if (st != FL_OK) return st;

  const int H = d.Hq, L = d.Lq;
  KParams p{};
  p.B = d.B; p.Hq = H; p.Hkv = H; p.Lq = L; p.Lk = L; p.group = 1;
  p.n_qtiles = (L + fl::kBlockM - 1) / fl::kBlockM;
  const float scale = d.scale > 0.f ? d.scale : 0.125f;
  p.scale = scale;
  p.scale_log2 = scale * static_cast<float>(kLog2e);
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

  CUtensorMap maps[8];
  const int64_t sl = 64, sh = static_cast<int64_t>(L) * 64, sb = static_cast<int64_t>(H) * L * 64;
  if (!encode_bhlc(&maps[0], q1, 64, L, H, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[1], k1, 64, L, H, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[2], v, 128, L, H, d.B, 128, static_cast<int64_t>(L) * 128,
                   static_cast<int64_t>(H) * L * 128, 64) ||
      !encode_bhlc(&maps[3], q2, 64, L, H, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[4], k2, 64, L, H, d.B, sl, sh, sb, 64) ||
      !encode_bhlc(&maps[5], out, 128, L, H, d.B, 128, static_cast<int64_t>(L) * 128,
                   static_cast<int64_t>(H) * L * 128, 64))
    return cuda_fail("cuTensorMapEncodeTiled", cudaSuccess);
  maps[6] = maps[0];
  maps[7] = maps[0];
  const int grid = static_cast<int>(units < ds->sm_count ? units : ds->sm_count);
  return launched("differential attention launch", fl::launch_diff_d64(maps, p, grid, static_cast<cudaStream_t>(d.stream)));
}

fl_status fl_evoformer_gated_attn_fwd(const void* q, const void* k, const void* v, const float* pair_bias,
                                      const float* mask_bias, const void* gate, void* out, float* lse, int32_t B,
                                      int32_t N_seq, int32_t N_res, int32_t H, int32_t d, float scale,
                                      void* stream) {
  if (!q || !k || !v || !gate || !out) return FL_ERR_INVALID_ARG;
  if (B < 1 || N_seq < 1 || N_res < 1 || H < 1 || !std::isfinite(scale)) return FL_ERR_INVALID_ARG;
  if (d != 32) return FL_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(gate) || !aligned16(out)) return FL_ERR_ALIGNMENT;
  if ((pair_bias && !aligned16(pair_bias)) || (mask_bias && !aligned16(mask_bias)) || (lse && !aligned4(lse)))
    return FL_ERR_ALIGNMENT;
  if ((pair_bias || mask_bias) && (N_res % 4) != 0) return FL_ERR_UNSUPPORTED;  // 16-byte bias rows

  DeviceState* ds = nullptr;
  fl_status st = device_state(&ds);
  if (st != FL_OK) return st;

  const int64_t Bf = static_cast<int64_t>(B) * N_seq;
  KParams p{};
  p.B = static_cast<int>(Bf); p.Hq = H; p.Hkv = H; p.Lq = N_res; p.Lk = N_res; p.group = 1;
  p.n_qtiles = (N_res + fl::kBlockM - 1) / fl::kBlockM;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d));
  p.scale = sc;
  p.scale_log2 = sc * static_cast<float>(kLog2e);
  p.mask_kind = fl::MASK_NONE;
  p.out = out; p.o_sl = d; p.o_sh = static_cast<int64_t>(N_res) * d; p.o_sb = static_cast<int64_t>(H) * N_res * d;
  p.lse = lse;
  p.gate = gate;
  p.evo_b = B; p.evo_h = H; p.evo_n = N_seq;
  p.has_pb = pair_bias != nullptr;
  p.has_mb = mask_bias != nullptr;
  p.status = ds->status;
  p.timeout_ns = kDefaultWaitNs;
  p.dbg_skip_tile = -1;
  p.slot_mode = fl::SLOT_PAIR;
  p.chunked = 1;
  const int64_t units = static_cast<int64_t>(B) * H * p.n_qtiles * ((N_seq + 1) / 2);
  if (units > 0x7fffffff || Bf > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(units);

  CUtensorMap maps[8];
  const int bw = box_width(d);
  const int64_t sl = d, sh = static_cast<int64_t>(N_res) * d, sb = static_cast<int64_t>(H) * N_res * d;
  if (!encode_bhlc(&maps[0], q, d, N_res, H, Bf, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[1], k, d, N_res, H, Bf, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[2], v, d, N_res, H, Bf, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[5], out, d, N_res, H, Bf, sl, sh, sb, bw))
    return cuda_fail("cuTensorMapEncodeTiled", cudaSuccess);
  maps[3] = maps[0];
  maps[4] = maps[1];
  maps[6] = maps[0];
  maps[7] = maps[0];
  if (pair_bias && !encode_pair_bias(&maps[6], pair_bias, B, H, N_res))
    return cuda_fail("cuTensorMapEncodeTiled (pair bias)", cudaSuccess);
  if (mask_bias && !encode_rows_f32(&maps[7], mask_bias, Bf, N_res))
    return cuda_fail("cuTensorMapEncodeTiled (mask bias)", cudaSuccess);
  const int grid = static_cast<int>(units < ds->sm_count ? units : ds->sm_count);
  return launched("Evoformer kernel launch", fl::launch_evo_row(maps, p, grid, static_cast<cudaStream_t>(stream)));
}

fl_status fl_evoformer_col_gated_attn_fwd(const void* q, const void* k, const void* v, const float* mask_bias,
                                          const void* gate, void* out, float* lse, int32_t B, int32_t N_seq,
                                          int32_t N_res, int32_t H, int32_t d, float scale, void* stream) {
  if (!q || !k || !v || !gate || !out) return FL_ERR_INVALID_ARG;
  if (B < 1 || N_seq < 1 || N_res < 1 || H < 1 || !std::isfinite(scale)) return FL_ERR_INVALID_ARG;
  if (d != 32 && d != 64) return FL_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(gate) || !aligned16(out)) return FL_ERR_ALIGNMENT;
  if ((mask_bias && !aligned16(mask_bias)) || (lse && !aligned4(lse))) return FL_ERR_ALIGNMENT;
  if (mask_bias && (N_seq % 4) != 0) return FL_ERR_UNSUPPORTED;  // 16-byte bias rows

  DeviceState* ds = nullptr;
  fl_status st = device_state(&ds);
  if (st != FL_OK) return st;

  // heads of the kernel: (h, r) with stride d; rows: MSA rows s with stride H * N_res * d
  const int64_t HR = static_cast<int64_t>(H) * N_res;
  if (HR > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  KParams p{};
  p.B = B; p.Hq = static_cast<int>(HR); p.Hkv = p.Hq; p.Lq = N_seq; p.Lk = N_seq; p.group = 1;
  p.n_qtiles = (N_seq + fl::kBlockM - 1) / fl::kBlockM;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d));
  p.scale = sc;
  p.scale_log2 = sc * static_cast<float>(kLog2e);
  p.mask_kind = fl::MASK_NONE;
  const int64_t sl = HR * d, sh = d, sb = static_cast<int64_t>(N_seq) * HR * d;
  p.out = out; p.o_sl = sl; p.o_sh = sh; p.o_sb = sb;
  p.lse = lse;
  p.gate = gate;
  p.evo_b = B; p.evo_h = H; p.evo_n = N_res;
  p.has_pb = 0;
  p.has_mb = mask_bias != nullptr;
  p.status = ds->status;
  p.timeout_ns = kDefaultWaitNs;
  p.dbg_skip_tile = -1;
  p.slot_mode = fl::SLOT_PAIR;
  p.chunked = 1;
  const int64_t units = static_cast<int64_t>(B) * H * ((N_res + 1) / 2) * p.n_qtiles;
  if (units > 0x7fffffff) return FL_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(units);

  CUtensorMap maps[8];
  const int bw = box_width(d);
  if (!encode_bhlc(&maps[0], q, d, N_seq, HR, B, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[1], k, d, N_seq, HR, B, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[2], v, d, N_seq, HR, B, sl, sh, sb, bw) ||
      !encode_bhlc(&maps[5], out, d, N_seq, HR, B, sl, sh, sb, bw))
    return cuda_fail("cuTensorMapEncodeTiled", cudaSuccess);
  maps[3] = maps[0];
  maps[4] = maps[1];
  maps[6] = maps[0];
  maps[7] = maps[0];
  if (mask_bias && !encode_rows_f32(&maps[7], mask_bias, static_cast<int64_t>(B) * N_res, N_seq))
    return cuda_fail("cuTensorMapEncodeTiled (mask bias)", cudaSuccess);
  const int grid = static_cast<int>(units < ds->sm_count ? units : ds->sm_count);
  return launched("Evoformer kernel launch", fl::launch_evo_col(d, maps, p, grid, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
