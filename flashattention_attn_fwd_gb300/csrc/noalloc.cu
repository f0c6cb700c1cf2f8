// fl_attn_fwd_noalloc: the fused attention forward for callers that must not
// allocate device memory.
//
// fl_attn_fwd allocates (with cudaMalloc, on its first call on a device) the
// small status word its kernel writes when a pipeline wait gives up.  Some
// callers cannot allow that: processes whose device memory is handed out
// only by their own pool or arena and is fully reserved up front (serving
// engines, plugins living inside another framework's allocator), code that
// must not call cudaMalloc while a stream is being captured into a CUDA
// graph, and callers holding a hard device-memory budget.  This entry point
// runs the same kernel but puts that status word in a fixed array compiled
// into the library, so it calls no cudaMalloc, cudaFree or allocating
// library routine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "flattn.h"
#include "kernels.h"
#include "params.h"

namespace {

// Scratch of the allocation-free path: 256 bytes in every GPU that loads the
// library, held until the process exits.  The attention kernel uses two
// words of it ([0] error bits, [1] which wait gave up).
constexpr int kScratchWords = 64;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kScratchWords];
constexpr size_t kStatusBytes = 2 * sizeof(uint32_t);
constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 2000ull * 1000ull * 1000ull;

struct NoAllocDevice {
  bool ready = false;
  int sm_count = 0;
  uint32_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_na_mutex;
NoAllocDevice g_na_dev[kMaxDevices];

// One-time set-up per device, with that device current: the SM count and
// the device address of the scratch array (the array's name is only a host
// stand-in, never a device pointer).
fl_status na_setup(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice& d = g_na_dev[dev];
  if (!d.ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return FL_ERR_CUDA;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return FL_ERR_CUDA;
    d.sm_count = sms;
    d.scratch = static_cast<uint32_t*>(ptr);
    d.ready = true;
  }
  *out = &d;
  return FL_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn na_encode_fn() {
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

bool na_map(CUtensorMap* m, const void* base, int64_t C, int64_t L, int64_t H, int64_t B, int64_t sl, int64_t sh,
            int64_t sb, int box_c) {
  EncodeTiledFn enc = na_encode_fn();
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
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct NaStrides {
  int64_t b, h, l;
};

bool na_strides(const int64_t s[4], int64_t H, int64_t L, int64_t C, NaStrides* out) {
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

bool na_aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool na_strides_aligned(const NaStrides& s) {
  return (s.b * 2) % 16 == 0 && (s.h * 2) % 16 == 0 && (s.l * 2) % 16 == 0;
}

// Status query: wait for the stream, then return and clear the scratch's
// error bits.  No allocation: a synchronous copy into a host stack value.
fl_status na_query(NoAllocDevice* nd, cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FL_ERR_CUDA;
  uint32_t h[2] = {0u, 0u};
  if (cudaMemcpy(h, nd->scratch, kStatusBytes, cudaMemcpyDeviceToHost) != cudaSuccess) return FL_ERR_CUDA;
  if (h[0] == 0u) return FL_OK;
  if (cudaMemset(nd->scratch, 0, kStatusBytes) != cudaSuccess) return FL_ERR_CUDA;
  return (h[0] & 1u) ? FL_ERR_TIMEOUT : FL_ERR_DEVICE_BOUNDS;
}

}  // namespace

extern "C" {

fl_status fl_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                              const fl_attn_desc* desc) {
  if (!desc) return FL_ERR_INVALID_ARG;
  const fl_attn_desc& d = *desc;
  cudaStream_t stream = static_cast<cudaStream_t>(d.stream);
  if (!q && !k && !v && !out && !lse) {
    NoAllocDevice* nd = nullptr;
    const fl_status st = na_setup(&nd);
    return st != FL_OK ? st : na_query(nd, stream);
  }
  if (!q || !k || !v || !out) return FL_ERR_INVALID_ARG;
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
  NaStrides sq, sk, sv, so;
  if (!na_strides(d.q_strides, d.Hq, d.Lq, d.d, &sq) || !na_strides(d.k_strides, d.Hkv, d.Lk, d.d, &sk) ||
      !na_strides(d.v_strides, d.Hkv, d.Lk, d.dv, &sv) || !na_strides(d.o_strides, d.Hq, d.Lq, d.dv, &so))
    return FL_ERR_INVALID_ARG;
  if (!na_aligned(q) || !na_aligned(k) || !na_aligned(v) || !na_aligned(out) || !na_strides_aligned(sq) ||
      !na_strides_aligned(sk) || !na_strides_aligned(sv) || !na_strides_aligned(so))
    return FL_ERR_ALIGNMENT;
  if (d.mask_kind == FL_MASK_DOCUMENT && (reinterpret_cast<uintptr_t>(d.doc_offsets) & 3u)) return FL_ERR_ALIGNMENT;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FL_ERR_ALIGNMENT;
  // The scratch this launch needs (the kernel's status words) must fit the
  // fixed array; it does not grow with the problem size.
  if (kStatusBytes > sizeof(g_noalloc_scratch)) return FL_ERR_UNSUPPORTED;

  NoAllocDevice* nd = nullptr;
  fl_status st = na_setup(&nd);
  if (st != FL_OK) return st;

  fl::KParams p{};
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
  p.status = nd->scratch;
  p.timeout_ns = d.wait_limit_ms ? static_cast<uint64_t>(d.wait_limit_ms) * 1000000ull : kDefaultWaitNs;
  p.dbg_skip_tile = (d.debug_flags & FL_DEBUG_SKIP_KV_LOAD) ? (d.debug_arg < 0 ? 0 : d.debug_arg) : -1;
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
  const int bq = d.d >= 64 ? 64 : d.d;
  if (!na_map(&maps[0], q, d.d, d.Lq, d.Hq, d.B, sq.l, sq.h, sq.b, bq) ||
      !na_map(&maps[1], k, d.d, d.Lk, d.Hkv, d.B, sk.l, sk.h, sk.b, bq) ||
      !na_map(&maps[2], v, d.dv, d.Lk, d.Hkv, d.B, sv.l, sv.h, sv.b, bq) ||
      !na_map(&maps[5], out, d.dv, d.Lq, d.Hq, d.B, so.l, so.h, so.b, bq))
    return FL_ERR_CUDA;
  maps[3] = maps[0];
  maps[4] = maps[1];
  const int grid = static_cast<int>(units < nd->sm_count ? units : nd->sm_count);
  cudaError_t e;
  switch (d.d) {
    case 32: e = fl::launch_attn_d32(d.score_mod, maps, p, grid, stream); break;
    case 64: e = fl::launch_attn_d64(d.score_mod, maps, p, grid, stream); break;
    default: e = fl::launch_attn_d128(d.score_mod, maps, p, grid, stream); break;
  }
  return e == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

}  // extern "C"
