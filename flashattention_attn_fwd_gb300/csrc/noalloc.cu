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

#include <cstdint>
#include <mutex>

#include "flattn.h"
#include "host.h"

namespace {

// Scratch of the allocation-free path: 256 bytes in every GPU that loads the
// library, held until the process exits.  The attention kernel uses two
// words of it ([0] error bits, [1] which wait gave up).
constexpr int kScratchWords = 64;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kScratchWords];
constexpr size_t kStatusBytes = 2 * sizeof(uint32_t);
constexpr int kMaxDevices = 64;

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
  // the device's primary context current on this thread (the tensor-map
  // encoder is a driver call)
  if (cudaSetDevice(dev) != cudaSuccess) return FL_ERR_CUDA;
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
  if (!q && !k && !v && !out && !lse) {
    NoAllocDevice* nd = nullptr;
    const fl_status st = na_setup(&nd);
    return st != FL_OK ? st : na_query(nd, static_cast<cudaStream_t>(desc->stream));
  }
  // argument errors come back before any CUDA call
  const fl_status chk = fl::attn_fwd_check(q, k, v, out, lse, desc);
  if (chk != FL_OK) return chk;
  // The scratch this launch needs (the kernel's status words) must fit the
  // fixed array; it does not grow with the problem size.
  if (kStatusBytes > sizeof(g_noalloc_scratch)) return FL_ERR_UNSUPPORTED;
  NoAllocDevice* nd = nullptr;
  const fl_status st = na_setup(&nd);
  if (st != FL_OK) return st;
  // the same validation, parameters, tensor maps and launch as fl_attn_fwd;
  // only the status words differ
  return fl::attn_fwd_launch(q, k, v, out, lse, desc, nd->scratch, nd->sm_count);
}

}  // extern "C"
