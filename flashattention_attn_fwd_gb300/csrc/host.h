// Host-side pieces shared by the C ABI entry points (internal header).
#pragma once

#include <cstdint>

#include "flattn.h"

namespace fl {

// Everything fl_attn_fwd does after its own set-up: validation, strides,
// kernel parameters, tensor maps and the launch.  `status` is the device
// status word (two uint32) the kernel reports timeouts in, `sm_count` the
// grid cap.  Allocates nothing.
fl_status attn_fwd_launch(const void* q, const void* k, const void* v, void* out, float* lse,
                          const fl_attn_desc* desc, uint32_t* status, int sm_count);

// Argument checks of attn_fwd_launch alone (no CUDA call).
fl_status attn_fwd_check(const void* q, const void* k, const void* v, void* out, float* lse,
                         const fl_attn_desc* desc);

}  // namespace fl
