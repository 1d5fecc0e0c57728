// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <string>

#include "../../include/kvc.h"

namespace kvc {

// Records a one-line reason for the calling thread and returns `s`.
kvc_status fail(kvc_status s, const char* fmt, ...);
void clear_error();

// Converts a CUDA error into KVC_ERR_CUDA with the call site in the message.
kvc_status cuda_fail(cudaError_t e, const char* what);

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int max_smem_optin = 0;
  int l2_bytes = 0;
  unsigned int* error_word = nullptr;  // device address of this device's error word
};

// Properties of the current device, cached per device id.
kvc_status current_device(DeviceInfo** out);

// Options (process-wide).
int64_t option(kvc_option opt);

// In checked mode: synchronise `stream`, read and clear the error word.
kvc_status finish_call(cudaStream_t stream);

inline size_t dtype_size(kvc_dtype t) { return t == KVC_F32 ? 4 : 2; }
inline bool dtype_ok(int t) { return t == KVC_F32 || t == KVC_F16 || t == KVC_BF16; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace kvc
