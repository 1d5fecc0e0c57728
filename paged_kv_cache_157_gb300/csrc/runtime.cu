// Status strings, per-thread error messages, options, device properties and
// the device error word.
#include <cstdio>
#include <mutex>
#include <vector>

#include "kvc_internal.h"

// One error word per device (each device that loads this library gets its
// own copy of this variable). Kernels receive its address as an argument.
static __device__ unsigned int g_kvc_error_word;

namespace kvc {

static thread_local std::string t_message;

kvc_status fail(kvc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_message = buf;
  return s;
}

void clear_error() { t_message.clear(); }

kvc_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

static std::mutex g_dev_mutex;
static std::vector<DeviceInfo*> g_devices;

kvc_status current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (dev >= static_cast<int>(g_devices.size())) g_devices.resize(dev + 1, nullptr);
  if (g_devices[dev] == nullptr) {
    DeviceInfo* info = new DeviceInfo();
    info->device = dev;
    if ((e = cudaDeviceGetAttribute(&info->num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&info->max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&info->l2_bytes, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) {
      delete info;
      return cuda_fail(e, "cudaDeviceGetAttribute");
    }
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_kvc_error_word);
    if (e != cudaSuccess) {
      delete info;
      return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    }
    info->error_word = static_cast<unsigned int*>(addr);
    g_devices[dev] = info;
  }
  *out = g_devices[dev];
  return KVC_OK;
}

static int64_t g_options[7] = {0, 0, 0, 0, 0, 0, 0};

int64_t option(kvc_option opt) { return g_options[static_cast<int>(opt)]; }

static kvc_status read_and_clear_flags(cudaStream_t stream, uint32_t* flags) {
  DeviceInfo* dev = nullptr;
  kvc_status s = current_device(&dev);
  if (s != KVC_OK) return s;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int host = 0;
  e = cudaMemcpyFromSymbol(&host, g_kvc_error_word, sizeof(host));
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_kvc_error_word, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  *flags = host;
  return KVC_OK;
}

kvc_status finish_call(cudaStream_t stream) {
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "kernel launch");
  }
  if (g_options[KVC_OPT_CHECKED] == 0) return KVC_OK;
  uint32_t flags = 0;
  kvc_status s = read_and_clear_flags(stream, &flags);
  if (s != KVC_OK) return s;
  if (flags != 0) return fail(KVC_ERR_OUT_OF_RANGE, "device error word 0x%x", flags);
  return KVC_OK;
}

}  // namespace kvc

extern "C" {

int kvc_abi_version(void) { return KVC_ABI_VERSION; }

const char* kvc_status_string(kvc_status s) {
  switch (s) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_INVALID_ARG: return "KVC_ERR_INVALID_ARG";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED";
    case KVC_ERR_NO_BLOCKS: return "KVC_ERR_NO_BLOCKS";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA";
    case KVC_ERR_OUT_OF_RANGE: return "KVC_ERR_OUT_OF_RANGE";
    case KVC_ERR_WORKSPACE: return "KVC_ERR_WORKSPACE";
  }
  return "KVC_ERR_UNKNOWN";
}

const char* kvc_last_error_message(void) { return kvc::t_message.c_str(); }

kvc_status kvc_set_option(kvc_option opt, int64_t value) {
  int o = static_cast<int>(opt);
  if (o < 0 || o > 6) return kvc::fail(KVC_ERR_INVALID_ARG, "unknown option %d", o);
  if (value < 0) return kvc::fail(KVC_ERR_INVALID_ARG, "option value must be >= 0");
  if (opt == KVC_OPT_CHECKED && value > 1) return kvc::fail(KVC_ERR_INVALID_ARG, "checked mode is 0 or 1");
  if (opt == KVC_OPT_GQA_ENGINE && value > 3) return kvc::fail(KVC_ERR_INVALID_ARG, "GQA engine is 0, 1, 2 or 3");
  if (opt == KVC_OPT_DYNAMIC_SHARE && value > 256) return kvc::fail(KVC_ERR_INVALID_ARG, "dynamic share is 0 to 256");
  if (opt == KVC_OPT_DYNAMIC_CHUNK && value > 4096) return kvc::fail(KVC_ERR_INVALID_ARG, "dynamic chunk is 0 to 4096");
  if (opt == KVC_OPT_WAIT_POLLS && value > (1 << 20)) return kvc::fail(KVC_ERR_INVALID_ARG, "wait polls is 0 to 2^20");
  kvc::g_options[o] = value;
  return KVC_OK;
}

kvc_status kvc_set_checked(int enabled) { return kvc_set_option(KVC_OPT_CHECKED, enabled != 0 ? 1 : 0); }

kvc_status kvc_get_option(kvc_option opt, int64_t* value) {
  int o = static_cast<int>(opt);
  if (o < 0 || o > 6 || value == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "bad option query");
  *value = kvc::g_options[o];
  return KVC_OK;
}

kvc_status kvc_get_error_flags(kvc_stream stream, uint32_t* flags) {
  if (flags == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "flags is NULL");
  return kvc::read_and_clear_flags(static_cast<cudaStream_t>(stream), flags);
}

}  // extern "C"
