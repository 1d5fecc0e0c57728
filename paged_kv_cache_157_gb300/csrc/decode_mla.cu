// MLA absorbed decode (tensor cores). Placeholder until the tcgen05 kernel lands.
#include "kvc_internal.h"

extern "C" {

kvc_status kvc_decode_mla_workspace_size(int, int, int, int, int, int, size_t* bytes) {
  if (bytes) *bytes = 0;
  return kvc::fail(KVC_ERR_UNSUPPORTED, "MLA decode not built yet");
}

kvc_status kvc_decode_attention_mla(const void*, const void*, const int32_t*, int, const int32_t*, int, float, int,
                                    int, int, int, int64_t, kvc_dtype, void*, kvc_dtype, void*, size_t,
                                    kvc_stream) {
  return kvc::fail(KVC_ERR_UNSUPPORTED, "MLA decode not built yet");
}

}  // extern "C"
