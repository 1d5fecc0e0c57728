// Explicit instantiation of the GQA decode kernels for INT8 caches with bf16
// queries (per-channel K scales, per-token V scales).
#include "decode_gqa_launch.cuh"

namespace kvc {

kvc_status gqa_dispatch_int8(const GqaParams& p, int D, int GH, int grid, size_t smem, cudaStream_t stream, int mode,
                             int* occ) {
  switch (D) {
    case 64: return gqa_run_gh<s8q, 64, __nv_bfloat16, false>(p, GH, grid, smem, stream, mode, occ);
    case 128: return gqa_run_gh<s8q, 128, __nv_bfloat16, false>(p, GH, grid, smem, stream, mode, occ);
    case 256: return gqa_run_gh<s8q, 256, __nv_bfloat16, false>(p, GH, grid, smem, stream, mode, occ);
  }
  return fail(KVC_ERR_UNSUPPORTED, "INT8 decode head_dim %d (supported: 64, 128, 256)", D);
}

}  // namespace kvc
