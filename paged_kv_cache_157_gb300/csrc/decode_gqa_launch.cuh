// Kernel selection for the GQA decode path (one explicit instantiation file
// per cache dtype so they compile in parallel).
#pragma once

#include "decode_gqa_impl.cuh"
#include "kvc_internal.h"

namespace kvc {

// mode 0: launch; mode 1: only report the occupancy (CTAs per SM) in *occ.
template <typename T, int D, int GH, typename TQ, bool EXT>
static kvc_status gqa_run(const GqaParams& p, int grid, size_t smem, cudaStream_t stream, int mode, int* occ) {
  auto* k = gqa_decode_kernel<T, D, GH, TQ, EXT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gqa)");
  if (mode == 1) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, kGqaWarps * 32, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    return KVC_OK;
  }
  // The kernel may start while the previous kernel in the stream (the append
  // of this step) is still running; it waits for it before reading the cache.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGqaWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k, p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(gqa)");
  return KVC_OK;
}

template <typename T, int D, typename TQ, bool EXT>
static kvc_status gqa_run_gh(const GqaParams& p, int GH, int grid, size_t smem, cudaStream_t stream, int mode,
                             int* occ) {
  switch (GH) {
    case 1: return gqa_run<T, D, 1, TQ, EXT>(p, grid, smem, stream, mode, occ);
    case 2: return gqa_run<T, D, 2, TQ, EXT>(p, grid, smem, stream, mode, occ);
    case 4: return gqa_run<T, D, 4, TQ, EXT>(p, grid, smem, stream, mode, occ);
    case 8: return gqa_run<T, D, 8, TQ, EXT>(p, grid, smem, stream, mode, occ);
    case 16: return gqa_run<T, D, 16, TQ, EXT>(p, grid, smem, stream, mode, occ);
  }
  return fail(KVC_ERR_UNSUPPORTED, "head subgroup %d", GH);
}

template <typename T, bool EXT>
kvc_status gqa_dispatch(const GqaParams& p, int D, int GH, int grid, size_t smem, cudaStream_t stream, int mode,
                        int* occ) {
  switch (D) {
    case 32: return gqa_run_gh<T, 32, T, EXT>(p, GH, grid, smem, stream, mode, occ);
    case 64: return gqa_run_gh<T, 64, T, EXT>(p, GH, grid, smem, stream, mode, occ);
    case 128: return gqa_run_gh<T, 128, T, EXT>(p, GH, grid, smem, stream, mode, occ);
    case 256: return gqa_run_gh<T, 256, T, EXT>(p, GH, grid, smem, stream, mode, occ);
  }
  return fail(KVC_ERR_UNSUPPORTED, "head_dim %d (supported: 32, 64, 128, 256)", D);
}

}  // namespace kvc
