// Launch of the warp-MMA GQA decode kernel (one explicit instantiation file
// per cache dtype so they compile in parallel).
#pragma once

#include "decode_gqa_mma.cuh"
#include "kvc_internal.h"

namespace kvc {

// mode 0: launch; mode 1: only report the occupancy (CTAs per SM) in *occ.
template <typename T, int GH, bool EXT, int Q8 = 0>
static kvc_status gqa_mma_run(const GqaParams& p, int grid, size_t smem, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream, int mode, int* occ) {
  auto* k = gqa_mma_kernel<T, GH, EXT, Q8>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gqa mma)");
  if (mode == 1) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, kMmaThreads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    return KVC_OK;
  }
  // May start while the previous kernel of the stream runs; every thread
  // waits for it before it touches a caller buffer.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k, tk, tv, p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(gqa mma)");
  if (p.unit_mode) return KVC_OK;
  // The merge of split units, right behind (it may be scheduled early; it
  // waits for the decode grid before it reads anything).
  auto* mk = gqa_mma_merge_kernel<GH, EXT>;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(static_cast<unsigned int>(static_cast<int64_t>(p.batch) * p.n_chunks * p.n_hsub * p.hc *
                                                mma_warps_per_kvhead(GH)));
  mcfg.blockDim = dim3(merge_threads(GH));
  mcfg.dynamicSmemBytes = 0;
  mcfg.stream = stream;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&mcfg, mk, p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(gqa mma merge)");
  return KVC_OK;
}

template <typename T, bool EXT>
kvc_status gqa_mma_dispatch(const GqaParams& p, int GH, int grid, size_t smem, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t stream, int mode, int* occ) {
  switch (GH) {
    case 1: return gqa_mma_run<T, 1, EXT>(p, grid, smem, tk, tv, stream, mode, occ);
    case 2: return gqa_mma_run<T, 2, EXT>(p, grid, smem, tk, tv, stream, mode, occ);
    case 4: return gqa_mma_run<T, 4, EXT>(p, grid, smem, tk, tv, stream, mode, occ);
    case 8: return gqa_mma_run<T, 8, EXT>(p, grid, smem, tk, tv, stream, mode, occ);
    case 16: return gqa_mma_run<T, 16, EXT>(p, grid, smem, tk, tv, stream, mode, occ);
  }
  return fail(KVC_ERR_UNSUPPORTED, "head subgroup %d", GH);
}

template <int Q8>
kvc_status gqa_mma_dispatch_q8(const GqaParams& p, int GH, int grid, size_t smem, const CUtensorMap& tk,
                               const CUtensorMap& tv, cudaStream_t stream, int mode, int* occ) {
  using B = __nv_bfloat16;
  switch (GH) {
    case 1: return gqa_mma_run<B, 1, false, Q8>(p, grid, smem, tk, tv, stream, mode, occ);
    case 2: return gqa_mma_run<B, 2, false, Q8>(p, grid, smem, tk, tv, stream, mode, occ);
    case 4: return gqa_mma_run<B, 4, false, Q8>(p, grid, smem, tk, tv, stream, mode, occ);
    case 8: return gqa_mma_run<B, 8, false, Q8>(p, grid, smem, tk, tv, stream, mode, occ);
    case 16: return gqa_mma_run<B, 16, false, Q8>(p, grid, smem, tk, tv, stream, mode, occ);
  }
  return fail(KVC_ERR_UNSUPPORTED, "head subgroup %d", GH);
}

}  // namespace kvc
