// Explicit instantiation of the warp-MMA GQA decode kernels for FP8 (e4m3) caches
// with bf16 queries (single-token full attention).
#include "decode_gqa_mma_launch.cuh"

namespace kvc {
template kvc_status gqa_mma_dispatch_q8<1>(const GqaParams&, int, int, size_t, const CUtensorMap&, const CUtensorMap&,
                                            cudaStream_t, int, int*);
}  // namespace kvc
