// Explicit instantiation of the warp-MMA GQA decode kernels for __half caches
// (single-token full attention, and the extensions: window, several tokens,
// start rows, LSE output).
#include "decode_gqa_mma_launch.cuh"

namespace kvc {
template kvc_status gqa_mma_dispatch<__half, false>(const GqaParams&, int, int, size_t, const CUtensorMap&,
                                                const CUtensorMap&, cudaStream_t, int, int*);
template kvc_status gqa_mma_dispatch<__half, true>(const GqaParams&, int, int, size_t, const CUtensorMap&,
                                               const CUtensorMap&, cudaStream_t, int, int*);
}  // namespace kvc
