// Explicit instantiation of the sliding-window GQA decode kernels for __nv_bfloat16 storage.
#include "decode_gqa_launch.cuh"

namespace kvc {
template kvc_status gqa_dispatch<__nv_bfloat16, true>(const GqaParams&, int, int, int, size_t, cudaStream_t, int,
                                                         int*);
}  // namespace kvc
