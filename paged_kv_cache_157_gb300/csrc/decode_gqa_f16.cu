// Explicit instantiation of the GQA decode kernels for __half storage.
#include "decode_gqa_launch.cuh"

namespace kvc {
template kvc_status gqa_dispatch<__half, false>(const GqaParams&, int, int, int, size_t, cudaStream_t, int,
                                                         int*);
}  // namespace kvc
