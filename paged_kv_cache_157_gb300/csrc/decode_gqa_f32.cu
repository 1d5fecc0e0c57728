// Explicit instantiation of the GQA decode kernels for float storage.
#include "decode_gqa_launch.cuh"

namespace kvc {
template kvc_status gqa_dispatch<float, false>(const GqaParams&, int, int, int, size_t, cudaStream_t, int,
                                                         int*);
}  // namespace kvc
