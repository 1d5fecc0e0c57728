// Explicit instantiation of the GQA decode kernels with the extensions
// (sliding window, several new tokens per sequence) for __half storage.
#include "decode_gqa_launch.cuh"

namespace kvc {
template kvc_status gqa_dispatch<__half, true>(const GqaParams&, int, int, int, size_t, cudaStream_t, int,
                                                         int*);
}  // namespace kvc
