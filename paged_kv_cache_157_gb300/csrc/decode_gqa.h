// Parameters and shared-memory layout of the GQA decode kernels, shared by
// the host planner and the device code.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "kvc_internal.h"

namespace kvc {

struct GqaParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  float* rec_o;   // [W*2, GH, D] partial outputs of the W workers (split mode)
  float* rec_ml;  // [W*2, GH, 2] (max in log2 units, sum)
  unsigned int* counters;  // [units, warps per stream] records seen per split unit; zero between calls
  unsigned int* err;
  int64_t num_blocks;
  int batch;
  int n_q_heads;
  int n_kv_heads;
  int group;  // n_q_heads / n_kv_heads
  int n_hsub;  // group / GH
  int block_size;
  int max_blocks;
  int out_dtype;
  int stages;
  int unit_mode;  // 1: worker u handles unit u completely (no records)
  float qscale;   // scale * log2(e)
};

#ifndef KVC_GQA_PAIR_WARPS
#define KVC_GQA_PAIR_WARPS 0
#endif
#ifndef KVC_GQA_WARPS
#define KVC_GQA_WARPS 4
#endif
constexpr int kGqaWarps = KVC_GQA_WARPS;  // warps per CTA
constexpr float kNegInf = -__builtin_huge_valf();

// A unit's GH query heads are split over HW warps that share one stream of
// K/V pages; each warp holds GH / HW heads. KVC_GQA_PAIR_WARPS selects
// whether head groups of 2 or more are split over a warp pair (1) or kept in
// one warp (0).
__host__ __device__ constexpr int gqa_warps_per_stream(int GH) {
  return GH > 4 ? GH / 4 : ((KVC_GQA_PAIR_WARPS && GH >= 2) ? 2 : 1);
}
__host__ __device__ constexpr int gqa_streams(int GH) { return kGqaWarps / gqa_warps_per_stream(GH); }

// Shared-memory carve-up, identical on host and device. Each page stream
// has `stages` stages of [K page][V page][the unit's GH query rows].
struct GqaSmem {
  size_t stage_off, bar_off, scan_off, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t gqa_stage_bytes(int elt_bytes, int D, int GH, int block_size) {
  return (2ull * block_size * D + static_cast<size_t>(GH) * D) * elt_bytes;
}

__host__ __device__ inline GqaSmem gqa_smem_layout(int elt_bytes, int D, int GH, int block_size, int stages,
                                                  int batch) {
  GqaSmem s;
  const size_t np = static_cast<size_t>(gqa_streams(GH));
  s.stage_off = 0;
  s.bar_off = align_up(np * stages * gqa_stage_bytes(elt_bytes, D, GH, block_size), 16);
  s.scan_off = align_up(s.bar_off + np * stages * 2 * 8, 16);  // full and empty barrier per stage
  s.total = s.scan_off + static_cast<size_t>(batch + 1 + 32) * 4;
  return s;
}

template <typename T>
kvc_status gqa_dispatch(const GqaParams& p, int D, int GH, int grid, size_t smem, cudaStream_t stream, int mode,
                        int* occ);

}  // namespace kvc
