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
  float* rec_o;   // [G*2, GH, D] partial outputs (stream mode)
  float* rec_ml;  // [G*2, GH, 2] (max in log2 units, sum)
  unsigned int* counters;  // [units] records seen per split unit; zero between calls
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
  int unit_mode;  // 1: CTA u handles unit u completely (no records)
  float qscale;   // scale * log2(e)
};

constexpr int kGqaWarps = 4;
constexpr float kNegInf = -__builtin_huge_valf();

// Shared-memory carve-up, identical on host and device.
struct GqaSmem {
  size_t stage_off, bar_off, o_off, ml_off, scan_off, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline GqaSmem gqa_smem_layout(int elt_bytes, int D, int GH, int block_size, int stages,
                                                  int batch) {
  GqaSmem s;
  const size_t page = static_cast<size_t>(block_size) * D * elt_bytes;
  s.stage_off = 0;
  s.bar_off = align_up(s.stage_off + static_cast<size_t>(kGqaWarps) * stages * 2 * page, 16);
  s.o_off = align_up(s.bar_off + static_cast<size_t>(kGqaWarps) * stages * 8, 16);
  s.ml_off = s.o_off + static_cast<size_t>(kGqaWarps) * GH * D * 4;
  s.scan_off = align_up(s.ml_off + static_cast<size_t>(kGqaWarps) * GH * 2 * 4, 16);
  s.total = s.scan_off + static_cast<size_t>(batch + 1 + 32) * 4;
  return s;
}

template <typename T>
kvc_status gqa_dispatch(const GqaParams& p, int D, int GH, int grid, size_t smem, cudaStream_t stream, int mode,
                        int* occ);

}  // namespace kvc
