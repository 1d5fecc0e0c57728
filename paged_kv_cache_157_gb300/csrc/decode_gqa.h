// Parameters and shared-memory layout of the GQA decode kernels, shared by
// the host planner and the device code.
#pragma once

#include <cuda.h>
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
  float* rec_o;   // [G*2, kGqaWarps/HW * GH, D] partial outputs of the G CTAs (split mode)
  float* rec_ml;  // [G*2, kGqaWarps/HW * GH, 2] (max in log2 units, sum)
  unsigned int* counters;  // [units] records seen per split unit; zero between calls
  unsigned int* err;
  int64_t num_blocks;
  int batch;
  int n_q_heads;
  int n_kv_heads;
  int group;     // n_q_heads / n_kv_heads
  int n_hsub;    // group / GH
  int hc;        // kv heads per CTA (a chunk): consecutive heads of a block, read as one copy
  int n_chunks;  // n_kv_heads / hc
  int block_size;
  int max_blocks;
  int out_dtype;
  int stages;
  int unit_mode;  // 1: CTA u handles unit u completely (no records)
  int window;     // sliding window: attend the newest `window` rows (0: all rows)
  int n_tok;      // new query tokens per sequence (q and out are [batch, n_tok, n_q_heads, D])
  int causal;     // n_tok > 1: 1 = token t sees rows up to n - n_tok + t; 0 = every row (a shared-prefix pass)
  float* lse;     // non-NULL: log2 of each output row's softmax denominator plus its max (log2 units) [rows]
  const int32_t* row_start;  // row_div > 0: sequence b attends rows from row_start[b / row_div]
  int row_div;
  const float* k_scale;  // FP8 caches: per-channel K scales [n_kv_heads, head_dim]
  const float* v_scale;  // FP8 caches: per-token V scales [num_blocks, n_kv_heads, block_size]
  float qscale;   // scale * log2(e)
  // warp-MMA kernel: dynamic tail of the work split
  unsigned int* sched;  // [claim counter, finished CTAs] in the workspace; zero between calls
  int dyn_share;        // positions claimed at run time, in 1/256 of all (0: none)
  int dyn_chunk;        // positions per claimed chunk (0: no dynamic tail)
  int dyn_min_static;   // keep the dynamic tail only if every CTA still gets this many static positions
  unsigned int wait_polls;  // 0: waits for copied data bounded by ~1 s; N: give up after N polls (test hook)
  // warp-MMA kernel: per unit [record count R][record slots 0 .. list_cap-1], written by the worker that
  // holds the unit's first block and read by the merge kernel; R = 0: no merge (one worker had it whole)
  int* unit_lists;
  int list_cap;
  int64_t rec_slots;        // record slots in the workspace (2 per record pair)
  int pair;                 // warp-MMA kernel, one-byte caches: two cache blocks of a segment per stage
};

#ifndef KVC_GQA_WARPS
#define KVC_GQA_WARPS 4
#endif
#ifndef KVC_GQA_CTAS_PER_SM
#define KVC_GQA_CTAS_PER_SM 2
#endif
constexpr int kGqaWarps = KVC_GQA_WARPS;            // warps per CTA
constexpr int kGqaCtasPerSm = KVC_GQA_CTAS_PER_SM;  // resident CTAs the register and shared-memory budgets aim at
constexpr float kNegInf = -__builtin_huge_valf();

// The GH query heads of a kv head are split over HW warps (GH / HW <= 4
// heads per warp); a CTA covers kGqaWarps / HW kv heads at most.
__host__ __device__ constexpr int gqa_warps_per_kvhead(int GH) { return GH > 4 ? GH / 4 : 1; }
__host__ __device__ constexpr int gqa_max_chunk(int GH) { return kGqaWarps / gqa_warps_per_kvhead(GH); }

// Shared-memory carve-up, identical on host and device. The CTA has one ring
// of `stages` stages, each [K chunk: hc pages][V chunk: hc pages][query rows
// of the unit: hc x GH][FP8 caches only: the chunk's per-token V scales,
// hc x block_size fp32]; every warp has a [heads of the warp][16 rows] fp32
// buffer for the softmax weights of its current tile. elt_bytes is the cache
// element size, q_bytes the query element size, vs_bytes 4 for FP8 caches
// (one scale per row) and 0 otherwise.
struct GqaSmem {
  size_t stage_off, p_off, bar_off, rel_off, misc_off, scan_off, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t gqa_stage_bytes(int elt_bytes, int q_bytes, int vs_bytes, int D, int GH,
                                                  int block_size, int hc) {
  return 2ull * hc * block_size * D * elt_bytes + static_cast<size_t>(hc) * GH * D * q_bytes +
         static_cast<size_t>(hc) * block_size * vs_bytes;
}

__host__ __device__ inline size_t gqa_p_bytes_per_warp(int GH) {
  return static_cast<size_t>(GH / gqa_warps_per_kvhead(GH)) * 16 * 4;
}

__host__ __device__ inline GqaSmem gqa_smem_layout(int elt_bytes, int q_bytes, int vs_bytes, int D, int GH,
                                                  int block_size, int hc, int stages, int batch) {
  GqaSmem s;
  s.stage_off = 0;
  s.p_off = align_up(static_cast<size_t>(stages) *
                         align_up(gqa_stage_bytes(elt_bytes, q_bytes, vs_bytes, D, GH, block_size, hc), 16),
                     16);
  s.bar_off = align_up(s.p_off + kGqaWarps * gqa_p_bytes_per_warp(GH), 16);
  s.rel_off = s.bar_off + static_cast<size_t>(stages) * 8;  // one "full" mbarrier per stage
  s.misc_off = align_up(s.rel_off + static_cast<size_t>(stages) * 8, 16);  // release and issue counts per stage
  s.scan_off = s.misc_off + 16;  // [abort flag, last flags]
  s.total = s.scan_off + static_cast<size_t>(batch + 1 + 32) * 4;
  return s;
}

// Tensor-core decode for kv heads with 8 to 32 queries (n_tok x group):
// bf16/f16 caches, head_dim 128, block size 16/32/64/128, no window.
struct WideArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  void* workspace;
  size_t workspace_bytes;
  int64_t num_blocks;
  int batch, n_q_heads, n_kv_heads, block_size, max_blocks, n_tok;
  int causal;  // several tokens: 1 = causal among them, 0 = every row (a shared-prefix pass)
  float* lse;  // non-NULL: per output row, max + log2(sum) (log2 units)
  kvc_dtype dtype, out_dtype;
  float scale;
  cudaStream_t stream;
};
// Whether the tensor-core kernel takes these shapes (and the engine option
// allows it), and whether the automatic choice picks it (large enough work).
bool wide_supported(int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size, int n_tok,
                    kvc_dtype dtype);
bool wide_preferred(int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_blocks,
                    int n_tok, kvc_dtype dtype);
size_t wide_workspace_bytes(const DeviceInfo* dev, int batch, int n_q_heads, int n_kv_heads, int block_size,
                            int max_blocks, int n_tok);
kvc_status wide_decode(const WideArgs& a, DeviceInfo* dev);

// EXT: kernels with the extensions compiled in (window, several tokens,
// start rows, LSE output).
template <typename T, bool EXT>
kvc_status gqa_dispatch(const GqaParams& p, int D, int GH, int grid, size_t smem, cudaStream_t stream, int mode,
                        int* occ);
// Warp-MMA kernel (bf16/f16 caches, head_dim 128; tk / tv: TMA maps over the
// K and V pools as [num_blocks * n_kv_heads * block_size rows, 128] with
// [hc * block_size x 64] boxes and the 128-byte swizzle).
template <typename T, bool EXT>
kvc_status gqa_mma_dispatch(const GqaParams& p, int GH, int grid, size_t smem, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t stream, int mode, int* occ);

// Warp-MMA kernel over one-byte caches (Q8 = 1: e4m3, 2: int8) with bf16
// queries, head_dim 128; tk / tv: TMA maps over the code pools as
// [num_blocks * n_kv_heads * block_size rows, 128 bytes] with
// [hc * block_size x 128] boxes and the 128-byte swizzle.
template <int Q8>
kvc_status gqa_mma_dispatch_q8(const GqaParams& p, int GH, int grid, size_t smem, const CUtensorMap& tk,
                               const CUtensorMap& tv, cudaStream_t stream, int mode, int* occ);

// FP8 e4m3 caches with bf16 queries (head_dim 64, 128 or 256).
kvc_status gqa_dispatch_fp8(const GqaParams& p, int D, int GH, int grid, size_t smem, cudaStream_t stream, int mode,
                            int* occ);
// INT8 caches with bf16 queries (head_dim 64, 128 or 256).
kvc_status gqa_dispatch_int8(const GqaParams& p, int D, int GH, int grid, size_t smem, cudaStream_t stream, int mode,
                             int* occ);

}  // namespace kvc
