// Host side of kvc_decode_attention: argument checks, work planning,
// workspace carve-up and launch.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "decode_gqa.h"
#include "decode_gqa_mma.cuh"
#include "kvc_device.cuh"

namespace kvc {

namespace {

// Shared memory per CTA (stages, weights, barriers, scan) so that
// kGqaCtasPerSm CTAs fit the 228 KB of an SM (1 KB of it reserved per CTA).
constexpr size_t kStageBudget = (228 * 1024) / kGqaCtasPerSm - 1024;
constexpr int kMaxCtasPerSm = 4;
constexpr int kMinBlocksPerCta = 2 * kGqaWarps;
constexpr int kMaxBatch = 4096;
constexpr int kMaxTokens = 256;  // new tokens per sequence in one multi-token call

struct GqaPlan {
  int GH = 1, n_hsub = 1, stages = 2, hc = 1, n_chunks = 1;
  int ctas_per_sm = kMaxCtasPerSm;  // most CTAs an SM can hold with this plan's shared memory
  int dyn_share = 0, dyn_chunk = 0;  // warp-MMA kernel: dynamic tail of the work split
  int pair = 0;                      // warp-MMA kernel, one-byte caches: two cache blocks per stage
  int64_t units = 0;
  size_t smem = 0;
  size_t rec_bytes_per_cta = 0;  // two records per CTA (per worker on the warp-MMA kernel)
};

// Workspace layout of the CUDA-core kernel: [counters, one per unit and warp
// slot][record outputs][record (max, sum)]. A unit of hc kv heads has hc * HW
// warp slots, so batch * n_kv_heads * n_hsub * HW counters cover every plan.
// (The warp-MMA kernel: [claim counter][unit record lists][records], see
// mma_counter_bytes.)
size_t counter_bytes(int batch, int n_kv_heads, const GqaPlan& pl) {
  return align_up(static_cast<size_t>(batch) * n_kv_heads * pl.n_hsub * gqa_warps_per_kvhead(pl.GH) * 4, 256);
}

// Query heads per unit: the largest power of two up to 16 that divides the
// group. Up to 4 heads share one warp; 8 and 16 split over 2 and 4 warps that
// read the same pages, so each page is loaded once for all of them.
int head_subgroup(int group) {
  for (int gh = 16; gh > 1; gh >>= 1)
    if (group % gh == 0) return gh;
  return 1;
}

// elt: cache element bytes; q_elt: query element bytes; vsb: V-scale bytes
// per cached row (4 for FP8 caches, else 0). n_tok new tokens per sequence
// give each kv head n_tok * group (virtual) query heads that share its pages.
kvc_status make_plan(int batch, int n_q_heads, int n_kv_heads, int D, int bs, int elt, int q_elt, int vsb, int max_smem,
                     GqaPlan* pl, int n_tok = 1) {
  const int group = n_tok * (n_q_heads / n_kv_heads);
  pl->GH = head_subgroup(group);
  pl->n_hsub = group / pl->GH;
  // kv heads per CTA: the largest power of two the CTA's warps can hold that
  // divides n_kv_heads; their pages of a block are adjacent, so one copy
  // moves all of them
  int hc = 1;
  while (hc * 2 <= gqa_max_chunk(pl->GH) && n_kv_heads % (hc * 2) == 0) hc *= 2;
  const size_t scan = static_cast<size_t>(batch + 1 + 32) * 4;
  const size_t fixed = scan + kGqaWarps * gqa_p_bytes_per_warp(pl->GH) + 8 * 16 + 16 + 512;
  const size_t budget = kStageBudget > fixed ? kStageBudget - fixed : 0;
  int S = 1;
  for (;;) {
    const size_t stage = align_up(gqa_stage_bytes(elt, q_elt, vsb, D, pl->GH, bs, hc), 16);
    S = std::max(1, std::min(static_cast<int>(budget / stage), 8));
    if (S >= 2 || hc == 1) break;
    hc /= 2;  // keep at least two stages in flight
  }
  GqaSmem L = gqa_smem_layout(elt, q_elt, vsb, D, pl->GH, bs, hc, S, batch);
  while (S > 1 && L.total > static_cast<size_t>(max_smem))
    L = gqa_smem_layout(elt, q_elt, vsb, D, pl->GH, bs, hc, --S, batch);
  if (L.total > static_cast<size_t>(max_smem))
    return fail(KVC_ERR_UNSUPPORTED, "block_size %d x head_dim %d needs %zu bytes of shared memory (max %d)", bs, D,
                L.total, max_smem);
  pl->hc = hc;
  pl->n_chunks = n_kv_heads / hc;
  pl->units = static_cast<int64_t>(batch) * pl->n_chunks * pl->n_hsub;
  pl->stages = S;
  pl->smem = L.total;
  pl->rec_bytes_per_cta =
      2ull * gqa_max_chunk(pl->GH) * pl->GH * (static_cast<size_t>(D) + 2) * sizeof(float);
  return KVC_OK;
}

// Warp-MMA kernel: bf16/f16 caches (q8 = 0) or one-byte caches with bf16
// queries (q8 = 1: e4m3, 2: int8), head_dim 128, block sizes that are
// multiples of 16 up to 128, and pool rows addressable by a TMA coordinate.
bool mma_supported(kvc_dtype dtype, int head_dim, int block_size, int64_t num_blocks, int n_kv_heads, int qn,
                   int q8 = 0) {
  const int64_t engine = option(KVC_OPT_GQA_ENGINE);
  if (engine == 1) return false;
  // One query per kv head (MHA): the CUDA-core kernel, whose two CTAs per SM
  // read blocks shared by forked sequences close enough in time to hit in L2
  // (measured on the 64-fork batch: 244 us against 348 us), unless forced.
  if (qn == 1 && engine != 3) return false;
  if (dtype != KVC_BF16 && (dtype != KVC_F16 || q8 != 0)) return false;
  if (head_dim != 128 || block_size % 16 != 0 || block_size > 128) return false;
  return num_blocks * n_kv_heads * block_size < (1ll << 31);
}

void mma_dynamic(GqaPlan* pl);

#ifndef KVC_MMA_DYN_SHARE
#define KVC_MMA_DYN_SHARE 256
#endif
constexpr int kDefaultDynShare = KVC_MMA_DYN_SHARE;  // 256: static ranges only

// kMmaCtasPerSm CTAs per SM, each with the deepest ring that fits its share
// of shared memory: a stage holds the K and V pages of hc kv heads of one
// block (each a [hc * block_size x 64] box pair, at most 256 rows per box)
// and the unit's query rows.
kvc_status make_plan_mma(int batch, int n_q_heads, int n_kv_heads, int bs, int q_elt, int max_smem, GqaPlan* pl,
                         int n_tok = 1, bool q8 = false) {
  const int group = n_tok * (n_q_heads / n_kv_heads);
  pl->GH = head_subgroup(group);
  pl->n_hsub = group / pl->GH;
  int hc = 1;
  while (hc * 2 <= mma_max_chunk(pl->GH) && n_kv_heads % (hc * 2) == 0 && hc * 2 * bs <= 256) hc *= 2;
  const int share = std::min(max_smem, (228 * 1024) / kMmaCtasPerSm - 1024);
  // one-byte caches with 16-row blocks: stages of two blocks (per-stage costs
  // bound that loop, and 32-row blocks ran ~5 % faster than 16-row ones)
  const bool pair = q8 && bs == 16;
  int S = 0;
  for (;;) {
    S = 8;
    while (S > 1 && gqa_mma_smem_layout(q_elt, pl->GH, bs, hc, S, batch, q8, pair).total > static_cast<size_t>(share))
      --S;
    if (S >= 3 || hc == 1) break;
    hc /= 2;  // keep at least three stages in flight
  }
  while (S > 1 &&
         gqa_mma_smem_layout(q_elt, pl->GH, bs, hc, S, batch, q8, pair).total > static_cast<size_t>(max_smem))
    --S;
  const GqaMmaSmem L = gqa_mma_smem_layout(q_elt, pl->GH, bs, hc, S, batch, q8, pair);
  pl->pair = pair ? 1 : 0;
  if (L.total > static_cast<size_t>(max_smem))
    return fail(KVC_ERR_UNSUPPORTED, "block_size %d needs %zu bytes of shared memory (max %d)", bs, L.total, max_smem);
  pl->hc = hc;
  pl->n_chunks = n_kv_heads / hc;
  pl->units = static_cast<int64_t>(batch) * pl->n_chunks * pl->n_hsub;
  pl->stages = S;
  pl->smem = L.total;
  pl->rec_bytes_per_cta = 2ull * mma_max_chunk(pl->GH) * pl->GH * (128 + 2) * sizeof(float);
  // an SM holds 228 KB of shared memory (1 KB of it reserved per CTA); the
  // kernel's ~250 registers per thread allow two 128-thread CTAs at most
  pl->ctas_per_sm = std::max(1, std::min<int>(kMmaCtasPerSm, static_cast<int>((228 * 1024) / (L.total + 1024))));
  mma_dynamic(pl);
  return KVC_OK;
}

// Dynamic tail of the warp-MMA work split, from the options: a quarter of
// the positions in chunks of 8 by default; none when the caller forced a
// block count per CTA (unless a chunk size is forced too).
void mma_dynamic(GqaPlan* pl) {
  const int64_t share = option(KVC_OPT_DYNAMIC_SHARE), chunk = option(KVC_OPT_DYNAMIC_CHUNK);
  pl->dyn_share = share == 0 ? kDefaultDynShare : static_cast<int>(share);
  pl->dyn_chunk = chunk == 0 ? 8 : static_cast<int>(chunk);
  if (pl->dyn_share >= 256 || (option(KVC_OPT_BLOCKS_PER_CTA) > 0 && chunk == 0)) pl->dyn_share = pl->dyn_chunk = 0;
}

// Record pairs of the warp-MMA split: one per worker (G static ranges plus
// at most K claimed chunks, K bounded through the table width, the most the
// host knows about the lengths) and, with claimed chunks, one per unit.
int64_t mma_workers(const GqaPlan& pl, int64_t G, int max_blocks) {
  if (pl.dyn_chunk == 0) return G;
  const int64_t n_max = pl.units * max_blocks;
  return G + (n_max * pl.dyn_share / 256 + pl.dyn_chunk - 1) / pl.dyn_chunk + pl.units;
}

// Contributors a unit can have at most: the G static ranges, plus the
// claimed chunks when the split has a dynamic share.
int64_t mma_list_cap(const GqaPlan& pl, int64_t G, int max_blocks) {
  return pl.dyn_chunk == 0 ? G : mma_workers(pl, G, max_blocks) - pl.units;
}

// Bytes ahead of the warp-MMA kernel's records: 256 holding the claim
// counter and the finished-CTA count, then every unit's record list for the
// merge kernel ([count][cap slots] ints).
size_t mma_counter_bytes(const GqaPlan& pl, int64_t cap) {
  return 256 + align_up(static_cast<size_t>(pl.units) * static_cast<size_t>(1 + cap) * 4, 256);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// TMA maps over the K and V pools as [num_blocks * n_kv_heads * block_size
// rows, 128] with the 128-byte swizzle: 16-bit elements in [rows_per_box x 64]
// boxes, or (one_byte) codes in [rows_per_box x 128] boxes.
kvc_status pool_maps(const void* k_cache, const void* v_cache, int64_t num_blocks, int n_kv_heads, int block_size,
                     int rows_per_box, kvc_dtype dtype, CUtensorMap* tk, CUtensorMap* tv, bool one_byte = false) {
  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const CUtensorMapDataType dt = one_byte            ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(num_blocks * n_kv_heads * block_size)};
  const cuuint64_t strides[1] = {one_byte ? 128u : 256u};
  const cuuint32_t box[2] = {one_byte ? 128u : 64u, static_cast<cuuint32_t>(rows_per_box)};
  const cuuint32_t es[2] = {1, 1};
  for (int i = 0; i < 2; ++i) {
    CUresult r = encode(i == 0 ? tk : tv, dt, 2, const_cast<void*>(i == 0 ? k_cache : v_cache), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(KVC_ERR_CUDA, "tensor map for the %s cache: CUresult %d", i ? "V" : "K", static_cast<int>(r));
  }
  return KVC_OK;
}

// Number of CTAs for the balanced split: never more than the blocks allow,
// at most kMaxCtasPerSm per SM unless the caller forced a block count.
int64_t plan_ctas(const DeviceInfo* dev, int occ, int64_t units, int max_blocks) {
  const int64_t upper = units * max_blocks;  // upper bound on cache blocks
  int64_t G;
  const int64_t forced = option(KVC_OPT_BLOCKS_PER_CTA);
  if (forced > 0) {
    G = (upper + forced - 1) / forced;
  } else {
    // at least kMinBlocksPerCta blocks per CTA, but never fewer CTAs than
    // units: small batches are latency-bound, and a CTA per unit finishes
    // them without any split-K merge
    G = static_cast<int64_t>(dev->num_sms) * std::max(1, std::min(occ, kMaxCtasPerSm));
    G = std::min(G, std::max<int64_t>({1, upper / kMinBlocksPerCta, units}));
  }
  const int64_t cap = option(KVC_OPT_MAX_CTAS);
  if (cap > 0) G = std::min(G, cap);
  return std::max<int64_t>(1, std::min<int64_t>(G, 1 << 30));
}

kvc_status check_shapes(int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_blocks) {
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1 || block_size < 1 || max_blocks < 1)
    return fail(KVC_ERR_INVALID_ARG, "batch, heads, head_dim, block_size and max_blocks_per_seq must be >= 1");
  if (n_q_heads % n_kv_heads != 0)
    return fail(KVC_ERR_INVALID_ARG, "n_q_heads (%d) must be a multiple of n_kv_heads (%d)", n_q_heads, n_kv_heads);
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(KVC_ERR_UNSUPPORTED, "head_dim %d (supported: 32, 64, 128, 256)", head_dim);
  if (block_size % 16 != 0 || block_size > 128)
    return fail(KVC_ERR_UNSUPPORTED, "block_size %d (supported: multiples of 16 up to 128)", block_size);
  if (batch > kMaxBatch) return fail(KVC_ERR_UNSUPPORTED, "batch %d > %d", batch, kMaxBatch);
  if (static_cast<int64_t>(max_blocks) * block_size > (1ll << 30))
    return fail(KVC_ERR_UNSUPPORTED, "max_blocks_per_seq x block_size too large");
  if (static_cast<int64_t>(batch) * n_q_heads * head_dim >= (1ll << 31))
    return fail(KVC_ERR_UNSUPPORTED, "batch x n_q_heads x head_dim must be below 2^31");
  return KVC_OK;
}

// The extension kernels serve a sliding window, several new tokens, start
// rows or the LSE output.
bool uses_ext(const GqaParams& p) { return p.window > 0 || p.n_tok > 1 || p.row_div > 0 || p.lse != nullptr; }

// Options of the passes of a shared-prefix decode.
struct DecodeExtra {
  int causal = 1;
  float* lse = nullptr;
  const int32_t* row_start = nullptr;
  int row_div = 0;
  bool int8 = false;  // with k_scale / v_scale: INT8 codes instead of e4m3
};

template <typename T>
kvc_status occupancy(const GqaParams& p, int D, const GqaPlan& pl, int* occ) {
  return uses_ext(p) ? gqa_dispatch<T, true>(p, D, pl.GH, 0, pl.smem, nullptr, 1, occ)
                     : gqa_dispatch<T, false>(p, D, pl.GH, 0, pl.smem, nullptr, 1, occ);
}

// dt -1: FP8 caches, -2: INT8 caches (both with bf16 queries)
kvc_status occupancy_for(int dt, const GqaParams& p, int D, const GqaPlan& pl, int* occ) {
  if (dt == -1) return gqa_dispatch_fp8(p, D, pl.GH, 0, pl.smem, nullptr, 1, occ);
  if (dt == -2) return gqa_dispatch_int8(p, D, pl.GH, 0, pl.smem, nullptr, 1, occ);
  switch (static_cast<kvc_dtype>(dt)) {
    case KVC_F32: return occupancy<float>(p, D, pl, occ);
    case KVC_F16: return occupancy<__half>(p, D, pl, occ);
    case KVC_BF16: return occupancy<__nv_bfloat16>(p, D, pl, occ);
  }
  return fail(KVC_ERR_INVALID_ARG, "dtype");
}

}  // namespace

// Workspace bytes for every engine's plan; with_dynamic = false leaves out the
// records of the warp-MMA kernel's claimed chunks (it then splits statically).
kvc_status decode_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, bool with_dynamic, size_t* bytes) {
  if (bytes == nullptr) return fail(KVC_ERR_INVALID_ARG, "bytes is NULL");
  kvc_status s = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq);
  if (s != KVC_OK) return s;
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != KVC_OK) return s;
  GqaPlan pl;
  if ((s = make_plan(batch, n_q_heads, n_kv_heads, head_dim, block_size, 2, 2, 0, dev->max_smem_optin, &pl)) !=
      KVC_OK)
    return s;
  const int64_t G = plan_ctas(dev, kMaxCtasPerSm, static_cast<int64_t>(batch) * n_kv_heads * pl.n_hsub,
                             max_blocks_per_seq);
  *bytes = align_up(counter_bytes(batch, n_kv_heads, pl) + static_cast<size_t>(G) * pl.rec_bytes_per_cta, 256);
  // the warp-MMA kernel's records (up to 8 query heads per warp, and the
  // claimed chunks' records) may be larger
  GqaPlan pm;
  if (head_dim == 128 && block_size % 16 == 0 && block_size <= 128 &&
      make_plan_mma(batch, n_q_heads, n_kv_heads, block_size, 2, dev->max_smem_optin, &pm) == KVC_OK) {
    const int64_t Gm = plan_ctas(dev, pm.ctas_per_sm, pm.units, max_blocks_per_seq);
    if (!with_dynamic) pm.dyn_share = pm.dyn_chunk = 0;
    const int64_t Wm = mma_workers(pm, Gm, max_blocks_per_seq);
    *bytes = std::max(*bytes, align_up(mma_counter_bytes(pm, mma_list_cap(pm, Gm, max_blocks_per_seq)) +
                                           static_cast<size_t>(Wm) * pm.rec_bytes_per_cta, 256));
  }
  clear_error();
  // the tensor-core kernel for wide groups (any dtype it takes) may need more
  // (n_q_heads here already counts every new token of a multi-token call)
  if (wide_supported(batch, n_q_heads, n_kv_heads, head_dim, block_size, 1, KVC_BF16))
    *bytes = std::max(*bytes, align_up(wide_workspace_bytes(dev, batch, n_q_heads, n_kv_heads, block_size,
                                                            max_blocks_per_seq, 1),
                                       256));
  return KVC_OK;
}

}  // namespace kvc

extern "C" {

kvc_status kvc_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                     int max_blocks_per_seq, size_t* bytes) {
  kvc::clear_error();
  return kvc::decode_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq, true,
                                     bytes);
}

}  // extern "C"

namespace kvc {
namespace {

// Decode over the newest `window` rows of every sequence (window 0: all rows).
// k_scale / v_scale non-NULL: one-byte caches (e4m3, or int8 with
// ex->int8) with bf16 queries (dtype is then the query dtype and must be BF16). n_tok > 1: that many new tokens per
// sequence, q and out [batch, n_tok, n_q_heads, head_dim], causal among them.
kvc_status decode_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int batch, float scale, int n_q_heads,
                       int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, int window, kvc_dtype dtype,
                       void* out, kvc_dtype out_dtype, void* workspace, size_t workspace_bytes, kvc_stream stream,
                       const float* k_scale = nullptr, const float* v_scale = nullptr, int n_tok = 1,
                       const DecodeExtra* ex = nullptr) {
  const DecodeExtra none;
  if (ex == nullptr) ex = &none;
  const bool fp8 = k_scale != nullptr;  // one-byte codes, e4m3 or int8
  if (n_tok < 1 || n_tok > kMaxTokens)
    return fail(KVC_ERR_INVALID_ARG, "n_tokens %d (supported: 1 to %d)", n_tok, kMaxTokens);
  if (n_tok > 1 && (fp8 || window > 0))
    return fail(KVC_ERR_UNSUPPORTED, "several new tokens with a one-byte cache or a sliding window");
  if (!dtype_ok(dtype) || !dtype_ok(out_dtype)) return fail(KVC_ERR_INVALID_ARG, "unknown dtype");
  if (fp8 && dtype != KVC_BF16) return fail(KVC_ERR_UNSUPPORTED, "one-byte cache decode takes bf16 queries");
  if (fp8 && head_dim == 32)
    return fail(KVC_ERR_UNSUPPORTED, "one-byte cache decode head_dim 32 (supported: 64, 128, 256)");
  if (fp8 && (v_scale == nullptr || !aligned16(k_scale) || !aligned16(v_scale)))
    return fail(KVC_ERR_INVALID_ARG, "k_scale and v_scale must be non-NULL and 16-byte aligned");
  kvc_status s = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq);
  if (s != KVC_OK) return s;
  if (static_cast<int64_t>(batch) * n_tok * n_q_heads * head_dim >= (1ll << 31))
    return fail(KVC_ERR_UNSUPPORTED, "batch x n_tokens x n_q_heads x head_dim must be below 2^31");
  if (num_blocks < 1) return fail(KVC_ERR_INVALID_ARG, "num_blocks must be >= 1");
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_tables == nullptr || context_lens == nullptr ||
      out == nullptr)
    return fail(KVC_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(KVC_ERR_INVALID_ARG, "q and caches must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(KVC_ERR_INVALID_ARG, "scale must be finite");
  if (workspace_bytes > 0 && workspace == nullptr) return fail(KVC_ERR_INVALID_ARG, "workspace is NULL");
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(KVC_ERR_INVALID_ARG, "workspace must be 256-byte aligned");

  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != KVC_OK) return s;
  // Engine: the warp-MMA kernel for up to 16 queries per kv head (measured
  // faster than the tcgen05 kernel there: 260 against 270 us on the long
  // split-K batch at 8, 118 against 125 us on the 4-token step at 16), the
  // tcgen05 kernel for 17 to 32 (where the warp-MMA kernel would read the
  // pages once per 16 queries), the CUDA-core kernel for the rest.
  const int qn = n_tok * (n_q_heads / n_kv_heads);
  // one-byte caches: the warp-MMA kernel for single-token full attention
  const int q8 = fp8 ? (ex->int8 ? 2 : 1) : 0;
  const bool use_mma =
      (!fp8 || (window == 0 && n_tok == 1 && ex->row_div == 0 && ex->lse == nullptr)) &&
      mma_supported(dtype, head_dim, block_size, num_blocks, n_kv_heads, qn, q8);
  const bool force_wide = option(KVC_OPT_GQA_ENGINE) == 2;
  if (!fp8 && window == 0 && ex->row_div == 0 && (force_wide || !use_mma || qn > 16) &&
      wide_preferred(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq, n_tok, dtype)) {
    WideArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = out;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.num_blocks = num_blocks;
    a.batch = batch;
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.block_size = block_size;
    a.max_blocks = max_blocks_per_seq;
    a.n_tok = n_tok;
    a.causal = ex->causal;
    a.lse = ex->lse;
    a.dtype = dtype;
    a.out_dtype = out_dtype;
    a.scale = scale;
    a.stream = static_cast<cudaStream_t>(stream);
    return wide_decode(a, dev);
  }
  const int q_elt = static_cast<int>(dtype_size(dtype));
  const int elt = fp8 ? 1 : q_elt;
  GqaPlan pl;
  if (use_mma) {
    if ((s = make_plan_mma(batch, n_q_heads, n_kv_heads, block_size, q_elt, dev->max_smem_optin, &pl, n_tok,
                           q8 != 0)) != KVC_OK)
      return s;
  } else if ((s = make_plan(batch, n_q_heads, n_kv_heads, head_dim, block_size, elt, q_elt, fp8 ? 4 : 0,
                            dev->max_smem_optin, &pl, n_tok)) != KVC_OK) {
    return s;
  }

  GqaParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.err = dev->error_word;
  p.num_blocks = num_blocks;
  p.batch = batch;
  p.n_q_heads = n_q_heads;
  p.n_kv_heads = n_kv_heads;
  p.group = n_q_heads / n_kv_heads;
  p.n_hsub = pl.n_hsub;
  p.hc = pl.hc;
  p.n_chunks = pl.n_chunks;
  p.block_size = block_size;
  p.max_blocks = max_blocks_per_seq;
  p.out_dtype = static_cast<int>(out_dtype);
  p.stages = pl.stages;
  p.window = window;
  p.n_tok = n_tok;
  p.causal = ex->causal;
  p.lse = ex->lse;
  p.row_start = ex->row_start;
  p.row_div = ex->row_div;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.qscale = scale * 1.4426950408889634f;  // log2(e): softmax is evaluated with exp2
  p.wait_polls = static_cast<unsigned int>(option(KVC_OPT_WAIT_POLLS));

  int occ = 1;
  CUtensorMap tk, tv;
  const bool ext = uses_ext(p);
  if (use_mma) {
    if ((s = pool_maps(k_cache, v_cache, num_blocks, n_kv_heads, block_size, pl.hc * block_size, dtype, &tk, &tv,
                       q8 != 0)) != KVC_OK)
      return s;
    s = q8 == 1 ? gqa_mma_dispatch_q8<1>(p, pl.GH, 0, pl.smem, tk, tv, nullptr, 1, &occ)
        : q8 == 2 ? gqa_mma_dispatch_q8<2>(p, pl.GH, 0, pl.smem, tk, tv, nullptr, 1, &occ)
        : dtype == KVC_BF16 ? (ext ? gqa_mma_dispatch<__nv_bfloat16, true>(p, pl.GH, 0, pl.smem, tk, tv, nullptr, 1, &occ)
                                 : gqa_mma_dispatch<__nv_bfloat16, false>(p, pl.GH, 0, pl.smem, tk, tv, nullptr, 1, &occ))
                          : (ext ? gqa_mma_dispatch<__half, true>(p, pl.GH, 0, pl.smem, tk, tv, nullptr, 1, &occ)
                                 : gqa_mma_dispatch<__half, false>(p, pl.GH, 0, pl.smem, tk, tv, nullptr, 1, &occ));
    if (s != KVC_OK) return s;
  } else if ((s = occupancy_for(fp8 ? (ex->int8 ? -2 : -1) : static_cast<int>(dtype), p, head_dim, pl, &occ)) !=
             KVC_OK) {
    return s;
  }
  if (use_mma) occ = std::min(occ, pl.ctas_per_sm);  // never more records than the size query counted
  int64_t G = plan_ctas(dev, occ, pl.units, max_blocks_per_seq);
  const int64_t list_cap = use_mma ? mma_list_cap(pl, G, max_blocks_per_seq) : 0;
  const size_t cbytes = use_mma ? mma_counter_bytes(pl, list_cap) : counter_bytes(batch, n_kv_heads, pl);
  const int64_t rec_fit = workspace_bytes > cbytes
                              ? static_cast<int64_t>((workspace_bytes - cbytes) / pl.rec_bytes_per_cta)
                              : 0;
  int64_t W = G;  // record slots: one pair per worker
  if (use_mma) {
    W = mma_workers(pl, G, max_blocks_per_seq);
    if (W > rec_fit) {  // no room for the claimed chunks' records: static ranges only
      pl.dyn_share = pl.dyn_chunk = 0;
      W = G;
    }
  }
  G = std::min<int64_t>(G, rec_fit);
  W = std::max<int64_t>(W, G);
  const int HS = (use_mma ? mma_max_chunk(pl.GH) : gqa_max_chunk(pl.GH)) * pl.GH;  // query heads per record
  int grid;
  p.pair = use_mma ? pl.pair : 0;  // the stage layout the plan sized
  if (G >= 1) {
    p.unit_mode = 0;
    p.counters = static_cast<unsigned int*>(workspace);
    if (use_mma) {
      p.sched = static_cast<unsigned int*>(workspace);
      p.unit_lists = reinterpret_cast<int*>(static_cast<char*>(workspace) + 256);
      p.list_cap = static_cast<int>(list_cap);
      p.dyn_share = pl.dyn_share;
      p.dyn_chunk = pl.dyn_chunk;
      // automatic split: claimed chunks only when every CTA keeps two rings'
      // worth of static work; a forced chunk size applies at any size
      p.dyn_min_static = option(KVC_OPT_DYNAMIC_CHUNK) > 0 ? 0 : 2 * pl.stages;
    }
    p.rec_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + cbytes);
    p.rec_ml = p.rec_o + static_cast<size_t>(W) * 2 * HS * head_dim;
    p.rec_slots = 2 * W;
    grid = static_cast<int>(G);
  } else {
    p.unit_mode = 1;
    grid = static_cast<int>(pl.units);
  }
  if (pl.units > (1ll << 31) - 1) return fail(KVC_ERR_UNSUPPORTED, "too many (sequence, kv-head chunk) units");
  if (pl.units * max_blocks_per_seq / grid + 1 >= (1ll << 31))
    return fail(KVC_ERR_UNSUPPORTED, "too many cache blocks per CTA");
  if (num_blocks * n_kv_heads >= (1ll << 31))
    return fail(KVC_ERR_UNSUPPORTED, "num_blocks x n_kv_heads must be below 2^31");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (use_mma) {
    s = q8 == 1 ? gqa_mma_dispatch_q8<1>(p, pl.GH, grid, pl.smem, tk, tv, st, 0, nullptr)
        : q8 == 2 ? gqa_mma_dispatch_q8<2>(p, pl.GH, grid, pl.smem, tk, tv, st, 0, nullptr)
        : dtype == KVC_BF16 ? (ext ? gqa_mma_dispatch<__nv_bfloat16, true>(p, pl.GH, grid, pl.smem, tk, tv, st, 0, nullptr)
                                 : gqa_mma_dispatch<__nv_bfloat16, false>(p, pl.GH, grid, pl.smem, tk, tv, st, 0, nullptr))
                          : (ext ? gqa_mma_dispatch<__half, true>(p, pl.GH, grid, pl.smem, tk, tv, st, 0, nullptr)
                                 : gqa_mma_dispatch<__half, false>(p, pl.GH, grid, pl.smem, tk, tv, st, 0, nullptr));
    if (s != KVC_OK) return s;
    return finish_call(st);
  }
  if (fp8) {
    s = ex->int8 ? gqa_dispatch_int8(p, head_dim, pl.GH, grid, pl.smem, st, 0, nullptr)
                 : gqa_dispatch_fp8(p, head_dim, pl.GH, grid, pl.smem, st, 0, nullptr);
    if (s != KVC_OK) return s;
    return finish_call(st);
  }
  const bool win = ext;
  switch (dtype) {
    case KVC_F32:
      s = win ? gqa_dispatch<float, true>(p, head_dim, pl.GH, grid, pl.smem, st, 0, nullptr)
              : gqa_dispatch<float, false>(p, head_dim, pl.GH, grid, pl.smem, st, 0, nullptr);
      break;
    case KVC_F16:
      s = win ? gqa_dispatch<__half, true>(p, head_dim, pl.GH, grid, pl.smem, st, 0, nullptr)
              : gqa_dispatch<__half, false>(p, head_dim, pl.GH, grid, pl.smem, st, 0, nullptr);
      break;
    case KVC_BF16:
      s = win ? gqa_dispatch<__nv_bfloat16, true>(p, head_dim, pl.GH, grid, pl.smem, st, 0, nullptr)
              : gqa_dispatch<__nv_bfloat16, false>(p, head_dim, pl.GH, grid, pl.smem, st, 0, nullptr);
      break;
  }
  if (s != KVC_OK) return s;
  return finish_call(st);
}

}  // namespace
}  // namespace kvc

extern "C" {

kvc_status kvc_decode_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens, int batch, float scale,
                                int n_q_heads, int n_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                size_t workspace_bytes, kvc_stream stream) {
  kvc::clear_error();
  return kvc::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch, scale, n_q_heads,
                          n_kv_heads, head_dim, block_size, num_blocks, 0, dtype, out, out_dtype, workspace,
                          workspace_bytes, stream);
}

kvc_status kvc_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                                    const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int batch, float scale, int n_q_heads,
                                    int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, void* out,
                                    kvc_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                    kvc_stream stream) {
  kvc::clear_error();
  if (k_scale == nullptr || v_scale == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "k_scale / v_scale is NULL");
  return kvc::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch, scale, n_q_heads,
                          n_kv_heads, head_dim, block_size, num_blocks, 0, KVC_BF16, out, out_dtype, workspace,
                          workspace_bytes, stream, k_scale, v_scale);
}

kvc_status kvc_decode_attention_int8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                                     const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int batch, float scale, int n_q_heads,
                                     int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, void* out,
                                     kvc_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                     kvc_stream stream) {
  kvc::clear_error();
  if (k_scale == nullptr || v_scale == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "k_scale / v_scale is NULL");
  kvc::DecodeExtra ex;
  ex.int8 = true;
  return kvc::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch, scale, n_q_heads,
                          n_kv_heads, head_dim, block_size, num_blocks, 0, KVC_BF16, out, out_dtype, workspace,
                          workspace_bytes, stream, k_scale, v_scale, 1, &ex);
}

kvc_status kvc_decode_attention_window(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int batch, float scale, int n_q_heads,
                                       int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, int window,
                                       kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                       size_t workspace_bytes, kvc_stream stream) {
  kvc::clear_error();
  if (window < 1) return kvc::fail(KVC_ERR_INVALID_ARG, "window must be >= 1 (got %d)", window);
  return kvc::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch, scale, n_q_heads,
                          n_kv_heads, head_dim, block_size, num_blocks, window, dtype, out, out_dtype, workspace,
                          workspace_bytes, stream);
}

kvc_status kvc_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int batch, int n_tokens, float scale,
                                      int n_q_heads, int n_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                      kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                      size_t workspace_bytes, kvc_stream stream) {
  kvc::clear_error();
  return kvc::decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch, scale, n_q_heads,
                          n_kv_heads, head_dim, block_size, num_blocks, 0, dtype, out, out_dtype, workspace,
                          workspace_bytes, stream, nullptr, nullptr, n_tokens);
}

}  // extern "C"

// ------------------------------------------------------------------------
// Decode without any caller-provided scratch.
//
// Some callers cannot allocate device memory at the moment they decode: a
// plugin or runtime that only receives pre-allocated input and output buffers
// from its host framework, code that must not touch the allocator on the
// decode path (fixed memory budgets, allocator locks), or a C caller that
// has no CUDA allocator of its own. For them the split-K scratch lives in the
// library itself: one fixed array per device, reserved when the library is
// loaded and held until the process exits.

namespace kvc {
namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch per device, with the context it was
// looked up in: a device reset (or a destroyed and recreated primary
// context) loads the module again, so an address from an older context is
// stale and is looked up again.
struct StaticScratch {
  CUcontext ctx = nullptr;
  void* ptr = nullptr;
};
std::mutex g_static_mutex;
std::vector<StaticScratch> g_static;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

// Looks up (once per device and context, with that device current) the
// device address of the scratch array. Host code must not use the symbol
// itself as a pointer: on the host it names a host-side stand-in.
kvc_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) return fail(KVC_ERR_CUDA, "cuCtxGetCurrent is unavailable");
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (dev >= static_cast<int>(g_static.size())) g_static.resize(dev + 1);
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "cuCtxGetCurrent failed");
  if (ctx == nullptr || g_static[dev].ptr == nullptr || g_static[dev].ctx != ctx) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);  // also makes the device's primary context current
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
    if (get_ctx(&ctx) != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "cuCtxGetCurrent failed");
    g_static[dev].ctx = ctx;
    g_static[dev].ptr = ptr;
  }
  *out = g_static[dev].ptr;
  return KVC_OK;
}

}  // namespace
}  // namespace kvc

extern "C" {

kvc_status kvc_decode_attention_static(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int batch, float scale, int n_q_heads,
                                       int n_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                       kvc_dtype dtype, void* out, kvc_dtype out_dtype, kvc_stream stream) {
  using namespace kvc;
  clear_error();
  if (!dtype_ok(dtype) || !dtype_ok(out_dtype)) return fail(KVC_ERR_INVALID_ARG, "unknown dtype");
  // The least scratch these shapes need: without room for the records of
  // claimed chunks the warp-MMA kernel splits its work statically.
  size_t need = 0;
  kvc_status s =
      decode_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq, false, &need);
  if (s != KVC_OK) return s;
  if (need > kStaticScratchBytes)
    return fail(KVC_ERR_WORKSPACE,
                "these shapes need %zu bytes of decode scratch; the built-in scratch holds %zu bytes "
                "(use kvc_decode_attention with a caller-provided workspace)",
                need, kStaticScratchBytes);
  void* scratch = nullptr;
  if ((s = static_scratch(&scratch)) != KVC_OK) return s;
  // The array keeps the previous call's contents; only the per-unit counters
  // at its start must be zero on entry.
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != KVC_OK) return s;
  GqaPlan pl;
  const int elt_s = static_cast<int>(dtype_size(dtype));
  if ((s = make_plan(batch, n_q_heads, n_kv_heads, head_dim, block_size, elt_s, elt_s, 0, dev->max_smem_optin, &pl)) !=
      KVC_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch, 0, counter_bytes(batch, n_kv_heads, pl) + 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(decode scratch counters)");
  return kvc_decode_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch, scale,
                              n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, dtype, out, out_dtype, scratch,
                              kStaticScratchBytes, stream);
}

}  // extern "C"

// ------------------------------------------------------------------------
// Decode with shared prefixes (sequences forked from one prompt).
//
// Sequences [g * group_size, (g + 1) * group_size) hold the same first
// prefix_lens[g] rows (the shared blocks of a fork). Reading those rows once
// per sequence reads every shared block group_size times; instead the decode
// runs in two passes whose softmax states are merged:
//   1. the shared rows, once per group: the group's group_size x group
//      queries of a kv head are its virtual heads over the group's first
//      table row (the multi-token path without the causal rule),
//   2. each sequence's own rows, [prefix_lens[g], n), through its table,
// each writing its normalised output and log-sum-exp, then
//   out = (o1 2^(lse1 - M) + o2 2^(lse2 - M)) / (2^(lse1 - M) + 2^(lse2 - M)),
// M = max(lse1, lse2), which is the softmax over all n rows.

namespace kvc {
namespace {

__global__ void lse_combine_kernel(const float* __restrict__ o1, const float* __restrict__ lse1,
                                   const float* __restrict__ o2, const float* __restrict__ lse2, void* out,
                                   int out_dtype, int64_t rows, int D) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const float a = lse1[row], b = lse2[row];
  const float m = fmaxf(a, b);
  float wa = 0.f, wb = 0.f;
  if (m != kNegInf) {
    wa = fast_exp2(a - m);  // a = -inf (no row in that pass): 0
    wb = fast_exp2(b - m);
  }
  const float inv = (wa + wb) > 0.f ? 1.0f / (wa + wb) : 0.f;
  for (int d = lane * 4; d < D; d += 128) {
    const float4 x = *reinterpret_cast<const float4*>(o1 + row * D + d);
    const float4 y = *reinterpret_cast<const float4*>(o2 + row * D + d);
    const float v[4] = {(x.x * wa + y.x * wb) * inv, (x.y * wa + y.y * wb) * inv, (x.z * wa + y.z * wb) * inv,
                        (x.w * wa + y.w * wb) * inv};
    store_out_vec<4>(out, row * D + d, v, out_dtype);
  }
}

// Workspace of the shared-prefix decode: each pass has its own decode
// workspace (the first pass's split-K records must never land on the second
// pass's counters, which have to be zero when it starts), then the two
// passes' outputs and log-sum-exps.
struct PrefixLayout {
  size_t inner1, inner2, o1, o2, l1, l2, total;
};

kvc_status prefix_layout(int batch, int group_size, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                         int max_blocks, PrefixLayout* L) {
  if (group_size < 1 || batch % group_size != 0)
    return fail(KVC_ERR_INVALID_ARG, "batch (%d) must be a multiple of group_size (%d >= 1)", batch, group_size);
  if (group_size > kMaxTokens) return fail(KVC_ERR_UNSUPPORTED, "group_size %d > %d", group_size, kMaxTokens);
  if (static_cast<int64_t>(max_blocks) * group_size > (1 << 30))
    return fail(KVC_ERR_UNSUPPORTED, "max_blocks_per_seq x group_size too large");
  size_t w1 = 0, w2 = 0;
  kvc_status s = kvc_decode_workspace_size(batch / group_size, group_size * n_q_heads, n_kv_heads, head_dim,
                                           block_size, group_size * max_blocks, &w1);
  if (s != KVC_OK) return s;
  if ((s = kvc_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks, &w2)) != KVC_OK)
    return s;
  const size_t rows = static_cast<size_t>(batch) * n_q_heads;
  L->inner1 = 0;
  L->inner2 = align_up(w1, 256);
  L->o1 = L->inner2 + align_up(w2, 256);
  L->o2 = L->o1 + align_up(rows * head_dim * 4, 256);
  L->l1 = L->o2 + align_up(rows * head_dim * 4, 256);
  L->l2 = L->l1 + align_up(rows * 4, 256);
  L->total = L->l2 + align_up(rows * 4, 256);
  return KVC_OK;
}

}  // namespace
}  // namespace kvc

extern "C" {

kvc_status kvc_decode_shared_prefix_workspace_size(int batch, int group_size, int n_q_heads, int n_kv_heads,
                                                   int head_dim, int block_size, int max_blocks_per_seq,
                                                   size_t* bytes) {
  using namespace kvc;
  clear_error();
  if (bytes == nullptr) return fail(KVC_ERR_INVALID_ARG, "bytes is NULL");
  kvc_status s = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq);
  if (s != KVC_OK) return s;
  PrefixLayout L;
  if ((s = prefix_layout(batch, group_size, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq, &L)) !=
      KVC_OK)
    return s;
  *bytes = L.total;
  return KVC_OK;
}

kvc_status kvc_decode_attention_shared_prefix(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_tables, int max_blocks_per_seq,
                                              const int32_t* context_lens, int batch, int group_size,
                                              const int32_t* prefix_lens, float scale, int n_q_heads,
                                              int n_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                              kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                              size_t workspace_bytes, kvc_stream stream) {
  using namespace kvc;
  clear_error();
  if (!dtype_ok(dtype) || !dtype_ok(out_dtype)) return fail(KVC_ERR_INVALID_ARG, "unknown dtype");
  if (prefix_lens == nullptr) return fail(KVC_ERR_INVALID_ARG, "prefix_lens is NULL");
  kvc_status s = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq);
  if (s != KVC_OK) return s;
  PrefixLayout L;
  if ((s = prefix_layout(batch, group_size, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq, &L)) !=
      KVC_OK)
    return s;
  if (workspace == nullptr || workspace_bytes < L.total)
    return fail(KVC_ERR_WORKSPACE, "shared-prefix decode needs %zu bytes of workspace (got %zu)", L.total,
                workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(KVC_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  char* ws = static_cast<char*>(workspace);
  float* o1 = reinterpret_cast<float*>(ws + L.o1);
  float* o2 = reinterpret_cast<float*>(ws + L.o2);
  float* l1 = reinterpret_cast<float*>(ws + L.l1);
  float* l2 = reinterpret_cast<float*>(ws + L.l2);
  // pass 1: the shared rows once per group (q, o1 viewed as [groups, group_size, n_q_heads, D])
  DecodeExtra e1;
  e1.causal = 0;
  e1.lse = l1;
  s = decode_impl(q, k_cache, v_cache, block_tables, group_size * max_blocks_per_seq, prefix_lens,
                  batch / group_size, scale, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, 0, dtype, o1,
                  KVC_F32, ws + L.inner1, L.inner2 - L.inner1, stream, nullptr, nullptr, group_size, &e1);
  if (s != KVC_OK) return s;
  // pass 2: each sequence's own rows
  DecodeExtra e2;
  e2.lse = l2;
  e2.row_start = prefix_lens;
  e2.row_div = group_size;
  s = decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch, scale, n_q_heads,
                  n_kv_heads, head_dim, block_size, num_blocks, 0, dtype, o2, KVC_F32, ws + L.inner2, L.o1 - L.inner2,
                  stream, nullptr, nullptr, 1, &e2);
  if (s != KVC_OK) return s;
  const int64_t rows = static_cast<int64_t>(batch) * n_q_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  lse_combine_kernel<<<static_cast<unsigned int>((rows + 7) / 8), 256, 0, st>>>(o1, l1, o2, l2, out,
                                                                               static_cast<int>(out_dtype), rows,
                                                                               head_dim);
  return finish_call(st);
}

}  // extern "C"
