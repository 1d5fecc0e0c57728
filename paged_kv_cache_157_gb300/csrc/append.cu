// Append kernel: scatters the new tokens' K/V rows (or latent rows) to the
// slots their slot mapping names. One thread moves one 16-byte chunk, so a
// warp writes whole 512-byte spans of consecutive chunks of a row.
//
// Source: in-place write at the current position of a preallocated cache
// ("单请求 KV Cache", production practice section), into fixed-size
// PagedAttention blocks ("KV Cache（键值缓存）" section 2.3).
#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {

// Copies rows src[t, h, :] (row_chunks 16-byte chunks each) into
// dst[slot/bs, h, slot%bs, :] for n_src tensors (1 or 2).
__global__ void __launch_bounds__(256) append_kernel(const uint4* __restrict__ src0, const uint4* __restrict__ src1,
                                                     uint4* __restrict__ dst0, uint4* __restrict__ dst1,
                                                     const int64_t* __restrict__ slots, int64_t num_tokens,
                                                     int64_t num_slots, int block_size, int n_heads, int row_chunks,
                                                     unsigned int* err) {
  // a decode launched behind this kernel may start its prologue now; it
  // waits for this grid to finish before it reads any cached row
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t per_token = static_cast<int64_t>(n_heads) * row_chunks;
  const int64_t total = num_tokens * per_token;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_token;
    const int64_t r = i - t * per_token;
    const int h = static_cast<int>(r / row_chunks);
    const int c = static_cast<int>(r - static_cast<int64_t>(h) * row_chunks);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (h == 0 && c == 0) set_flag(err, 0x4u);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t d = ((blk * n_heads + h) * block_size + off) * row_chunks + c;
    dst0[d] = __ldg(src0 + i);
    if (src1 != nullptr) dst1[d] = __ldg(src1 + i);
  }
}

static kvc_status launch_append(bool two, const void* s0, const void* s1, void* d0, void* d1, const int64_t* slots,
                                 int64_t num_tokens, int64_t num_blocks, int block_size, int n_heads, int width,
                                 kvc_dtype dtype, cudaStream_t stream) {
  if (!dtype_ok(dtype)) return fail(KVC_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || n_heads < 1 || width < 1)
    return fail(KVC_ERR_INVALID_ARG, "sizes must be positive (num_tokens >= 0)");
  if (num_tokens == 0) return KVC_OK;
  if (s0 == nullptr || d0 == nullptr || slots == nullptr || (two && (s1 == nullptr || d1 == nullptr)))
    return fail(KVC_ERR_INVALID_ARG, "NULL pointer");
  const size_t row_bytes = static_cast<size_t>(width) * dtype_size(dtype);
  if (row_bytes % 16 != 0) return fail(KVC_ERR_UNSUPPORTED, "row width x element size must be a multiple of 16 bytes");
  if (!aligned16(s0) || !aligned16(d0) || (s1 && !aligned16(s1)) || (d1 && !aligned16(d1)))
    return fail(KVC_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  DeviceInfo* dev = nullptr;
  kvc_status st = current_device(&dev);
  if (st != KVC_OK) return st;
  const int row_chunks = static_cast<int>(row_bytes / 16);
  const int64_t total = num_tokens * n_heads * row_chunks;
  const int64_t want = (total + 255) / 256;
  const int grid = static_cast<int>(want < dev->num_sms * 16LL ? want : dev->num_sms * 16LL);
  append_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(s0), static_cast<const uint4*>(s1),
                                          static_cast<uint4*>(d0), static_cast<uint4*>(d1), slots, num_tokens,
                                          num_blocks * block_size, block_size, n_heads, row_chunks,
                                          dev->error_word);
  return finish_call(stream);
}

// One-byte append: one warp per (token, kv head). K is divided by its
// per-channel scale, V by its row's scale s = max |v| / QMAX (1 for an
// all-zero row), both in fp32 with correctly rounded division, and rounded to
// the code format: e4m3 (QMAX 448; nearest, ties to even, saturating) or, with
// INT8, symmetric int8 (QMAX 127; nearest, ties to even, saturating at +-127).
// Codes go to the pools, s to the V-scale pool [num_blocks, n_heads, block_size].
__device__ __forceinline__ unsigned short encode_pair(float a, float b, bool int8) {
  if (!int8) return float2_to_fp8x2(a, b);
  return static_cast<unsigned short>((float_to_s8(a) & 0xff) | ((float_to_s8(b) & 0xff) << 8));
}

template <typename T, bool INT8>
__global__ void __launch_bounds__(256) append_q8_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                         const int64_t* __restrict__ slots, int64_t num_tokens,
                                                         int n_heads, int D, int block_size, int64_t num_slots,
                                                         const float* __restrict__ k_scale, unsigned char* kc,
                                                         unsigned char* vc, float* vs, unsigned int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t wi = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; wi < num_tokens * n_heads;
       wi += warps) {
    const int64_t t = wi / n_heads;
    const int h = static_cast<int>(wi - t * n_heads);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0) set_flag(err, 0x4u);
      continue;
    }
    const int64_t blk = slot / block_size, off = slot - blk * block_size;
    const T* kr = k + wi * D;
    const T* vr = v + wi * D;
    float vmax = 0.f;
    for (int d = 2 * lane; d < D; d += 64)
      vmax = fmaxf(vmax, fmaxf(fabsf(Elem<T>::to_float(vr[d])), fabsf(Elem<T>::to_float(vr[d + 1]))));
    vmax = warp_max(vmax);
    const float s = vmax > 0.f ? __fdiv_rn(vmax, INT8 ? 127.0f : 448.0f) : 1.0f;
    const int64_t row = ((blk * n_heads + h) * block_size + off) * D;
    for (int d = 2 * lane; d < D; d += 64) {
      const float k0 = __fdiv_rn(Elem<T>::to_float(kr[d]), __ldg(k_scale + h * D + d));
      const float k1 = __fdiv_rn(Elem<T>::to_float(kr[d + 1]), __ldg(k_scale + h * D + d + 1));
      const float v0 = __fdiv_rn(Elem<T>::to_float(vr[d]), s);
      const float v1 = __fdiv_rn(Elem<T>::to_float(vr[d + 1]), s);
      *reinterpret_cast<unsigned short*>(kc + row + d) = encode_pair(k0, k1, INT8);
      *reinterpret_cast<unsigned short*>(vc + row + d) = encode_pair(v0, v1, INT8);
    }
    if (lane == 0) vs[(blk * n_heads + h) * block_size + off] = s;
  }
}

// Copy-on-write: block pairs[2i] -> block pairs[2i + 1] inside one pool,
// block_chunks 16-byte chunks per block. Pairs with a block id outside the
// pool are skipped and flagged; src == dst is a no-op.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* cache, const int64_t* __restrict__ pairs,
                                                          int64_t n_pairs, int64_t num_blocks, int64_t block_chunks,
                                                          unsigned int* err) {
  const int64_t total = n_pairs * block_chunks;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t pr = i / block_chunks;
    const int64_t c = i - pr * block_chunks;
    const int64_t src = __ldg(pairs + 2 * pr), dst = __ldg(pairs + 2 * pr + 1);
    if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) {
      if (c == 0) set_flag(err, 0x1u);
      continue;
    }
    if (src == dst) continue;
    cache[dst * block_chunks + c] = cache[src * block_chunks + c];
  }
}

}  // namespace kvc

namespace kvc {

template <bool INT8>
static void launch_q8(int grid, cudaStream_t s, kvc_dtype dtype, const void* k, const void* v,
                      const int64_t* slot_mapping, int64_t num_tokens, int n_kv_heads, int head_dim, int block_size,
                      int64_t num_slots, const float* k_scale, unsigned char* kc, unsigned char* vc, float* v_scale,
                      unsigned int* err) {
  switch (dtype) {
    case KVC_F32:
      append_q8_kernel<float, INT8><<<grid, 256, 0, s>>>(static_cast<const float*>(k), static_cast<const float*>(v),
                                                          slot_mapping, num_tokens, n_kv_heads, head_dim, block_size,
                                                          num_slots, k_scale, kc, vc, v_scale, err);
      break;
    case KVC_F16:
      append_q8_kernel<__half, INT8><<<grid, 256, 0, s>>>(static_cast<const __half*>(k),
                                                           static_cast<const __half*>(v), slot_mapping, num_tokens,
                                                           n_kv_heads, head_dim, block_size, num_slots, k_scale, kc,
                                                           vc, v_scale, err);
      break;
    case KVC_BF16:
      append_q8_kernel<__nv_bfloat16, INT8><<<grid, 256, 0, s>>>(
          static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), slot_mapping, num_tokens,
          n_kv_heads, head_dim, block_size, num_slots, k_scale, kc, vc, v_scale, err);
      break;
  }
}

// Quantising append to one-byte codes (e4m3 or int8).
kvc_status append_q8(bool int8, const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                     void* k_cache, void* v_cache, float* v_scale, const float* k_scale, int64_t num_blocks,
                     int block_size, int n_kv_heads, int head_dim, kvc_dtype dtype, kvc_stream stream) {
  if (!dtype_ok(dtype)) return fail(KVC_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || n_kv_heads < 1 || head_dim < 2 || head_dim % 2 != 0)
    return fail(KVC_ERR_INVALID_ARG, "sizes must be positive (num_tokens >= 0, head_dim even)");
  if (num_tokens == 0) return KVC_OK;
  if (k == nullptr || v == nullptr || slot_mapping == nullptr || k_cache == nullptr || v_cache == nullptr ||
      v_scale == nullptr || k_scale == nullptr)
    return fail(KVC_ERR_INVALID_ARG, "NULL pointer");
  DeviceInfo* dev = nullptr;
  kvc_status st = current_device(&dev);
  if (st != KVC_OK) return st;
  const int64_t warps = num_tokens * n_kv_heads;
  const int64_t want = (warps + 7) / 8;
  const int grid = static_cast<int>(want < dev->num_sms * 16LL ? want : dev->num_sms * 16LL);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* kc = static_cast<unsigned char*>(k_cache);
  unsigned char* vc = static_cast<unsigned char*>(v_cache);
  const int64_t num_slots = num_blocks * block_size;
  if (int8)
    launch_q8<true>(grid, s, dtype, k, v, slot_mapping, num_tokens, n_kv_heads, head_dim, block_size, num_slots,
                    k_scale, kc, vc, v_scale, dev->error_word);
  else
    launch_q8<false>(grid, s, dtype, k, v, slot_mapping, num_tokens, n_kv_heads, head_dim, block_size, num_slots,
                     k_scale, kc, vc, v_scale, dev->error_word);
  return finish_call(s);
}

}  // namespace kvc

extern "C" {

kvc_status kvc_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                      void* v_cache, int64_t num_blocks, int block_size, int n_kv_heads, int head_dim,
                      kvc_dtype dtype, kvc_stream stream) {
  kvc::clear_error();
  return kvc::launch_append(true, k, v, k_cache, v_cache, slot_mapping, num_tokens, num_blocks, block_size, n_kv_heads,
                            head_dim, dtype, static_cast<cudaStream_t>(stream));
}

kvc_status kvc_append_latent(const void* c, const int64_t* slot_mapping, int64_t num_tokens, void* latent_cache,
                             int64_t num_blocks, int block_size, int d_c, int d_r, kvc_dtype dtype,
                             kvc_stream stream) {
  kvc::clear_error();
  if (d_c < 1 || d_r < 0) return kvc::fail(KVC_ERR_INVALID_ARG, "d_c must be >= 1 and d_r >= 0");
  return kvc::launch_append(false, c, nullptr, latent_cache, nullptr, slot_mapping, num_tokens, num_blocks, block_size,
                            1, d_c + d_r, dtype, static_cast<cudaStream_t>(stream));
}

kvc_status kvc_append_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                          void* v_cache, float* v_scale, const float* k_scale, int64_t num_blocks, int block_size,
                          int n_kv_heads, int head_dim, kvc_dtype dtype, kvc_stream stream) {
  kvc::clear_error();
  return kvc::append_q8(false, k, v, slot_mapping, num_tokens, k_cache, v_cache, v_scale, k_scale, num_blocks,
                        block_size, n_kv_heads, head_dim, dtype, stream);
}

kvc_status kvc_append_int8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                           void* k_cache, void* v_cache, float* v_scale, const float* k_scale, int64_t num_blocks,
                           int block_size, int n_kv_heads, int head_dim, kvc_dtype dtype, kvc_stream stream) {
  kvc::clear_error();
  return kvc::append_q8(true, k, v, slot_mapping, num_tokens, k_cache, v_cache, v_scale, k_scale, num_blocks,
                        block_size, n_kv_heads, head_dim, dtype, stream);
}

kvc_status kvc_copy_blocks(void* cache, int64_t num_blocks, int64_t block_bytes, const int64_t* pairs, int64_t n_pairs,
                           kvc_stream stream) {
  using namespace kvc;
  clear_error();
  if (num_blocks < 1 || block_bytes < 16 || block_bytes % 16 != 0 || n_pairs < 0)
    return fail(KVC_ERR_INVALID_ARG, "num_blocks >= 1, block_bytes a positive multiple of 16, n_pairs >= 0");
  if (n_pairs == 0) return KVC_OK;
  if (cache == nullptr || pairs == nullptr) return fail(KVC_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(cache)) return fail(KVC_ERR_INVALID_ARG, "cache must be 16-byte aligned");
  DeviceInfo* dev = nullptr;
  kvc_status st = current_device(&dev);
  if (st != KVC_OK) return st;
  const int64_t chunks = block_bytes / 16;
  const int64_t want = (n_pairs * chunks + 255) / 256;
  const int grid = static_cast<int>(want < dev->num_sms * 16LL ? want : dev->num_sms * 16LL);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  copy_blocks_kernel<<<grid, 256, 0, s>>>(static_cast<uint4*>(cache), pairs, n_pairs, num_blocks, chunks,
                                          dev->error_word);
  return finish_call(s);
}

}  // extern "C"
