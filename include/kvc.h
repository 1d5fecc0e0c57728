/*
 * kvc.h: C ABI of the paged KV-cache decode library for GB300 (sm_103a).
 *
 * What the library computes (source pages, by title and section):
 *
 *   "KV缓存原理与显存估算" (LLM Systems Wiki), knowledge point 2: one new
 *   query per sequence attends over every cached row after the current K/V
 *   has been appended: z_i = scale * q.k_i, a = softmax(z) with the maximum
 *   subtracted, o = sum_i a_i v_i.
 *   "KV Cache（键值缓存）" (llm-compass) section 2.3 (PagedAttention): the
 *   cache of a sequence is cut into fixed-size blocks; a block table maps
 *   logical block j to a physical block in a shared pool; section 2.2:
 *   MHA / MQA / GQA head sharing and the MLA latent cache (d_c + d_R per
 *   token, W^UK / W^UV absorbed into the query / output side).
 *   "单请求 KV Cache" (mini-vllm step 07): preallocated storage written in
 *   place at the new position, never copied.
 *
 * Conventions for every call:
 *   - All calls return kvc_status; KVC_OK is 0. No C++ exception crosses
 *     this boundary. kvc_last_error_message() gives a one-line reason for
 *     the most recent failure on the calling thread.
 *   - Device pointers are plain CUDA device addresses on the current device.
 *     The caller owns every buffer it passes; the library never allocates,
 *     frees or retains device memory at run time and keeps no pointer after a
 *     call returns. The only device memory of its own is static: a 4-byte
 *     error word and the 16 MiB scratch of kvc_decode_attention_static, per
 *     device that loads the library.
 *   - Compute calls are asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) unless checked mode is on.
 *   - Arguments are validated on the host first (KVC_ERR_INVALID_ARG,
 *     KVC_ERR_UNSUPPORTED). Values that live in device memory (block ids,
 *     context lengths, slots) are checked inside the kernels: an out-of-range
 *     value is never dereferenced, the affected output is left as zeros or
 *     skipped, and a bit is set in the device error word
 *     (kvc_get_error_flags). No kernel traps, asserts or waits without a
 *     bound.
 *
 * Layouts (row-major, element type given by a kvc_dtype):
 *   k_cache, v_cache  [num_blocks, n_kv_heads, block_size, head_dim]
 *   latent_cache      [num_blocks, block_size, d_c + d_r]
 *   block_tables      int32 [batch, max_blocks_per_seq]; entry j of row i is
 *                     the physical block holding logical positions
 *                     j*block_size .. j*block_size+block_size-1 of sequence i
 *   context_lens      int32 [batch]; rows attended by sequence i, including the
 *                     token appended this step (must be >= 1)
 *   slot_mapping      int64 [num_tokens]; slot = physical_block*block_size +
 *                     position%block_size; a negative slot means "skip"
 *   q, out            [batch, n_q_heads, head_dim]; query head h reads kv
 *                     head h / (n_q_heads / n_kv_heads)
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_ABI_VERSION 1

typedef enum kvc_status {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = 1,  /* a host-checkable argument is wrong */
  KVC_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
  KVC_ERR_NO_BLOCKS = 3,    /* block pool exhausted; nothing was allocated */
  KVC_ERR_CUDA = 4,         /* a CUDA runtime call failed */
  KVC_ERR_OUT_OF_RANGE = 5, /* checked mode: a kernel saw a bad device value */
  KVC_ERR_WORKSPACE = 6     /* workspace smaller than the size query asked for */
} kvc_status;

typedef enum kvc_dtype { KVC_F32 = 0, KVC_F16 = 1, KVC_BF16 = 2 } kvc_dtype;

/* Bits of the device error word. */
#define KVC_FLAG_BAD_BLOCK 0x1u   /* block table entry outside [0, num_blocks) */
#define KVC_FLAG_BAD_LEN 0x2u     /* context_len < 1 (multi-token: < n_tokens) or > max_blocks_per_seq*block_size */
#define KVC_FLAG_BAD_SLOT 0x4u    /* slot >= num_blocks*block_size */
#define KVC_FLAG_TIMEOUT 0x8u     /* a bounded wait on an async copy gave up */
#define KVC_FLAG_WORKSPACE 0x10u  /* decode workspace counters were not zero at entry */

typedef void* kvc_stream; /* cudaStream_t */

/* ---------------------------------------------------------------- runtime */

int kvc_abi_version(void);
const char* kvc_status_string(kvc_status s);
/* Reason for the last non-OK status returned on this thread ("" if none).
 * The string stays valid until the next call on the same thread. */
const char* kvc_last_error_message(void);

typedef enum kvc_option {
  /* 0 (default): calls are asynchronous. 1: every compute call synchronises
   * its stream, reads the device error word of the current device, clears
   * it, and returns KVC_ERR_OUT_OF_RANGE if any bit was set. */
  KVC_OPT_CHECKED = 0,
  /* Decode work split: 0 (default) = automatic. N > 0 = every CTA of the
   * decode kernels takes about N cache blocks (used by tests to force many
   * split-K partials). Process-wide. */
  KVC_OPT_BLOCKS_PER_CTA = 1,
  /* Upper bound on decode CTAs (0 = automatic, SM count x resident CTAs). */
  KVC_OPT_MAX_CTAS = 2,
  /* GQA decode engine. Three kernels compute the same decode:
   *  - the tcgen05 tensor-core kernel: bf16/f16 caches, head_dim 128, block
   *    sizes 16/32/64/128, no window, kv heads with 8 to 32 queries (qn =
   *    n_tokens x n_q_heads / n_kv_heads);
   *  - the warp-MMA kernel: bf16/f16 caches, and the one-byte caches of
   *    kvc_decode_attention_fp8 / _int8, head_dim 128, block sizes that are
   *    multiples of 16 up to 128 (16-bit caches: every feature, windows,
   *    several new tokens, shared prefixes);
   *  - the CUDA-core kernel: every dtype, head size and feature.
   * 0 (default) = automatic: the warp-MMA kernel where it applies and qn is
   * 2 to 16; else the tensor-core kernel where it applies and the cache it
   * may read (batch x n_kv_heads x max_blocks_per_seq x block_size rows of K
   * and V) is at least 512 MiB / qn; else the warp-MMA kernel where it
   * applies (qn > 32); else the CUDA-core kernel; 1 = always the CUDA-core
   * kernel;
   * 2 = the tensor-core kernel wherever it applies, at any size (else as 0);
   * 3 = the warp-MMA kernel wherever it applies, else the CUDA-core kernel. */
  KVC_OPT_GQA_ENGINE = 3,
  /* Warp-MMA kernel work split. Each CTA streams a static range of the cache
   * blocks; optionally the last share of every (sequence, kv-head chunk)
   * unit's blocks is instead cut into chunks that CTAs claim as they finish,
   * so faster SMs take more of it. Every segment that covers part of a unit
   * leaves a partial record, which a merge kernel launched behind the decode
   * combines, so small chunks trade balance for records. DYNAMIC_SHARE: the
   * claimed part in 1/256 of each unit's blocks (0 = automatic, currently
   * none; 1..255 as given; 256 = none). DYNAMIC_CHUNK: blocks (of one
   * kv-head chunk) per claimed chunk (0 = automatic, 8; N >= 1 as given, and
   * then used at any size). Process-wide. */
  KVC_OPT_DYNAMIC_SHARE = 4,
  KVC_OPT_DYNAMIC_CHUNK = 5,
  /* Test hook for the failure path of the GQA decode kernels (CUDA-core and
   * warp-MMA). 0 (default): a wait for copied data gives up after about one
   * second. N > 0: it gives up after N polls, normally long before the data
   * lands, so the kernel takes its abort path on a healthy GPU: it sets
   * KVC_FLAG_TIMEOUT, stops its warps, waits (with the normal bound) for its
   * own copies still in flight, and returns with the output undefined. After
   * any call that set KVC_FLAG_TIMEOUT the decode workspace must be
   * zero-filled again before its next use. Process-wide. */
  KVC_OPT_WAIT_POLLS = 6
} kvc_option;
kvc_status kvc_set_option(kvc_option opt, int64_t value);
kvc_status kvc_get_option(kvc_option opt, int64_t* value);
/* Checked mode on (enabled != 0) or off: the same as
 * kvc_set_option(KVC_OPT_CHECKED, enabled != 0). The checks follow the input
 * validation of the cached_attention listing of "KV缓存原理与显存估算"
 * (knowledge point 2: non-empty input, in-range data) for the values that live
 * in device memory. */
kvc_status kvc_set_checked(int enabled);

/* Synchronises `stream`, then returns (in *flags) and clears the error word
 * of the current device. */
kvc_status kvc_get_error_flags(kvc_stream stream, uint32_t* flags);

/* ----------------------------------------------------------------- append */

/* Writes token t's rows k[t, :, :] and v[t, :, :] (both [num_tokens,
 * n_kv_heads, head_dim], dtype `dtype`) into k_cache / v_cache at
 * slot_mapping[t], for every kv head: cache[slot/bs, h, slot%bs, :] = k[t,h,:].
 * Bit-exact copy. Negative slots are skipped; slots >= num_blocks*block_size
 * are skipped and set KVC_FLAG_BAD_SLOT. Two tokens mapped to the same slot
 * race (the result is one of them). num_tokens == 0 is a no-op.
 * Requires head_dim*element_size to be a multiple of 16 bytes and all
 * pointers 16-byte aligned.
 * Source: the in-place write at the current position ("单请求 KV Cache",
 * production practice section) into PagedAttention blocks (llm-compass 2.3). */
kvc_status kvc_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                      void* k_cache, void* v_cache, int64_t num_blocks, int block_size, int n_kv_heads,
                      int head_dim, kvc_dtype dtype, kvc_stream stream);

/* MLA form: writes row c[t, :] (width d_c + d_r) into
 * latent_cache[slot/bs, slot%bs, :]. Same rules as kvc_append.
 * Source: llm-compass section 2.2 (one shared latent plus decoupled RoPE part
 * cached per token). */
kvc_status kvc_append_latent(const void* c, const int64_t* slot_mapping, int64_t num_tokens,
                             void* latent_cache, int64_t num_blocks, int block_size, int d_c, int d_r,
                             kvc_dtype dtype, kvc_stream stream);

/* FP8 KV cache append: quantises token t's K/V rows (k, v: [num_tokens,
 * n_kv_heads, head_dim] in `dtype`, F32/F16/BF16) and writes them at
 * slot_mapping[t] (negative: skipped; >= num_blocks*block_size: skipped and
 * KVC_FLAG_BAD_SLOT) into k_cache / v_cache: uint8 e4m3 codes
 * [num_blocks, n_kv_heads, block_size, head_dim]. K code = e4m3(k /
 * k_scale[h, d]) with the caller's per-channel scales k_scale [n_kv_heads,
 * head_dim] fp32; V code = e4m3(v / s) with one scale per (token, kv head)
 * s = max_d |v| / 448 (1 for an all-zero row), written to v_scale
 * [num_blocks, n_kv_heads, block_size] fp32. Divisions are fp32, correctly
 * rounded; e4m3 rounding is to nearest, ties to even, saturating at +-448.
 * head_dim must be even. Source: "KV-Cache——为什么AI回复越来越快" section 08
 * (KV-Cache quantisation to FP8: per-token scales for V, per-channel scales
 * for K). */
kvc_status kvc_append_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                          void* k_cache, void* v_cache, float* v_scale, const float* k_scale, int64_t num_blocks,
                          int block_size, int n_kv_heads, int head_dim, kvc_dtype dtype, kvc_stream stream);

/* INT8 KV cache append: as kvc_append_fp8 with int8 codes (int8 pools
 * [num_blocks, n_kv_heads, block_size, head_dim]): K code = q(k / k_scale[h, d]),
 * V code = q(v / s) with s = max_d |v| / 127 (1 for an all-zero row) written
 * to v_scale [num_blocks, n_kv_heads, block_size] fp32; q rounds an fp32 value
 * to the nearest integer, ties to even, and saturates at +-127 (symmetric:
 * -128 is never written). Divisions are fp32, correctly rounded. Same slot,
 * flag and error rules as kvc_append_fp8. Source: "KV-Cache——为什么AI回复越来越快"
 * section 08 (KV-Cache quantisation, INT8 named beside FP8). */
kvc_status kvc_append_int8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                           void* k_cache, void* v_cache, float* v_scale, const float* k_scale, int64_t num_blocks,
                           int block_size, int n_kv_heads, int head_dim, kvc_dtype dtype, kvc_stream stream);

/* Copy-on-write block copy inside one pool: for i < n_pairs, block
 * pairs[2i + 1] becomes a byte copy of block pairs[2i]. cache: device pool of
 * num_blocks blocks of block_bytes bytes each (for a K or V pool,
 * n_kv_heads * block_size * head_dim * element size; for a latent pool,
 * block_size * (d_c + d_r) * element size), 16-byte aligned; block_bytes a
 * multiple of 16. pairs: int64 [n_pairs, 2] in device memory. Destination
 * blocks must be distinct and must not be sources in the same call (copies
 * run concurrently). Pairs naming a block outside the pool are skipped and set
 * KVC_FLAG_BAD_BLOCK. Asynchronous on `stream`.
 * Source: llm-compass 2.3 (copy-on-write of shared PagedAttention blocks). */
kvc_status kvc_copy_blocks(void* cache, int64_t num_blocks, int64_t block_bytes, const int64_t* pairs,
                           int64_t n_pairs, kvc_stream stream);

/* ----------------------------------------------------------------- decode */

/* Bytes of scratch that kvc_decode_attention needs for these shapes on the
 * current device (split-K partial results). 0 is a valid answer. The size
 * depends on the device's SM count and on KVC_OPT_MAX_CTAS. Errors: the
 * shape checks of kvc_decode_attention (KVC_ERR_INVALID_ARG /
 * KVC_ERR_UNSUPPORTED). The split itself is this library's; the pages define
 * only the result it must equal ("KV缓存原理与显存估算", knowledge point 2). */
kvc_status kvc_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                     int max_blocks_per_seq, size_t* bytes);

/* Single-step paged decode attention (MHA, GQA, MQA).
 *   out[i, h, :] = sum_t a_t v_t,  a = softmax_t(scale * q[i,h,:] . k_t)
 * over t = 0 .. context_lens[i]-1, rows read through block_tables[i] from
 * kv head h / (n_q_heads/n_kv_heads). Accumulation is fp32; `out` is written
 * in out_dtype (F32, F16 or BF16).
 * Supported: head_dim in {32, 64, 128, 256}; block_size a multiple of 16 up
 * to 128; n_q_heads % n_kv_heads == 0; batch <= 4096.
 * workspace: device scratch of at least kvc_decode_workspace_size() bytes,
 * 256-byte aligned. It must be zero-filled once before its first use (for
 * example cudaMemset after allocation); every complete call leaves it zeroed
 * again (it holds split-K partial results and one counter per (sequence,
 * head group) that the kernel resets). If a call finds a counter that was not
 * zero it sets KVC_FLAG_WORKSPACE and the affected outputs are not written:
 * zero the workspace again. May be NULL with workspace_bytes 0 (then every
 * (sequence, head group) is handled by one CTA, which balances less well on
 * long contexts). Calls that may run concurrently must not share a workspace.
 * Sources: knowledge point 2 of "KV缓存原理与显存估算"; head grouping from
 * "KV-Cache——为什么AI回复越来越快" section 03 and llm-compass 2.2. */
kvc_status kvc_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                                int batch, float scale, int n_q_heads, int n_kv_heads, int head_dim,
                                int block_size, int64_t num_blocks, kvc_dtype dtype, void* out,
                                kvc_dtype out_dtype, void* workspace, size_t workspace_bytes, kvc_stream stream);

/* Sliding-window decode: as kvc_decode_attention, but sequence i attends only
 * its newest `window` rows, t = max(0, n_i - window) .. n_i - 1 with
 * n_i = context_lens[i] (the token appended this step is the newest row).
 * window >= n_i is full attention; window < 1 is KVC_ERR_INVALID_ARG. Table
 * entries before the block that holds row n_i - window are never read, so a
 * caller may drop (free) those blocks. Same arguments, workspace and error
 * rules as kvc_decode_attention (the same workspace size query applies).
 * Source: "KV-Cache——为什么AI回复越来越快" section 08 (Window Attention /
 * Sliding Window: only the most recent W tokens' K/V are kept) and the
 * closing section of "KV缓存原理与显存估算" (the dropped state is outside the
 * model's visible range). */
kvc_status kvc_decode_attention_window(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int batch, float scale, int n_q_heads,
                                       int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, int window,
                                       kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                       size_t workspace_bytes, kvc_stream stream);

/* Several new query tokens per sequence (chunked prefill of a prompt
 * continuation, or verification of n_tokens speculated tokens), attending
 * the paged cache causally in one pass over each sequence's pages:
 *   out[i, t, h, :] = softmax-weighted sum over rows 0 .. n_i - n_tokens + t
 * with n_i = context_lens[i], which counts every cached row including the
 * n_tokens new ones (append them first, e.g. with kvc_append). Token t sits
 * at position n_i - n_tokens + t and sees itself and every earlier row.
 * q: [batch, n_tokens, n_q_heads, head_dim] contiguous, dtype; out: the same
 * shape in out_dtype. 1 <= n_tokens <= 256 (n_tokens 1 is
 * kvc_decode_attention); a context with fewer than n_tokens rows is invalid
 * (KVC_FLAG_BAD_LEN, zero outputs). Every page is read once for all
 * n_tokens x (n_q_heads / n_kv_heads) queries of its kv head.
 * workspace: at least kvc_decode_workspace_size(batch, n_tokens * n_q_heads,
 * n_kv_heads, head_dim, block_size, max_blocks_per_seq) bytes; otherwise the
 * arguments, workspace and error rules of kvc_decode_attention. F32, F16 and
 * BF16 caches; not combined with a window or an FP8 cache.
 * Source: the prefill/decode mask rule of "单请求 KV Cache" (query row i of a
 * chunk sees columns up to past_len + i) applied through the block table of
 * "KV缓存原理与显存估算" knowledge point 2. */
kvc_status kvc_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int batch, int n_tokens, float scale,
                                      int n_q_heads, int n_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                      kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                      size_t workspace_bytes, kvc_stream stream);

/* Scratch bytes kvc_decode_attention_shared_prefix needs for these shapes
 * (256-byte aligned, zero-filled once before first use; complete calls leave
 * its counters zeroed again). Same shape errors as the call it sizes. */
kvc_status kvc_decode_shared_prefix_workspace_size(int batch, int group_size, int n_q_heads, int n_kv_heads,
                                                   int head_dim, int block_size, int max_blocks_per_seq,
                                                   size_t* bytes);

/* Decode for sequences that share a prefix (forks of one prompt: parallel
 * sampling, beam search): the same result as kvc_decode_attention, but each
 * shared block is read once per group instead of once per sequence.
 * Sequences [g * group_size, (g + 1) * group_size) form group g; their first
 * prefix_lens[g] rows (device int32 [batch / group_size]) must hold the same
 * keys and values in every member (shared blocks, or copies of them), with
 * 1 <= prefix_lens[g] <= each member's context length (KVC_FLAG_BAD_LEN
 * otherwise). Runs three kernels on `stream`: the shared rows once per group
 * (the group's queries of a kv head as virtual heads over the first member's
 * table row), each sequence's rows from prefix_lens[g] on, and a merge of the
 * two softmax states by their log-sum-exp. workspace: at least
 * kvc_decode_shared_prefix_workspace_size() bytes (KVC_ERR_WORKSPACE if
 * smaller or NULL). Other arguments, dtypes and errors as
 * kvc_decode_attention. 1 <= group_size <= 256.
 * Source: the shared physical blocks of "KV缓存原理与显存估算" (closing
 * section: logical blocks of several sequences pointing at one physical block)
 * and "KV Cache（键值缓存）" section 2.3 (sharing and copy-on-write of forks);
 * the result is the decode of knowledge point 2 of the former. */
kvc_status kvc_decode_attention_shared_prefix(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_tables, int max_blocks_per_seq,
                                              const int32_t* context_lens, int batch, int group_size,
                                              const int32_t* prefix_lens, float scale, int n_q_heads,
                                              int n_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                              kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                              size_t workspace_bytes, kvc_stream stream);

/* FP8 KV cache decode: as kvc_decode_attention over the caches written by
 * kvc_append_fp8, attending k = e4m3value(code) * k_scale[h, d] and
 * v = e4m3value(code) * v_scale[row] (the scales fold into the query and into
 * the softmax weights, so the kernel reads one byte per cached element; with
 * head_dim 128 and 2 to 16 queries per kv head the warp-MMA kernel runs the
 * products on f16 MMAs, the codes converted exactly, the scaled query and
 * the weights as f16 hi + lo parts). q is bf16 [batch, n_q_heads, head_dim];
 * head_dim 64, 128 or 256; k_scale and v_scale 16-byte aligned. Same
 * tables, lengths, workspace (size query: kvc_decode_workspace_size) and
 * error rules as kvc_decode_attention.
 * Source: "KV-Cache——为什么AI回复越来越快" section 08 (FP8 KV cache). */
kvc_status kvc_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                                    const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int batch, float scale, int n_q_heads,
                                    int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, void* out,
                                    kvc_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                    kvc_stream stream);

/* INT8 KV cache decode: as kvc_decode_attention_fp8 over the caches written
 * by kvc_append_int8, attending k = code * k_scale[h, d] and
 * v = code * v_scale[row]. q is bf16 [batch, n_q_heads, head_dim]; head_dim
 * 64, 128 or 256; k_scale and v_scale 16-byte aligned. Same tables, lengths,
 * workspace and error rules as kvc_decode_attention. Source:
 * "KV-Cache——为什么AI回复越来越快" section 08 (KV-Cache quantisation). */
kvc_status kvc_decode_attention_int8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                                     const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int batch, float scale, int n_q_heads,
                                     int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, void* out,
                                     kvc_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                     kvc_stream stream);

/* kvc_decode_attention for callers that cannot allocate device memory.
 *
 * There is no counterpart of this call on the source pages: it exists for
 * callers that must not or cannot allocate on the decode path, such as a
 * plugin that only receives its input and output buffers from a host
 * framework, code running under a fixed device-memory budget or an allocator
 * lock, or plain C code with no allocator of its own. It computes exactly what
 * kvc_decode_attention computes (same arguments, minus the workspace) and
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *
 * Its split-K scratch is one fixed 16 MiB array inside the library, reserved
 * on every device that loads the library and held until the process exits.
 * Shapes whose kvc_decode_workspace_size exceeds 16 MiB are refused with
 * KVC_ERR_WORKSPACE and a message giving both sizes (use kvc_decode_attention
 * with your own workspace for those).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture. The address is looked up again when the
 * device's current context is a new one (after cudaDeviceReset, say). Every call then clears the counters at the start
 * of the array with an asynchronous memset on `stream`; the array keeps the
 * rest of the last call's contents. All calls share the one array, so calls
 * whose kernels may overlap on the GPU (different streams, or several host
 * threads) race: serialise them, or use kvc_decode_attention with one
 * workspace per stream. */
kvc_status kvc_decode_attention_static(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int batch, float scale, int n_q_heads,
                                       int n_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                       kvc_dtype dtype, void* out, kvc_dtype out_dtype, kvc_stream stream);

/* Scratch bytes for kvc_decode_attention_mla on the current device (split-K
 * records; 0 is a valid answer). Same shape errors as that call. */
kvc_status kvc_decode_mla_workspace_size(int batch, int n_q_heads, int d_c, int d_r, int block_size,
                                         int max_blocks_per_seq, size_t* bytes);

/* MLA absorbed decode on tensor cores (tcgen05):
 *   out[i, h, :] = sum_t a_t c_t[:d_c],  a = softmax_t(scale * q_absorbed[i,h,:] . c_t)
 * where c_t is the cached row of width d_c + d_r (keys use the whole row,
 * values its first d_c elements). The caller applies W^UV and the output
 * projection to `out`. dtype must be BF16; out_dtype F32 or BF16.
 * Supported: d_c = 512, d_r = 64, n_q_heads = 128, block_size a multiple of
 * 16 up to 256, batch up to 128. Source: llm-compass section 2.2. */
kvc_status kvc_decode_attention_mla(const void* q_absorbed, const void* latent_cache, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens, int batch, float scale,
                                    int n_q_heads, int d_c, int d_r, int block_size, int64_t num_blocks,
                                    kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                    size_t workspace_bytes, kvc_stream stream);

/* ------------------------------------------------------------- block pool */

/* Host-side refcounted block pool ("KV Cache（键值缓存）" 2.3: blocks on
 * demand, shared blocks counted by reference; "KV缓存原理与显存估算",
 * closing section: a block is reusable when its count reaches zero).
 * Policy: a new block is the lowest-numbered free block; sequence ids are
 * 0, 1, 2, ... and never reused. Not thread-safe: one thread per pool. */
typedef struct kvc_pool kvc_pool;

typedef struct kvc_pool_stats {
  int64_t num_blocks;
  int64_t free_blocks;
  int64_t unique_blocks;   /* blocks with refcount > 0 */
  int64_t table_entries;   /* sum over live sequences of their table lengths */
  int64_t useful_tokens;   /* sum over live sequences of their lengths */
  int64_t live_seqs;
  int32_t block_size;
} kvc_pool_stats;

/* A pool of num_blocks blocks of block_size token rows, all free; *pool
 * receives a handle the caller releases with kvc_pool_destroy. Source:
 * "KV Cache（键值缓存）" 2.3 (a shared pool of fixed-size physical blocks). */
kvc_status kvc_pool_create(int64_t num_blocks, int block_size, kvc_pool** pool);
void kvc_pool_destroy(kvc_pool* pool);
/* A new empty sequence (length 0, no blocks); *seq receives its id. Source:
 * "KV Cache（键值缓存）" 2.3 (each sequence owns a block table, empty until its
 * first token). */
kvc_status kvc_seq_add(kvc_pool* pool, int64_t* seq);
/* New sequence sharing all of parent's blocks (each gains one reference);
 * KVC_ERR_INVALID_ARG for an unknown parent. Source: "KV Cache（键值缓存）"
 * 2.3 (blocks shared between sequences by reference count). */
kvc_status kvc_seq_fork(kvc_pool* pool, int64_t parent, int64_t* child);
/* Extends `seq` by n_new tokens and writes their slots to slots_out[n_new].
 * Allocates a block at every block boundary. KVC_ERR_NO_BLOCKS if the pool
 * cannot supply them (nothing allocated, length unchanged).
 * KVC_ERR_UNSUPPORTED if the last block is partly filled and shared
 * (would need copy-on-write). slots_out is host memory owned by the caller.
 * Source: "KV Cache（键值缓存）" 2.3 (fixed-size blocks allocated on demand). */
kvc_status kvc_seq_reserve(kvc_pool* pool, int64_t seq, int64_t n_new, int64_t* slots_out);
/* kvc_seq_reserve for n distinct sequences in one call (a decode step's host
 * work): each of seqs[0..n) gains n_new tokens, in that order, and
 * slots_out[i * n_new + t] receives sequence i's slot for its token t (host
 * memory, caller-owned, n * n_new entries). All or nothing: an unknown or
 * repeated id (KVC_ERR_INVALID_ARG), a sequence whose partly filled last
 * block is shared (KVC_ERR_UNSUPPORTED) or too few free blocks for the whole
 * batch (KVC_ERR_NO_BLOCKS) changes nothing. The result equals n calls of
 * kvc_seq_reserve in order. Source: "KV Cache（键值缓存）" 2.3. */
kvc_status kvc_seq_reserve_batch(kvc_pool* pool, const int64_t* seqs, int n, int64_t n_new, int64_t* slots_out);
/* kvc_seq_reserve with copy-on-write: if the sequence's last block is partly
 * filled and held by other sequences too, the sequence first gets a fresh
 * block (the lowest free id) in its place, drops its reference to the shared
 * block, and copy_pair (2 entries, host memory) receives (shared, fresh):
 * the caller must run kvc_copy_blocks on every pool (K and V, or the latent
 * pool) with that pair before it writes the new rows. copy_pair is (-1, -1)
 * when nothing has to be copied. KVC_ERR_NO_BLOCKS if the fresh block and
 * the new tail blocks are not all free (then nothing changes).
 * Source: llm-compass 2.3 (blocks shared by reference count are copied
 * before a holder writes into them: parallel sampling, beam search). */
kvc_status kvc_seq_reserve_cow(kvc_pool* pool, int64_t seq, int64_t n_new, int64_t* slots_out, int64_t* copy_pair);
/* Drops the sequence; each of its blocks loses one reference and returns to
 * the free list at zero. KVC_ERR_INVALID_ARG for an unknown sequence.
 * Source: "KV Cache（键值缓存）" 2.3. */
kvc_status kvc_seq_free(kvc_pool* pool, int64_t seq);
/* Tokens held by `seq` (the useful rows of its blocks). Source:
 * "KV缓存原理与显存估算" knowledge point 1 (useful bytes count each sequence's
 * own length, not the block-rounded size). */
kvc_status kvc_seq_length(kvc_pool* pool, int64_t seq, int64_t* length);
/* Number of sequences holding `block` (0: free). Source: "KV Cache（键值缓存）"
 * 2.3 (shared blocks are counted by reference). */
kvc_status kvc_block_refcount(kvc_pool* pool, int64_t block, int32_t* refcount);
/* Writes table rows (int32 [n, max_blocks], unused entries 0) and lengths
 * (int32 [n]) for the given sequences, into caller-owned host memory.
 * KVC_ERR_INVALID_ARG for an unknown sequence or one with more blocks than
 * max_blocks. Source: "KV Cache（键值缓存）" 2.3 (the per-sequence block table
 * from logical to physical blocks). */
kvc_status kvc_build_block_tables(kvc_pool* pool, const int64_t* seqs, int n, int32_t* table_out,
                                  int max_blocks, int32_t* lens_out);
/* Pool counters: free and unique (referenced) blocks, table entries, useful
 * tokens. (Not named kvc_pool_stats: C keeps functions and typedefs in one
 * name space, and that name is the struct's.) Source: the closing section of "KV缓存原理与显存估算" (memory counted
 * over unique physical blocks, not table entries) and knowledge point 1
 * (useful tokens against allocated slots). */
kvc_status kvc_pool_get_stats(kvc_pool* pool, kvc_pool_stats* stats);

/* Host helper: slots of (row, position) pairs for an existing host-side
 * block table (int32 [rows, max_blocks]): slot = table[row][pos / block_size]
 * * block_size + pos % block_size. All pointers are caller-owned host memory.
 * Out-of-table positions give KVC_ERR_INVALID_ARG. Source: "KV Cache（键值缓存）"
 * 2.3 (block table lookup); the slot encoding is this library's. */
kvc_status kvc_slots_from_tables(const int32_t* block_tables, int rows, int max_blocks, int block_size,
                                 const int32_t* row_index, const int64_t* positions, int64_t n,
                                 int64_t* slots_out);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
