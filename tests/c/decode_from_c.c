/* A plain C (C11) client of the whole path on the GPU: the host pool hands
 * out slots and block tables, kvc_append writes a prompt's K/V rows into
 * zeroed bf16 pools, kvc_decode_attention attends over them. Buffers are
 * the caller's (cudaMalloc). Inputs come from a fixed linear congruential
 * generator; inputs and results are written as raw little-endian arrays to
 * the directory argv[1] for the oracle comparison in Python.
 *
 * Shapes: 3 sequences of 1, 17 and 40 tokens, 8 query / 2 kv heads,
 * head_dim 128, block 16, 16 physical blocks, tables 4 wide, bf16, fp32 out. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvc.h"

enum { B = 3, HQ = 8, HKV = 2, D = 128, BS = 16, NB = 16, MAXB = 4, T = 1 + 17 + 40 };

#define CHECK(x)                                                              \
  do {                                                                        \
    kvc_status s_ = (x);                                                      \
    if (s_ != KVC_OK) {                                                       \
      fprintf(stderr, "%s:%d: %s -> %d (%s)\n", __FILE__, __LINE__, #x, s_,   \
              kvc_last_error_message());                                      \
      return 1;                                                               \
    }                                                                         \
  } while (0)

#define CUDA(x)                                                               \
  do {                                                                        \
    cudaError_t e_ = (x);                                                     \
    if (e_ != cudaSuccess) {                                                  \
      fprintf(stderr, "%s:%d: %s -> %s\n", __FILE__, __LINE__, #x,            \
              cudaGetErrorString(e_));                                        \
      return 1;                                                               \
    }                                                                         \
  } while (0)

static uint64_t g_state = 0x9E3779B97F4A7C15ull;

/* uniform in [-1, 1) from a 64-bit LCG (Knuth's MMIX constants) */
static float next_uniform(void) {
  g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
  return (float)((double)(g_state >> 11) * (1.0 / 9007199254740992.0) * 2.0 - 1.0);
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static int dump(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (f == NULL) return 1;
  size_t w = fwrite(p, 1, bytes, f);
  fclose(f);
  return w == bytes ? 0 : 1;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s <output directory>\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  static const int lens_in[B] = {1, 17, 40};

  /* host pool: slots for every prompt token, then the tables */
  kvc_pool* pool = NULL;
  int64_t seqs[B], slots[T];
  int32_t table[B * MAXB], lens[B];
  CHECK(kvc_pool_create(NB, BS, &pool));
  int t0 = 0;
  for (int i = 0; i < B; ++i) {
    CHECK(kvc_seq_add(pool, &seqs[i]));
    CHECK(kvc_seq_reserve(pool, seqs[i], lens_in[i], slots + t0));
    t0 += lens_in[i];
  }
  CHECK(kvc_build_block_tables(pool, seqs, B, table, MAXB, lens));

  /* inputs */
  static uint16_t k_all[T * HKV * D], v_all[T * HKV * D], q[B * HQ * D];
  for (int i = 0; i < T * HKV * D; ++i) k_all[i] = to_bf16(next_uniform());
  for (int i = 0; i < T * HKV * D; ++i) v_all[i] = to_bf16(next_uniform());
  for (int i = 0; i < B * HQ * D; ++i) q[i] = to_bf16(next_uniform());

  const size_t pool_bytes = (size_t)NB * HKV * BS * D * 2;
  void *d_k = NULL, *d_v = NULL, *d_kc = NULL, *d_vc = NULL, *d_q = NULL, *d_out = NULL, *d_ws = NULL;
  void *d_slots = NULL, *d_table = NULL, *d_lens = NULL;
  CUDA(cudaMalloc(&d_k, sizeof k_all));
  CUDA(cudaMalloc(&d_v, sizeof v_all));
  CUDA(cudaMalloc(&d_q, sizeof q));
  CUDA(cudaMalloc(&d_kc, pool_bytes));
  CUDA(cudaMalloc(&d_vc, pool_bytes));
  CUDA(cudaMalloc(&d_out, (size_t)B * HQ * D * 4));
  CUDA(cudaMalloc(&d_slots, sizeof slots));
  CUDA(cudaMalloc(&d_table, sizeof table));
  CUDA(cudaMalloc(&d_lens, sizeof lens));
  CUDA(cudaMemset(d_kc, 0, pool_bytes));
  CUDA(cudaMemset(d_vc, 0, pool_bytes));
  CUDA(cudaMemcpy(d_k, k_all, sizeof k_all, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_v, v_all, sizeof v_all, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_q, q, sizeof q, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_slots, slots, sizeof slots, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_table, table, sizeof table, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_lens, lens, sizeof lens, cudaMemcpyHostToDevice));

  size_t ws_bytes = 0;
  CHECK(kvc_decode_workspace_size(B, HQ, HKV, D, BS, MAXB, &ws_bytes));
  if (ws_bytes > 0) {
    CUDA(cudaMalloc(&d_ws, ws_bytes));
    CUDA(cudaMemset(d_ws, 0, ws_bytes));
  }

  /* the path: append the prompts, then decode (default stream) */
  CHECK(kvc_append(d_k, d_v, (const int64_t*)d_slots, T, d_kc, d_vc, NB, BS, HKV, D, KVC_BF16, NULL));
  const float scale = 1.0f / sqrtf((float)D);
  CHECK(kvc_decode_attention(d_q, d_kc, d_vc, (const int32_t*)d_table, MAXB, (const int32_t*)d_lens, B, scale, HQ,
                             HKV, D, BS, NB, KVC_BF16, d_out, KVC_F32, d_ws, ws_bytes, NULL));
  uint32_t flags = 0;
  CHECK(kvc_get_error_flags(NULL, &flags));
  if (flags != 0) {
    fprintf(stderr, "device error flags 0x%x\n", flags);
    return 3;
  }

  static uint16_t kc[NB * HKV * BS * D], vc[NB * HKV * BS * D];
  static float out[B * HQ * D];
  CUDA(cudaMemcpy(kc, d_kc, pool_bytes, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(vc, d_vc, pool_bytes, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost));

  int bad = 0;
  bad |= dump(dir, "k_all.bin", k_all, sizeof k_all);
  bad |= dump(dir, "v_all.bin", v_all, sizeof v_all);
  bad |= dump(dir, "q.bin", q, sizeof q);
  bad |= dump(dir, "slots.bin", slots, sizeof slots);
  bad |= dump(dir, "table.bin", table, sizeof table);
  bad |= dump(dir, "lens.bin", lens, sizeof lens);
  bad |= dump(dir, "k_cache.bin", kc, sizeof kc);
  bad |= dump(dir, "v_cache.bin", vc, sizeof vc);
  bad |= dump(dir, "out.bin", out, sizeof out);
  if (bad) {
    fprintf(stderr, "could not write the results to %s\n", dir);
    return 4;
  }

  cudaFree(d_k);
  cudaFree(d_v);
  cudaFree(d_q);
  cudaFree(d_kc);
  cudaFree(d_vc);
  cudaFree(d_out);
  cudaFree(d_slots);
  cudaFree(d_table);
  cudaFree(d_lens);
  if (d_ws != NULL) cudaFree(d_ws);
  kvc_pool_destroy(pool);
  printf("decode from C ok\n");
  return 0;
}
