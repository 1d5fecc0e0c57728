/* A plain C (C11) client of the library's host calls: the header compiles
 * as C and the block pool works through the C ABI alone. Builds the sharing
 * example of "KV缓存原理与显存估算" (closing section): two sequences that
 * share the blocks of a common prefix. Exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>

#include "kvc.h"

#define CHECK(x)                                                              \
  do {                                                                        \
    kvc_status s_ = (x);                                                      \
    if (s_ != KVC_OK) {                                                       \
      fprintf(stderr, "%s:%d: %s -> %d (%s)\n", __FILE__, __LINE__, #x, s_,   \
              kvc_last_error_message());                                      \
      return 1;                                                               \
    }                                                                         \
  } while (0)

int main(void) {
  kvc_pool* pool = NULL;
  int64_t a = -1, b = -1, slots[64], seqs[2], copy[2];
  int32_t table[2 * 4], lens[2];
  kvc_pool_stats st;
  CHECK(kvc_pool_create(16, 16, &pool));
  CHECK(kvc_seq_add(pool, &a));
  CHECK(kvc_seq_reserve(pool, a, 32, slots)); /* two full blocks: 0 and 1 */
  if (slots[0] != 0 || slots[31] != 31) return 2;
  CHECK(kvc_seq_fork(pool, a, &b)); /* b shares blocks 0 and 1 */
  seqs[0] = a;
  seqs[1] = b;
  CHECK(kvc_seq_reserve_batch(pool, seqs, 2, 1, slots)); /* one new token each: blocks 2 and 3 */
  if (slots[0] != 2 * 16 || slots[1] != 3 * 16) return 3;
  CHECK(kvc_build_block_tables(pool, seqs, 2, table, 4, lens));
  if (table[0] != 0 || table[1] != 1 || table[2] != 2 || table[4] != 0 || table[5] != 1 || table[6] != 3) return 4;
  if (lens[0] != 33 || lens[1] != 33) return 5;
  CHECK(kvc_pool_get_stats(pool, &st));
  if (st.unique_blocks != 4 || st.table_entries != 6 || st.useful_tokens != 66) return 6;
  /* b's last block is private: no copy-on-write needed */
  CHECK(kvc_seq_reserve_cow(pool, b, 1, slots, copy));
  if (copy[0] != -1 || slots[0] != 3 * 16 + 1) return 7;
  /* errors come back as status codes with a message, never as exceptions */
  if (kvc_seq_free(pool, 999) != KVC_ERR_INVALID_ARG || kvc_last_error_message()[0] == '\0') return 8;
  CHECK(kvc_seq_free(pool, a));
  CHECK(kvc_seq_free(pool, b));
  CHECK(kvc_pool_get_stats(pool, &st));
  if (st.free_blocks != 16 || st.live_seqs != 0) return 9;
  kvc_pool_destroy(pool);
  printf("pool from C ok\n");
  return 0;
}
