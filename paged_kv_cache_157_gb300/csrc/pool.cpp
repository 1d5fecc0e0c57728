// Host-side refcounted block pool: block tables and slot mappings.
//
// Source: PagedAttention block management in "KV Cache（键值缓存）" section
// 2.3 (fixed-size blocks allocated on demand, a per-sequence table from
// logical to physical blocks, blocks shared between sequences by reference
// count) and the closing section of "KV缓存原理与显存估算" (a block is free
// again when its count reaches zero; physical capacity counts unique blocks).
//
// Policy: the free set is a min-heap, so a new block is always the lowest
// free id; sequence ids count up from 0 and are never reused. Appending into
// a partly filled block that another sequence also holds needs copy-on-write:
// kvc_seq_reserve refuses it, kvc_seq_reserve_cow first gives the writer a
// fresh block and reports the (shared, fresh) pair for kvc_copy_blocks.
#include <cstdint>
#include <functional>
#include <new>
#include <queue>
#include <unordered_map>
#include <vector>

#include "kvc_internal.h"

struct kvc_pool {
  int64_t num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> ref;
  std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> free_heap;
  struct Seq {
    std::vector<int64_t> blocks;
    int64_t length = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;
  int64_t next_id = 0;
};

namespace {

kvc_status find_seq(kvc_pool* pool, int64_t id, kvc_pool::Seq** out) {
  if (pool == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "pool is NULL");
  auto it = pool->seqs.find(id);
  if (it == pool->seqs.end()) return kvc::fail(KVC_ERR_INVALID_ARG, "unknown sequence %lld", static_cast<long long>(id));
  *out = &it->second;
  return KVC_OK;
}

}  // namespace

extern "C" {

kvc_status kvc_pool_create(int64_t num_blocks, int block_size, kvc_pool** pool) {
  kvc::clear_error();
  if (pool == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "pool is NULL");
  *pool = nullptr;
  if (num_blocks < 1 || block_size < 1) return kvc::fail(KVC_ERR_INVALID_ARG, "num_blocks and block_size must be >= 1");
  if (num_blocks > (1ll << 31) - 1) return kvc::fail(KVC_ERR_UNSUPPORTED, "num_blocks must fit in int32");
  kvc_pool* p = new (std::nothrow) kvc_pool();
  if (p == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "host allocation failed");
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->ref.assign(static_cast<size_t>(num_blocks), 0);
  std::vector<int64_t> ids(static_cast<size_t>(num_blocks));
  for (int64_t i = 0; i < num_blocks; ++i) ids[static_cast<size_t>(i)] = i;
  p->free_heap = decltype(p->free_heap)(std::greater<int64_t>(), std::move(ids));
  *pool = p;
  return KVC_OK;
}

void kvc_pool_destroy(kvc_pool* pool) { delete pool; }

kvc_status kvc_seq_add(kvc_pool* pool, int64_t* seq) {
  kvc::clear_error();
  if (pool == nullptr || seq == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "NULL argument");
  const int64_t id = pool->next_id++;
  pool->seqs[id] = kvc_pool::Seq{};
  *seq = id;
  return KVC_OK;
}

kvc_status kvc_seq_fork(kvc_pool* pool, int64_t parent, int64_t* child) {
  kvc::clear_error();
  kvc_pool::Seq* ps = nullptr;
  kvc_status s = find_seq(pool, parent, &ps);
  if (s != KVC_OK) return s;
  if (child == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "child is NULL");
  kvc_pool::Seq copy = *ps;
  for (int64_t b : copy.blocks) pool->ref[static_cast<size_t>(b)] += 1;
  const int64_t id = pool->next_id++;
  pool->seqs[id] = std::move(copy);
  *child = id;
  return KVC_OK;
}

kvc_status kvc_seq_reserve(kvc_pool* pool, int64_t seq, int64_t n_new, int64_t* slots_out) {
  kvc::clear_error();
  kvc_pool::Seq* sq = nullptr;
  kvc_status s = find_seq(pool, seq, &sq);
  if (s != KVC_OK) return s;
  if (n_new < 0) return kvc::fail(KVC_ERR_INVALID_ARG, "n_new must be >= 0");
  if (n_new == 0) return KVC_OK;
  if (slots_out == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "slots_out is NULL");
  const int64_t bs = pool->block_size;
  const int64_t n = sq->length;
  if (n % bs != 0 && pool->ref[static_cast<size_t>(sq->blocks.back())] > 1)
    return kvc::fail(KVC_ERR_UNSUPPORTED, "append into a shared, partly filled block needs copy-on-write");
  const int64_t need = (n + n_new + bs - 1) / bs - static_cast<int64_t>(sq->blocks.size());
  if (need > static_cast<int64_t>(pool->free_heap.size()))
    return kvc::fail(KVC_ERR_NO_BLOCKS, "need %lld blocks, %zu free", static_cast<long long>(need),
                     pool->free_heap.size());
  for (int64_t i = 0; i < n_new; ++i) {
    const int64_t pos = n + i;
    if (pos % bs == 0) {
      const int64_t b = pool->free_heap.top();
      pool->free_heap.pop();
      pool->ref[static_cast<size_t>(b)] = 1;
      sq->blocks.push_back(b);
    }
    slots_out[i] = sq->blocks[static_cast<size_t>(pos / bs)] * bs + pos % bs;
  }
  sq->length = n + n_new;
  return KVC_OK;
}

kvc_status kvc_seq_reserve_batch(kvc_pool* pool, const int64_t* seqs, int n, int64_t n_new, int64_t* slots_out) {
  kvc::clear_error();
  if (pool == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "pool is NULL");
  if (n < 0 || n_new < 0) return kvc::fail(KVC_ERR_INVALID_ARG, "n and n_new must be >= 0");
  if (n == 0 || n_new == 0) return KVC_OK;
  if (seqs == nullptr || slots_out == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "NULL argument");
  // check everything first, so that a refused batch changes nothing
  const int64_t bs = pool->block_size;
  std::vector<kvc_pool::Seq*> ss(static_cast<size_t>(n));
  std::unordered_map<int64_t, int> seen;
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    kvc_status s = find_seq(pool, seqs[i], &ss[static_cast<size_t>(i)]);
    if (s != KVC_OK) return s;
    if (!seen.emplace(seqs[i], i).second)
      return kvc::fail(KVC_ERR_INVALID_ARG, "sequence %lld appears twice", static_cast<long long>(seqs[i]));
    const kvc_pool::Seq* sq = ss[static_cast<size_t>(i)];
    if (sq->length % bs != 0 && pool->ref[static_cast<size_t>(sq->blocks.back())] > 1)
      return kvc::fail(KVC_ERR_UNSUPPORTED, "sequence %lld: append into a shared, partly filled block needs "
                       "copy-on-write", static_cast<long long>(seqs[i]));
    need += (sq->length + n_new + bs - 1) / bs - static_cast<int64_t>(sq->blocks.size());
  }
  if (need > static_cast<int64_t>(pool->free_heap.size()))
    return kvc::fail(KVC_ERR_NO_BLOCKS, "need %lld blocks, %zu free", static_cast<long long>(need),
                     pool->free_heap.size());
  for (int i = 0; i < n; ++i) {
    kvc_pool::Seq* sq = ss[static_cast<size_t>(i)];
    int64_t* out = slots_out + static_cast<int64_t>(i) * n_new;
    const int64_t len = sq->length;
    for (int64_t t = 0; t < n_new; ++t) {
      const int64_t pos = len + t;
      if (pos % bs == 0) {
        const int64_t b = pool->free_heap.top();
        pool->free_heap.pop();
        pool->ref[static_cast<size_t>(b)] = 1;
        sq->blocks.push_back(b);
      }
      out[t] = sq->blocks[static_cast<size_t>(pos / bs)] * bs + pos % bs;
    }
    sq->length = len + n_new;
  }
  return KVC_OK;
}

kvc_status kvc_seq_reserve_cow(kvc_pool* pool, int64_t seq, int64_t n_new, int64_t* slots_out, int64_t* copy_pair) {
  kvc::clear_error();
  kvc_pool::Seq* sq = nullptr;
  kvc_status s = find_seq(pool, seq, &sq);
  if (s != KVC_OK) return s;
  if (copy_pair == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "copy_pair is NULL");
  if (n_new < 0) return kvc::fail(KVC_ERR_INVALID_ARG, "n_new must be >= 0");
  copy_pair[0] = -1;
  copy_pair[1] = -1;
  const int64_t bs = pool->block_size;
  const int64_t n = sq->length;
  if (n_new > 0 && n % bs != 0 && pool->ref[static_cast<size_t>(sq->blocks.back())] > 1) {
    // the fresh copy and every new tail block must be available up front
    const int64_t need = 1 + (n + n_new + bs - 1) / bs - static_cast<int64_t>(sq->blocks.size());
    if (need > static_cast<int64_t>(pool->free_heap.size()))
      return kvc::fail(KVC_ERR_NO_BLOCKS, "need %lld blocks, %zu free", static_cast<long long>(need),
                       pool->free_heap.size());
    const int64_t old = sq->blocks.back();
    const int64_t fresh = pool->free_heap.top();
    pool->free_heap.pop();
    pool->ref[static_cast<size_t>(fresh)] = 1;
    pool->ref[static_cast<size_t>(old)] -= 1;
    sq->blocks.back() = fresh;
    copy_pair[0] = old;
    copy_pair[1] = fresh;
  }
  return kvc_seq_reserve(pool, seq, n_new, slots_out);
}

kvc_status kvc_seq_free(kvc_pool* pool, int64_t seq) {
  kvc::clear_error();
  kvc_pool::Seq* sq = nullptr;
  kvc_status s = find_seq(pool, seq, &sq);
  if (s != KVC_OK) return s;
  for (int64_t b : sq->blocks) {
    int32_t& r = pool->ref[static_cast<size_t>(b)];
    r -= 1;
    if (r == 0) pool->free_heap.push(b);
  }
  pool->seqs.erase(seq);
  return KVC_OK;
}

kvc_status kvc_seq_length(kvc_pool* pool, int64_t seq, int64_t* length) {
  kvc::clear_error();
  kvc_pool::Seq* sq = nullptr;
  kvc_status s = find_seq(pool, seq, &sq);
  if (s != KVC_OK) return s;
  if (length == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "length is NULL");
  *length = sq->length;
  return KVC_OK;
}

kvc_status kvc_block_refcount(kvc_pool* pool, int64_t block, int32_t* refcount) {
  kvc::clear_error();
  if (pool == nullptr || refcount == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "NULL argument");
  if (block < 0 || block >= pool->num_blocks) return kvc::fail(KVC_ERR_INVALID_ARG, "block out of range");
  *refcount = pool->ref[static_cast<size_t>(block)];
  return KVC_OK;
}

kvc_status kvc_build_block_tables(kvc_pool* pool, const int64_t* seqs, int n, int32_t* table_out, int max_blocks,
                                  int32_t* lens_out) {
  kvc::clear_error();
  if (pool == nullptr || (n > 0 && (seqs == nullptr || table_out == nullptr || lens_out == nullptr)))
    return kvc::fail(KVC_ERR_INVALID_ARG, "NULL argument");
  if (n < 0 || max_blocks < 1) return kvc::fail(KVC_ERR_INVALID_ARG, "n must be >= 0 and max_blocks >= 1");
  for (int i = 0; i < n; ++i) {
    kvc_pool::Seq* sq = nullptr;
    kvc_status s = find_seq(pool, seqs[i], &sq);
    if (s != KVC_OK) return s;
    if (static_cast<int64_t>(sq->blocks.size()) > max_blocks)
      return kvc::fail(KVC_ERR_INVALID_ARG, "sequence %lld has %zu blocks > max_blocks %d",
                       static_cast<long long>(seqs[i]), sq->blocks.size(), max_blocks);
    if (sq->length > INT32_MAX) return kvc::fail(KVC_ERR_UNSUPPORTED, "length exceeds int32");
  }
  for (int i = 0; i < n; ++i) {
    const kvc_pool::Seq& sq = pool->seqs[seqs[i]];
    int32_t* row = table_out + static_cast<int64_t>(i) * max_blocks;
    for (int j = 0; j < max_blocks; ++j)
      row[j] = j < static_cast<int>(sq.blocks.size()) ? static_cast<int32_t>(sq.blocks[static_cast<size_t>(j)]) : 0;
    lens_out[i] = static_cast<int32_t>(sq.length);
  }
  return KVC_OK;
}

kvc_status kvc_pool_get_stats(kvc_pool* pool, kvc_pool_stats* stats) {
  kvc::clear_error();
  if (pool == nullptr || stats == nullptr) return kvc::fail(KVC_ERR_INVALID_ARG, "NULL argument");
  kvc_pool_stats st{};
  st.num_blocks = pool->num_blocks;
  st.free_blocks = static_cast<int64_t>(pool->free_heap.size());
  st.unique_blocks = pool->num_blocks - st.free_blocks;
  for (const auto& kv : pool->seqs) {
    st.table_entries += static_cast<int64_t>(kv.second.blocks.size());
    st.useful_tokens += kv.second.length;
  }
  st.live_seqs = static_cast<int64_t>(pool->seqs.size());
  st.block_size = pool->block_size;
  *stats = st;
  return KVC_OK;
}

kvc_status kvc_slots_from_tables(const int32_t* block_tables, int rows, int max_blocks, int block_size,
                                 const int32_t* row_index, const int64_t* positions, int64_t n, int64_t* slots_out) {
  kvc::clear_error();
  if (n < 0 || rows < 0 || max_blocks < 1 || block_size < 1)
    return kvc::fail(KVC_ERR_INVALID_ARG, "bad sizes");
  if (n > 0 && (block_tables == nullptr || row_index == nullptr || positions == nullptr || slots_out == nullptr))
    return kvc::fail(KVC_ERR_INVALID_ARG, "NULL argument");
  for (int64_t i = 0; i < n; ++i) {
    const int32_t r = row_index[i];
    const int64_t pos = positions[i];
    if (r < 0 || r >= rows || pos < 0 || pos / block_size >= max_blocks)
      return kvc::fail(KVC_ERR_INVALID_ARG, "entry %lld outside the table", static_cast<long long>(i));
    const int64_t blk = block_tables[static_cast<int64_t>(r) * max_blocks + pos / block_size];
    slots_out[i] = blk * block_size + pos % block_size;
  }
  return KVC_OK;
}

}  // extern "C"
