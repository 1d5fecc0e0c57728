// GQA decode on the 5th-generation tensor cores for wide query groups.
//
// What is computed is the paged decode of "KV缓存原理与显存估算" knowledge
// point 2 (with the head grouping of "KV-Cache——为什么AI回复越来越快" section
// 03): every query head attends its kv head's cached rows read through the
// block table, softmax(scale * q . k) weighting v. With n_tok new tokens per
// sequence (the chunk mask of "单请求 KV Cache": query row t sees the rows up
// to past_len + t) the n_tok * group queries of a kv head are its "virtual
// heads" v = t * group + j.
//
// When a kv head has 8 to 32 queries the CUDA-core kernel is bound by its
// FMA issue rate (every cached element feeds one FMA per query), so this
// kernel runs the two contractions of a 128-row tile of one kv head on
// tcgen05.mma with the cache rows on the M side:
//     S^T [128 rows x NQ]  = K_tile [128 x 128] . Q^T [128 x NQ]
//     O^T [128 dims x NQ] += V_tile^T [128 x 128 rows] . P^T [128 rows x NQ]
// (NQ = the queries padded to 16 or 32, the MMA N). Both accumulators sit in
// TMEM. A softmax thread owns one row of S^T (all queries of that cache row)
// and, for the output, one dim of O^T. The running maximum of each query is
// shared by the 128 threads and only raised (with a rescale of O^T) when a
// score exceeds it by more than 2^8 (a barrier-reduced vote per tile); the
// sums are kept per thread and reduced once per segment. P = exp2(s - m) is
// written to shared memory in two bf16 (or f16) parts, hi and lo = p - hi,
// as the B operand of the PV products, so the weights keep ~2^-17 accuracy.
//
// * Pages reach shared memory by TMA (a 2-D tensor map over the pool viewed
//   as [num_blocks * n_kv_heads * block_size rows, 128]), one [block_size x
//   64] box per page and 64-column half, 128B-swizzled: the K tile is read
//   K-major as the A operand of S^T, the V tile MN-major as the A operand
//   of O^T. The query rows of a unit are staged by the softmax threads with
//   the same swizzle.
// * Roles: warps 0-3 softmax and epilogue, warp 4 TMA producer, warp 5 MMA
//   issuer and TMEM owner. Three K+V stages (64 KB each), S^T double
//   buffered, MMA order S(t), PV(t-1), S(t+1), PV(t).
// * Work split, records and merge as in the CUDA-core kernel: the tiles of
//   all (sequence, kv head) units are laid end to end, CTA c takes a
//   contiguous range, a unit cut by a range boundary leaves fp32 records
//   (m, l, O) and the last contributing CTA merges them (log-sum-exp rule).
// * Every wait is bounded; a wait that gives up sets KVC_FLAG_TIMEOUT and an
//   abort flag that stops every role, which then drains and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "decode_gqa.h"
#include "kvc_device.cuh"
#include "kvc_internal.h"
#include "umma.cuh"

namespace kvc {
namespace wide {

using namespace umma;

constexpr int kD = 128;          // head_dim
constexpr int kRows = 128;       // cache rows per tile (M of S^T)
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kMaxBatch = 512;
constexpr uint32_t kHalfBytes = kRows * 128;     // one 64-column half of a K or V tile
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // K or V tile
constexpr uint32_t kStageBytes = 2 * kTileBytes;  // K + V
constexpr uint32_t kTmemCols = 128;
constexpr int kMergeChunk = 64;

// Shared memory (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffQ = kStages * kStageBytes;
__host__ __device__ constexpr uint32_t off_p(int nq) { return kOffQ + nq * 256; }
__host__ __device__ constexpr uint32_t off_red(int nq) { return off_p(nq) + nq * 512; }
enum {
  B_QFULL = 0, B_QEMPTY, B_FULL0, B_EMPTY0 = B_FULL0 + kStages, B_SFULL0 = B_EMPTY0 + kStages,
  B_SEMPTY0 = B_SFULL0 + 2, B_PFULL = B_SEMPTY0 + 2, B_PEMPTY, B_OFREE, B_FINAL, B_COUNT
};
__host__ __device__ constexpr uint32_t off_hide(int nq) { return off_red(nq) + 4 * nq * 4; }
__host__ __device__ constexpr uint32_t off_bar(int nq) { return off_hide(nq) + nq * 4; }
__host__ __device__ constexpr uint32_t off_misc(int nq) { return off_bar(nq) + B_COUNT * 8; }
__host__ __device__ constexpr uint32_t off_rec(int nq) { return off_misc(nq) + 16; }
__host__ __device__ constexpr uint32_t off_scan(int nq) { return off_rec(nq) + kMergeChunk * 4; }
__host__ __device__ constexpr uint32_t smem_bytes(int nq, int batch) {
  return off_scan(nq) + (batch + 1 + 32) * 4 + 1024;
}

struct Params {
  const void* q;                 // [batch, n_tok, n_q_heads, 128]
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;                     // [batch, n_tok, n_q_heads, 128]
  float* rec_o;                  // [G * 2, NQ, 128]
  float* rec_ml;                 // [G * 2, NQ, 2]
  unsigned int* counters;        // [batch * n_kv_heads]
  unsigned int* err;
  int64_t num_blocks;
  int batch, n_q_heads, n_kv_heads, group, n_tok, qn;  // qn = n_tok * group queries per kv head
  int block_size, max_blocks, out_dtype, unit_mode;
  int causal;                    // n_tok > 1: token t sees rows up to n - n_tok + t (0: every row)
  float* lse;                    // non-NULL: per output row, max + log2(sum) in log2 units
  float qscale;                  // scale * log2(e)
};

// ------------------------------------------------------- work bookkeeping

__device__ __forceinline__ int seq_rows(const Params& p, int b) {
  const int n = __ldg(p.context_lens + b);
  if ((p.causal && n < p.n_tok) || n < 1) return 0;
  const int cap = p.block_size * p.max_blocks;
  return n < cap ? n : cap;
}
__device__ __forceinline__ int seq_tiles(const Params& p, int b) { return (seq_rows(p, b) + kRows - 1) / kRows; }

// Exclusive prefix sums of tiles per sequence into s_scan[0..B] (whole CTA).
__device__ inline void scan_tiles(const Params& p, int* s_scan) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    int run = 0;
    for (int base = 0; base < p.batch; base += 32) {
      const int b = base + tid;
      const int v = b < p.batch ? seq_tiles(p, b) : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += u;
      }
      if (b < p.batch) s_scan[b] = run + x - v;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (tid == 0) s_scan[p.batch] = run;
  }
  __syncthreads();
}

__device__ __forceinline__ int64_t range_start(int64_t c, int64_t G, int64_t N) { return c * N / G; }
__device__ __forceinline__ int64_t cta_of(int64_t t, int64_t G, int64_t N) { return ((t + 1) * G - 1) / N; }

// A run of tiles of one (sequence, kv head) unit inside this CTA's range.
// Positions: pos = H * S[seq] + kvh * nt + tile (H = n_kv_heads, nt = tiles
// of the sequence, S = exclusive prefix sums of nt).
struct Segment {
  int seq, kvh, t0, t1, nt;
  int64_t u0;  // position of the unit's first tile
  int which;   // record slot: 0 if the segment starts this CTA's range
};

struct Walker {
  int64_t pos, hi, lo;
  __device__ bool next(const Params& p, const int* s_scan, Segment& sg) {
    if (pos >= hi) return false;
    const int H = p.n_kv_heads;
    if (p.unit_mode) {
      sg.seq = static_cast<int>(pos / H);
      sg.kvh = static_cast<int>(pos - static_cast<int64_t>(sg.seq) * H);
      sg.nt = seq_tiles(p, sg.seq);
      sg.t0 = 0;
      sg.t1 = sg.nt;
      sg.u0 = 0;
      sg.which = 0;
      pos = hi;
      return true;
    }
    int a = 0, b = p.batch - 1;  // largest sequence with H * S[seq] <= pos
    while (a < b) {
      const int mid = (a + b + 1) >> 1;
      if (static_cast<int64_t>(H) * s_scan[mid] <= pos) a = mid; else b = mid - 1;
    }
    sg.seq = a;
    sg.nt = s_scan[a + 1] - s_scan[a];
    const int64_t r = pos - static_cast<int64_t>(H) * s_scan[a];
    sg.kvh = static_cast<int>(r / sg.nt);
    sg.t0 = static_cast<int>(r - static_cast<int64_t>(sg.kvh) * sg.nt);
    sg.u0 = pos - sg.t0;
    const int64_t end = (sg.u0 + sg.nt < hi) ? sg.u0 + sg.nt : hi;
    sg.t1 = static_cast<int>(end - sg.u0);
    sg.which = (pos == lo) ? 0 : 1;
    pos = end;
    return true;
  }
};

// Output row (of [batch * n_tok * n_q_heads]) of virtual head v of kv head kvh.
__device__ __forceinline__ int64_t out_row(const Params& p, int seq, int kvh, int v) {
  const int t = v / p.group, j = v - t * p.group;
  return (static_cast<int64_t>(seq) * p.n_tok + t) * p.n_q_heads + kvh * p.group + j;
}

__device__ __forceinline__ uint16_t to_bits(float x, bool bf16) {
  if (bf16) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t*>(&h);
  }
  const __half h = __float2half_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}
__device__ __forceinline__ float from_bits(uint16_t b, bool bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
  __half h;
  *reinterpret_cast<uint16_t*>(&h) = b;
  return __half2float(h);
}

// Warp max / sum.
__device__ __forceinline__ float wmax(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// OR of `pred` over the 128 softmax threads (named barrier 1).
__device__ __forceinline__ bool block_any128(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void sync128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// ------------------------------------------------------------------ kernel

template <int NQ, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    wide_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const Params p) {
  static_assert(NQ == 16 || NQ == 32, "queries per kv head padded to 16 or 32");
  constexpr int NC = NQ / 16;  // 16-column TMEM loads per row
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (base - raw_addr);
  const uint32_t sStage = base + kOffStage, sQ = base + kOffQ, sP = base + off_p(NQ);
  float* s_red = reinterpret_cast<float*>(sm + off_red(NQ));  // [4][NQ]
  // per query: rows it may not see at the end of a sequence (its later new
  // tokens), or a huge value for padding queries
  int* s_hide = reinterpret_cast<int*>(sm + off_hide(NQ));
  const uint32_t bar0 = base + off_bar(NQ);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + off_bar(NQ));
  volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(sm + off_misc(NQ));
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + off_misc(NQ) + 4);
  volatile int* s_last = reinterpret_cast<volatile int*>(sm + off_misc(NQ) + 8);
  int* s_rec = reinterpret_cast<int*>(sm + off_rec(NQ));
  int* s_scan = reinterpret_cast<int*>(sm + off_scan(NQ));
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  const int bs = p.block_size;

  if (tid < NQ)
    s_hide[tid] = tid < p.qn ? (p.causal ? p.n_tok - 1 - tid / p.group : 0) : (1 << 30);
  if (tid == 0) {
    *s_abort = 0;
    for (int i = 0; i < B_COUNT; ++i) {
      // Q full, S empty, P full, O free: the four softmax warps; all others: one.
      uint32_t cnt = 1;
      if (i == B_QFULL || i == B_SEMPTY0 || i == B_SEMPTY0 + 1 || i == B_PFULL || i == B_OFREE) cnt = 4;
      mbar_init(&bars[i], cnt);
    }
    fence_barrier_init();
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + off_misc(NQ)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Launched behind the previous kernel of the stream (programmatic stream
  // serialisation), the set-up above overlapped it; every thread waits for
  // that grid to finish before it reads or writes any caller buffer.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (blockIdx.x == 0) {
    for (int b = tid; b < p.batch; b += blockDim.x) {
      const int n = __ldg(p.context_lens + b);
      if ((p.causal && n < p.n_tok) || n < 1 || n > bs * p.max_blocks) set_flag(p.err, 0x2u);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *s_tmem;

  Walker walk;
  int64_t N_all = 0;
  if (p.unit_mode) {
    walk.lo = walk.pos = c;
    walk.hi = c + 1;
  } else {
    scan_tiles(p, s_scan);
    N_all = static_cast<int64_t>(p.n_kv_heads) * s_scan[p.batch];
    walk.lo = walk.pos = range_start(c, G, N_all);
    walk.hi = range_start(c + 1, G, N_all);
  }
  // Zero outputs of sequences with an invalid length (no tile visits them):
  // CTA 0 in the split mode, the unit's own CTA in the unit mode.
  {
    const int row_elems = p.n_tok * p.n_q_heads * kD;
    if (p.unit_mode) {
      const int seq = static_cast<int>(c / p.n_kv_heads), kvh = static_cast<int>(c % p.n_kv_heads);
      if (seq_tiles(p, seq) == 0) {
        for (int i = tid; i < p.qn * kD; i += blockDim.x)
          store_out(p.out, out_row(p, seq, kvh, i / kD) * kD + i % kD, 0.f, p.out_dtype);
        if (p.lse != nullptr && tid < p.qn) p.lse[out_row(p, seq, kvh, tid)] = -__builtin_huge_valf();
      }
    } else if (blockIdx.x == 0) {
      int bad = 0;
      for (int b = tid; b < p.batch; b += blockDim.x) bad |= (seq_tiles(p, b) == 0) ? 1 : 0;
      if (__syncthreads_or(bad)) {
        for (int b = 0; b < p.batch; ++b) {
          if (seq_tiles(p, b) != 0) continue;
          for (int i = tid; i < row_elems; i += blockDim.x)
            store_out(p.out, static_cast<int64_t>(b) * row_elems + i, 0.f, p.out_dtype);
          if (p.lse != nullptr)
            for (int i = tid; i < p.n_tok * p.n_q_heads; i += blockDim.x)
              p.lse[static_cast<int64_t>(b) * p.n_tok * p.n_q_heads + i] = -__builtin_huge_valf();
        }
      }
    }
  }
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // The whole warp: lane i reads the table entry of page i of the next tile
    // before the stage is free (hiding that load), lane 0 arms the stage's
    // barrier, then lane i issues the four copies of page i.
    uint32_t g = 0;
    uint32_t issued[kStages] = {};
    Segment sg;
    Walker w = walk;
    bool ok = true;
    while (ok && w.next(p, s_scan, sg)) {  // every decision below is uniform over the warp
      if (sg.nt == 0) continue;
      const int n_rows = seq_rows(p, sg.seq);
      const int32_t* bt = p.block_tables + static_cast<int64_t>(sg.seq) * p.max_blocks;
      for (int t = sg.t0; t < sg.t1; ++t, ++g) {
        if (__shfl_sync(0xffffffffu, *s_abort ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        const int st = g % kStages;
        const int r0 = t * kRows, r1 = min(n_rows, r0 + kRows);
        const int j0 = r0 / bs, npg = (r1 + bs - 1) / bs - j0;  // table entries of the tile (<= 128 / bs)
        int phys = lane < npg ? __ldg(bt + j0 + lane) : 0;
        bool got = true;
        if (lane == 0 && g >= kStages) got = wait_phase(bar(B_EMPTY0 + st), (g / kStages - 1) & 1u, s_abort, p.err);
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) arrive_expect(bar(B_FULL0 + st), static_cast<uint32_t>(npg) * bs * 512u);
        __syncwarp();
        if (lane < npg) {
          if (phys < 0 || phys >= p.num_blocks) {
            set_flag(p.err, 0x1u);
            phys = 0;  // keep the pipeline moving on valid memory; the output is flagged
          }
          const int y = (phys * p.n_kv_heads + sg.kvh) * bs;
          const uint32_t dk = sStage + st * kStageBytes, dv = dk + kTileBytes;
          const uint32_t off = static_cast<uint32_t>(lane * bs) * 128u;
          tma_load_2d(dk + off, &tm_k, 0, y, bar(B_FULL0 + st));
          tma_load_2d(dk + kHalfBytes + off, &tm_k, 64, y, bar(B_FULL0 + st));
          tma_load_2d(dv + off, &tm_v, 0, y, bar(B_FULL0 + st));
          tma_load_2d(dv + kHalfBytes + off, &tm_v, 64, y, bar(B_FULL0 + st));
        }
        ++issued[st];
      }
    }
    if (*s_abort && lane == 0) {
      // Copies still in flight must land before this shared memory goes away.
      for (int st = 0; st < kStages; ++st) {
        if (issued[st] == 0) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!try_wait(bar(B_FULL0 + st), (issued[st] - 1) & 1u) && globaltimer_ns() - t0 < kWaitNs) {
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = instr_desc(128, NQ, 0, 0, BF16);
      const uint32_t id_pv = instr_desc(128, NQ, 1, 0, BF16);
      const uint32_t d_o = tmem + 2 * NQ;
      uint32_t g = 0, seg_i = 0;
      Segment sg;
      Walker w = walk;
      bool ok = true;
      while (ok && !*s_abort && w.next(p, s_scan, sg)) {
        if (sg.nt == 0) continue;
        if (!wait_phase(bar(B_QFULL), seg_i & 1u, s_abort, p.err)) break;
        fence_after();
        const uint32_t g_first = g;
        // PV of tile gi: O^T (+)= V^T P_hi^T + V^T P_lo^T, A = V^T read MN-major.
        auto issue_pv = [&](uint32_t gi) -> bool {
          if (!wait_phase(bar(B_PFULL), gi & 1u, s_abort, p.err)) return false;
          const bool first = (gi == g_first);
          if (first && seg_i > 0 && !wait_phase(bar(B_OFREE), (seg_i - 1) & 1u, s_abort, p.err)) return false;
          fence_after();
          const uint32_t st = gi % kStages;
          const uint32_t v0 = sStage + st * kStageBytes + kTileBytes;
#pragma unroll
          for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int ks = 0; ks < kRows / 16; ++ks) {
              const uint64_t a = smem_desc(v0 + ks * 2048, kHalfBytes, 1024, 2);
              const uint64_t b = smem_desc(sP + part * (NQ * 256) + (ks >> 2) * (NQ * 128) + (ks & 3) * 32, 16,
                                           1024, 2);
              mma(d_o, a, b, id_pv, (first && part == 0 && ks == 0) ? 0u : 1u);
            }
          }
          commit(bar(B_EMPTY0 + st));
          commit(bar(B_PEMPTY));
          return true;
        };
        for (int t = sg.t0; t < sg.t1 && ok; ++t, ++g) {
          const uint32_t st = g % kStages, sb = g & 1u;
          if (!wait_phase(bar(B_FULL0 + st), (g / kStages) & 1u, s_abort, p.err)) { ok = false; break; }
          if (g >= 2 && !wait_phase(bar(B_SEMPTY0 + sb), ((g >> 1) - 1) & 1u, s_abort, p.err)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t k0 = sStage + st * kStageBytes;
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) {
            const uint64_t a = smem_desc(k0 + (ks >> 2) * kHalfBytes + (ks & 3) * 32, 16, 1024, 2);
            const uint64_t b = smem_desc(sQ + (ks >> 2) * (NQ * 128) + (ks & 3) * 32, 16, 1024, 2);
            mma(tmem + sb * NQ, a, b, id_s, ks == 0 ? 0u : 1u);
          }
          commit(bar(B_SFULL0 + sb));
          if (t == sg.t1 - 1) commit(bar(B_QEMPTY));
          if (t > sg.t0 && !issue_pv(g - 1)) { ok = false; break; }
        }
        if (ok && !issue_pv(g - 1)) ok = false;
        ++seg_i;
      }
      commit(bar(B_FINAL));
      const uint64_t t0 = globaltimer_ns();
      while (!try_wait(bar(B_FINAL), 0) && globaltimer_ns() - t0 < kWaitNs) {
      }
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    // Thread r: row r of every S^T tile, dim r of O^T (TMEM lane r).
    const int r = tid;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // The four warps meet at named barriers (the vote on the maxima, the
    // reductions), so they take every exit together: a wait that fails only
    // sets a local flag, and a barrier vote turns it into a common break.
    uint32_t g = 0, seg_i = 0;
    Segment sg;
    Walker w = walk;
    bool ok = true;
    while (ok && w.next(p, s_scan, sg)) {
      if (sg.nt == 0) continue;
      const int n_rows = seq_rows(p, sg.seq);
      // ---- stage the unit's query rows (NQ x 128, zero padded) as the
      // 128B-swizzled K-major B operand of S^T, once the previous segment's
      // S products are done with the buffer
      {
        const bool got = seg_i == 0 || wait_phase(bar(B_QEMPTY), (seg_i - 1) & 1u, s_abort, p.err);
        if (block_any128(!got || *s_abort)) {
          ok = false;
          break;
        }
      }
      {
        const uint16_t* qg = static_cast<const uint16_t*>(p.q);
        for (int i = tid; i < NQ * 16; i += 128) {
          const int v = i >> 4, ch = i & 15, half = ch >> 3, cc = ch & 7;
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (v < p.qn) x = __ldg(reinterpret_cast<const uint4*>(qg + out_row(p, sg.seq, sg.kvh, v) * kD + ch * 8));
          *reinterpret_cast<uint4*>(sm + kOffQ + half * (NQ * 128) + v * 128 + ((cc ^ (v & 7)) * 16)) = x;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) arrive(bar(B_QFULL));
      float m[NQ], lp[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        m[q] = -1e30f;  // finite: a query may meet only rows it may not see in a segment
        lp[q] = 0.f;
      }
      const uint32_t g_first = g;
      for (int t = sg.t0; t < sg.t1; ++t, ++g) {
        const uint32_t sb = g & 1u;
        // S^T(g) is in TMEM, and PV(g - 1) is done with P and O^T
        bool got = wait_phase_suspend(bar(B_SFULL0 + sb), (g >> 1) & 1u, s_abort, p.err);
        got = got && (g == 0 || wait_phase_suspend(bar(B_PEMPTY), (g - 1) & 1u, s_abort, p.err));
        if (block_any128(!got || *s_abort)) {
          ok = false;
          break;
        }
        fence_after();
        float s[NQ];
#pragma unroll
        for (int k = 0; k < NC; ++k) tmem_ld16(lane_addr + sb * NQ + 16 * k, s + 16 * k);
        fence_before();
        __syncwarp();
        if (lane == 0) arrive(bar(B_SEMPTY0 + sb));
        const int rows_left = n_rows - t * kRows;  // rows from this tile's first to the end
        bool need = false;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const bool vis = r + s_hide[q] < rows_left;
          s[q] = vis ? s[q] * p.qscale : -__builtin_huge_valf();
          need |= s[q] > m[q] + 8.0f;
        }
        if (block_any128(need)) {
          // raise the maxima to this tile's (all 128 threads agree)
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            const float mx = wmax(s[q]);
            if (lane == 0) s_red[warp * NQ + q] = mx;
          }
          sync128();
          float alpha[NQ];
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            const float mx = fmaxf(fmaxf(s_red[q], s_red[NQ + q]), fmaxf(s_red[2 * NQ + q], s_red[3 * NQ + q]));
            const float mn = fmaxf(m[q], mx);
            alpha[q] = fast_exp2(m[q] - mn);
            m[q] = mn;
            lp[q] *= alpha[q];
          }
          sync128();  // s_red is read by everyone before its next use
          if (g > g_first) {
            // O^T row r (dim r): column q scales by alpha[q]
#pragma unroll
            for (int k = 0; k < NC; ++k) {
              float o[16];
              tmem_ld16(lane_addr + 2 * NQ + 16 * k, o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= alpha[16 * k + i];
              tmem_st16(lane_addr + 2 * NQ + 16 * k, o);
            }
          }
        }
        // P^T hi / lo parts: element (query q, row r) of the K-major B operand
        {
          const int kb = r >> 6, cc = (r & 63) >> 3, e = r & 7;
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            const float pv = fast_exp2(s[q] - m[q]);
            lp[q] += pv;
            const uint16_t hb = to_bits(pv, BF16);
            const uint16_t lb = to_bits(pv - from_bits(hb, BF16), BF16);
            const uint32_t off = kb * (NQ * 128) + q * 128 + ((cc ^ (q & 7)) * 16) + e * 2;
            *reinterpret_cast<uint16_t*>(sm + off_p(NQ) + off) = hb;
            *reinterpret_cast<uint16_t*>(sm + off_p(NQ) + NQ * 256 + off) = lb;
          }
        }
        if (r >= rows_left) {
          // rows past the end of the sequence may hold anything (NaN too):
          // their weight is 0, but 0 x NaN is NaN, so their values are zeroed
          unsigned char* vrow = sm + kOffStage + (g % kStages) * kStageBytes + kTileBytes + r * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            *reinterpret_cast<uint4*>(vrow + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(vrow + kHalfBytes + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        fence_before();
        __syncwarp();
        if (lane == 0) arrive(bar(B_PFULL));
      }
      if (!ok) break;
      // ---- epilogue: sums over the 128 rows, O^T after the last PV
      float l[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const float v = wsum(lp[q]);
        if (lane == 0) s_red[warp * NQ + q] = v;
      }
      sync128();
#pragma unroll
      for (int q = 0; q < NQ; ++q) l[q] = (s_red[q] + s_red[NQ + q]) + (s_red[2 * NQ + q] + s_red[3 * NQ + q]);
      {
        const bool got = wait_phase(bar(B_PEMPTY), (g - 1) & 1u, s_abort, p.err);
        if (block_any128(!got || *s_abort)) break;  // after sync128: s_red is free again
      }
      fence_after();
      float o[NQ];
#pragma unroll
      for (int k = 0; k < NC; ++k) tmem_ld16(lane_addr + 2 * NQ + 16 * k, o + 16 * k);
      fence_before();
      __syncwarp();
      if (lane == 0) arrive(bar(B_OFREE));
      const bool whole = (sg.t0 == 0 && sg.t1 == sg.nt);
      const int64_t rec = c * 2 + sg.which;
      if (whole) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (q < p.qn) store_out(p.out, out_row(p, sg.seq, sg.kvh, q) * kD + r, o[q] / l[q], p.out_dtype);
          if (p.lse != nullptr && r == q && q < p.qn) p.lse[out_row(p, sg.seq, sg.kvh, q)] = m[q] + __log2f(l[q]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < NQ; ++q) p.rec_o[(rec * NQ + q) * kD + r] = o[q];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (r == q) {  // thread q writes query q's (max, sum)
            p.rec_ml[(rec * NQ + q) * 2] = m[q];
            p.rec_ml[(rec * NQ + q) * 2 + 1] = l[q];
          }
        }
        // count this record; the last contributor of the unit merges
        __threadfence();
        sync128();
        const int64_t c0 = cta_of(sg.u0, G, N_all), c1 = cta_of(sg.u0 + sg.nt - 1, G, N_all);
        const int64_t unit = static_cast<int64_t>(sg.seq) * p.n_kv_heads + sg.kvh;
        if (tid == 0) {
          int contributors = 0;
          for (int64_t x = c0; x <= c1; ++x)
            contributors += (range_start(x, G, N_all) != range_start(x + 1, G, N_all)) ? 1 : 0;
          const unsigned int old = atomicAdd(p.counters + unit, 1u);
          *s_last = 0;
          if (old + 1 == static_cast<unsigned int>(contributors)) {
            *s_last = 1;
          } else if (old + 1 > static_cast<unsigned int>(contributors)) {
            set_flag(p.err, 0x10u);
            atomicExch(p.counters + unit, 0u);
          }
        }
        sync128();
        if (*s_last) {
          __threadfence();
          // thread r merges dim r of every query over the unit's records
          const int span = static_cast<int>(c1 - c0 + 1);
          float M[NQ], L[NQ], O[NQ];
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            M[q] = -__builtin_huge_valf();
            L[q] = 0.f;
            O[q] = 0.f;
          }
          for (int b0 = 0; b0 < span; b0 += kMergeChunk) {
            const int nc = min(kMergeChunk, span - b0);
            sync128();
            if (tid < nc) {
              const int64_t x = c0 + b0 + tid;
              const int64_t f0 = range_start(x, G, N_all);
              s_rec[tid] =
                  (f0 == range_start(x + 1, G, N_all)) ? -1 : static_cast<int>(x * 2 + ((sg.u0 > f0) ? 1 : 0));
            }
            sync128();
            for (int i = 0; i < nc; ++i) {
              const int rs = s_rec[i];
              if (rs < 0) continue;
#pragma unroll
              for (int q = 0; q < NQ; ++q) {
                const int64_t rq = static_cast<int64_t>(rs) * NQ + q;
                const float mc = __ldcg(p.rec_ml + rq * 2);
                const float lc = __ldcg(p.rec_ml + rq * 2 + 1);
                const float oc = __ldcg(p.rec_o + rq * kD + r);
                const float mn = fmaxf(M[q], mc);
                const float a = fast_exp2(M[q] - mn), b = fast_exp2(mc - mn);  // M = -inf: a = 0
                L[q] = L[q] * a + lc * b;
                O[q] = O[q] * a + oc * b;
                M[q] = mn;
              }
            }
          }
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            if (q < p.qn) store_out(p.out, out_row(p, sg.seq, sg.kvh, q) * kD + r, O[q] / L[q], p.out_dtype);
            if (p.lse != nullptr && r == q && q < p.qn) p.lse[out_row(p, sg.seq, sg.kvh, q)] = M[q] + __log2f(L[q]);
          }
          if (tid == 0) p.counters[unit] = 0u;
        }
      }
      ++seg_i;
    }
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 5) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

int nq_for(int qn) { return qn <= 16 ? 16 : 32; }

size_t counter_bytes(int batch, int n_kv_heads) {
  return (static_cast<size_t>(batch) * n_kv_heads * 4 + 255) / 256 * 256;
}
size_t record_bytes_per_cta(int nq) { return 2ull * nq * (kD + 2) * sizeof(float); }

int64_t plan_ctas(const DeviceInfo* dev, int64_t units, int max_blocks, int block_size) {
  const int64_t tiles_upper = units * ((static_cast<int64_t>(max_blocks) * block_size + kRows - 1) / kRows);
  int64_t G = dev->num_sms;
  const int64_t forced = option(KVC_OPT_BLOCKS_PER_CTA);
  if (forced > 0) G = (tiles_upper * kRows / block_size + forced - 1) / forced;
  const int64_t cap = option(KVC_OPT_MAX_CTAS);
  if (cap > 0) G = std::min(G, cap);
  G = std::min(G, std::max<int64_t>(1, tiles_upper));
  return std::max<int64_t>(1, std::min<int64_t>(G, 1 << 20));
}

}  // namespace wide

bool wide_preferred(int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_blocks,
                    int n_tok, kvc_dtype dtype) {
  if (!wide_supported(batch, n_q_heads, n_kv_heads, head_dim, block_size, n_tok, dtype)) return false;
  if (option(KVC_OPT_GQA_ENGINE) == 2) return true;
  // Fixed cost per call ~31 us against ~14 us for the CUDA-core kernel, whose
  // streaming rate falls with the queries per kv head (~3.5 TB/s at 8, ~1.6 at
  // 16) where this kernel keeps ~6.1 TB/s: it pays from ~140 MB of cache at 8
  // queries and ~40 MB at 16. The bound below uses the table width, the most
  // the host knows about the lengths.
  const int qn = n_tok * (n_q_heads / n_kv_heads);
  const double rows = static_cast<double>(batch) * n_kv_heads * max_blocks * block_size;
  const double bytes = rows * head_dim * 2.0 * 2.0;  // K and V, 2-byte elements
  return bytes >= (512.0 * 1024.0 * 1024.0) / qn;
}

bool wide_supported(int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size, int n_tok,
                    kvc_dtype dtype) {
  const int64_t engine = option(KVC_OPT_GQA_ENGINE);
  if (engine == 1 || engine == 3) return false;
  if (dtype != KVC_BF16 && dtype != KVC_F16) return false;
  if (head_dim != wide::kD || batch > wide::kMaxBatch) return false;
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128) return false;
  const int qn = n_tok * (n_q_heads / n_kv_heads);
  return qn >= 8 && qn <= 32;
}

size_t wide_workspace_bytes(const DeviceInfo* dev, int batch, int n_q_heads, int n_kv_heads, int block_size,
                            int max_blocks, int n_tok) {
  const int qn = n_tok * (n_q_heads / n_kv_heads);
  const int nq = wide::nq_for(qn);
  const int64_t G = wide::plan_ctas(dev, static_cast<int64_t>(batch) * n_kv_heads, max_blocks, block_size);
  return wide::counter_bytes(batch, n_kv_heads) + static_cast<size_t>(G) * wide::record_bytes_per_cta(nq);
}

kvc_status wide_decode(const WideArgs& a, DeviceInfo* dev) {
  using namespace wide;
  const int group = a.n_q_heads / a.n_kv_heads;
  const int qn = a.n_tok * group;
  const int nq = nq_for(qn);
  const uint32_t smem = smem_bytes(nq, a.batch);
  if (smem > static_cast<uint32_t>(dev->max_smem_optin))
    return fail(KVC_ERR_UNSUPPORTED, "tensor-core decode needs %u bytes of shared memory", smem);
  if (a.num_blocks * a.n_kv_heads * a.block_size >= (1ll << 31))
    return fail(KVC_ERR_UNSUPPORTED, "pool too large for the tensor-core decode");
  auto encode = encode_fn();
  if (encode == nullptr) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  CUtensorMap tk, tv;
  const CUtensorMapDataType dt = a.dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD),
                              static_cast<cuuint64_t>(a.num_blocks * a.n_kv_heads * a.block_size)};
  const cuuint64_t strides[1] = {kD * 2ull};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(a.block_size)};
  const cuuint32_t es[2] = {1, 1};
  for (int i = 0; i < 2; ++i) {
    CUresult r = encode(i == 0 ? &tk : &tv, dt, 2, const_cast<void*>(i == 0 ? a.k_cache : a.v_cache), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "tensor map for the %s cache: CUresult %d", i ? "V" : "K",
                                       static_cast<int>(r));
  }
  Params p{};
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = a.out;
  p.err = dev->error_word;
  p.num_blocks = a.num_blocks;
  p.batch = a.batch;
  p.n_q_heads = a.n_q_heads;
  p.n_kv_heads = a.n_kv_heads;
  p.group = group;
  p.n_tok = a.n_tok;
  p.qn = qn;
  p.causal = a.causal;
  p.lse = a.lse;
  p.block_size = a.block_size;
  p.max_blocks = a.max_blocks;
  p.out_dtype = static_cast<int>(a.out_dtype);
  p.qscale = a.scale * 1.4426950408889634f;
  const int64_t units = static_cast<int64_t>(a.batch) * a.n_kv_heads;
  int64_t G = plan_ctas(dev, units, a.max_blocks, a.block_size);
  const size_t cb = counter_bytes(a.batch, a.n_kv_heads);
  const int64_t fit =
      a.workspace_bytes > cb ? static_cast<int64_t>((a.workspace_bytes - cb) / record_bytes_per_cta(nq)) : 0;
  int grid;
  if (fit >= 1) {
    G = std::min(G, fit);
    p.unit_mode = 0;
    p.counters = static_cast<unsigned int*>(a.workspace);
    p.rec_o = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + cb);
    p.rec_ml = p.rec_o + static_cast<size_t>(G) * 2 * nq * kD;
    grid = static_cast<int>(G);
  } else {
    p.unit_mode = 1;
    grid = static_cast<int>(units);
  }
  auto launch = [&](auto kernel) -> kvc_status {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(wide)");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tk, tv, p);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(wide)");
    return KVC_OK;
  };
  kvc_status s;
  const bool bf16 = a.dtype == KVC_BF16;
  if (nq == 16)
    s = bf16 ? launch(wide_decode_kernel<16, true>) : launch(wide_decode_kernel<16, false>);
  else
    s = bf16 ? launch(wide_decode_kernel<32, true>) : launch(wide_decode_kernel<32, false>);
  if (s != KVC_OK) return s;
  return finish_call(a.stream);
}

}  // namespace kvc
