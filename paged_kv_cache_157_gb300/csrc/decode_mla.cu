// MLA absorbed decode on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What is computed ("KV Cache（键值缓存）" section 2.2, with W^UK and W^UV
// absorbed into the query and output side): for sequence i and head h,
//     z_t = scale * q~_h . c_t          (c_t = cached row, d_c + d_r = 576 wide)
//     a   = softmax(z) over the context_lens[i] cached rows (paged, block 64)
//     o_h = sum_t a_t c_t[0 : d_c]      (d_c = 512)
//
// Design (sm_103a, one CTA per SM):
// * A CTA works on 48-token tiles and one half (256) of the 512 output
//   dimensions; its partner CTA (adjacent in the grid) takes the other half of
//   the same tiles, so the latent tile is fetched from HBM once and the second
//   read is served by L2. Both compute S = Q~ C^T in full: the O half (128 x
//   256 fp32) alone takes half of the 512 TMEM columns, which the whole O would
//   fill.
// * Tile size: a tcgen05.mma with M = 128 and K = 16 costs ~50 cycles for any
//   N up to 64 (probe: 1276 MACs/cycle at N = 32, 2553 at N = 64, 3950 at N =
//   256), so S, 36 MMAs per tile, costs per token in inverse proportion to
//   the tile. 48 tokens is the largest tile whose three stages fit next to
//   the part of Q~ kept in shared memory.
// * TMEM (512 columns): O half at 0..255; two 48-column S/P buffers at
//   256..351, where the softmax warps overwrite S(t) in place with P(t) as two
//   bf16 parts (hi = bf16(p), lo = bf16(p - hi), 24 columns each, so hi + lo
//   carries p to about 2^-17); Q~ columns 0..319 as bf16 pairs at 352..511,
//   the A operand of the first 20 K steps of S. Q~ columns 320..575 sit in
//   shared memory (64 KB) next to three latent tile stages [48 x 576] (54 KB
//   each, 128B-swizzled K-major as TMA writes them and the MMA descriptors
//   read them). A stage is held from S(t) until PV(t); with three, the next
//   tiles' copies are in flight meanwhile. A tile may straddle two 64-token
//   cache blocks, so it arrives as 27 boxes of 16 rows x 64 columns.
// * Warp roles: warps 0-3 = softmax and epilogue (thread = head = TMEM lane),
//   warp 4 = TMA producer, warp 5 = MMA issuer and TMEM owner.
//   Per tile: S(t) = Q~ C_t^T (36 MMAs, K = 16 each, N = 48) -> softmax reads
//   S from TMEM, updates the running max lazily (O in TMEM is rescaled only
//   when the max grows by more than 2^8, after waiting for the previous PV),
//   writes P over S -> O += P_hi V_t + P_lo V_t (6 MMAs with A read from TMEM,
//   N = 256, V = this CTA's half of the first 512 columns of the same tile,
//   read MN-major). S(t+1) is queued before PV(t), so the tensor core works
//   while the softmax runs; S(t+2) reuses the buffer of P(t) once PV(t) is done.
// * Work split: as in the GQA kernel, the tiles of all sequences are laid end
//   to end and CTA pair c takes a contiguous range; a sequence cut by a range
//   boundary leaves fp32 records (m, l, O), the CTA holding its first tile
//   lists them, and a merge kernel launched right behind this one combines
//   every (sequence, half) with the log-sum-exp rule, all in parallel.
// * Every mbarrier wait is bounded; a wait that gives up sets the error word
//   and a shared abort flag that stops every role, which then drains and
//   frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {

namespace mla {

constexpr int kHeads = 128;          // M of every MMA
constexpr int kDc = 512;             // latent (value) width
constexpr int kW = 576;              // cached row width
constexpr int kKB = kW / 64;         // 64-element (128 B) K blocks of a row: 9
constexpr int kTile = 48;            // tokens per tile (MMA N for S)
constexpr int kBoxRows = 16;         // rows per TMA box (a box never straddles a cache block)
constexpr int kBoxes = kTile / kBoxRows;  // boxes per 64-column block of a tile: 3
constexpr int kHalf = kDc / 2;       // output dims per CTA: 256
constexpr int kStages = 3;           // latent tile stages
constexpr int kSPBufs = 2;           // S/P buffers in TMEM
constexpr int kThreads = 192;        // 6 warps
constexpr int kMaxBatch = 128;

// Q~ is split: columns [0, 320) live in TMEM (the A operand of the first 20
// K steps), columns [320, 576) in shared memory (4 blocks of 64 columns).
constexpr int kQTmemK = 320;                          // Q~ columns held in TMEM
constexpr int kQSmemKB0 = kQTmemK / 64;               // first 64-column block in shared memory: 5
constexpr uint32_t kQSub = kHeads * 128;              // one 64-column block of Q~: 16384
constexpr uint32_t kQBytes = (kKB - kQSmemKB0) * kQSub;  // 65536
constexpr uint32_t kTileBytes = kTile * kW * 2;      // 55296
constexpr uint32_t kTileSub = kTile * 128;           // one 64-column block of a tile: 6144
constexpr uint32_t kBoxBytes = kBoxRows * 128;       // one TMA box: 2048

// TMEM columns: O half at 0..255, two S/P buffers of kTile columns at
// 256..351 (P: the high bf16 parts of the weights in the first kTile / 2
// columns, 2 per column, then the low parts), Q~ columns 0..319 as bf16 pairs
// at 352..511.
constexpr uint32_t kColO = 0;
constexpr uint32_t kColSP = 256;
constexpr uint32_t kColQ = kColSP + kSPBufs * kTile;  // 352
constexpr uint32_t kTmemCols = 512;
static_assert(kColQ + kQTmemK / 2 == kTmemCols, "TMEM budget");

// Shared memory carve-up (offsets from the 1024-byte aligned base of the
// dynamic shared memory).
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffC = kOffQ + kQBytes;
constexpr uint32_t kOffBar = kOffC + kStages * kTileBytes;
// barrier indices
enum {
  B_QFULL = 0, B_QEMPTY, B_CFULL0, B_CEMPTY0 = B_CFULL0 + kStages, B_SFULL0 = B_CEMPTY0 + kStages,
  B_PFULL0 = B_SFULL0 + kSPBufs, B_PEMPTY0 = B_PFULL0 + kSPBufs, B_OFREE = B_PEMPTY0 + kSPBufs, B_FINAL, B_COUNT
};
constexpr uint32_t kOffMisc = kOffBar + B_COUNT * 8;  // tmem address, abort flag, last flag
constexpr uint32_t kOffScan = kOffMisc + 16;
constexpr uint32_t smem_bytes(int batch) { return kOffScan + (batch + 1 + 32) * 4; }

struct Params {
  const __nv_bfloat16* q;  // absorbed queries [batch, 128, 576]
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  float* rec_o;   // [G * 2, 128, 256]
  float* rec_ml;  // [G * 2, 128, 2]
  int* unit_lists;  // per (sequence, half): [record count (0: written whole)][record slots 0 .. list_cap-1]
  int list_cap;
  int64_t rec_slots;
  unsigned int* err;
  int64_t num_blocks;
  int batch;
  int max_blocks;
  int block_size;
  int out_dtype;
  int unit_mode;  // 1: CTA pair s handles all of sequence s
  float qscale;   // scale * log2(e)
};

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void arrive_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of a phase (never suspends the thread).
__device__ __forceinline__ bool test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait that also gives up as soon as another role has aborted. It
// spins on the non-blocking test: the hand-offs between roles are on the
// critical path of every tile, so a suspended waiter would add its wake-up
// latency to each of them.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned int* err) {
  if (test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kWaitLimit; ++i) {
    if (test_wait(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitNs) break;
    }
  }
  *abort_flag = 1;
  set_flag(err, 0x8u);
  return false;
}

// The same bound, but each probe may suspend the thread (try_wait) until the
// phase completes or a time hint runs out: the producer and MMA-issuer warps
// share their SM sub-partitions with softmax warps, and a spinning waiter
// would take issue slots from them.
__device__ __forceinline__ bool wait_phase_yield(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                 unsigned int* err) {
  if (try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kWaitLimit; ++i) {
    if (try_wait(bar, parity)) return true;
    if ((i & 7u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitNs) break;
    }
  }
  *abort_flag = 1;
  set_flag(err, 0x8u);
  return false;
}

// UMMA shared-memory descriptor: start address, leading / stride byte offsets,
// the fixed version bits of sm_100 descriptors and the swizzle mode
// (2 = 128B, 4 = 64B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swizzle) << 61);
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, K- or MN-major.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same MMA with the A operand read from tensor memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
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

// ------------------------------------------------------- work bookkeeping

__device__ __forceinline__ int seq_tiles(const int32_t* lens, int b, int bs, int max_blocks) {
  const int n = __ldg(lens + b);
  if (n < 1) return 0;
  const int cap = bs * max_blocks;
  return ((n < cap ? n : cap) + kTile - 1) / kTile;
}

__device__ __forceinline__ int seq_rows(const int32_t* lens, int b, int bs, int max_blocks) {
  const int n = __ldg(lens + b);
  if (n < 1) return 0;
  const int cap = bs * max_blocks;
  return n < cap ? n : cap;
}

// Split positions a sequence occupies ahead of its tiles. Starting a segment
// (loading Q~, refilling the tile pipeline, writing the segment's output)
// costs about as much as 6 tiles (per-CTA timestamps: CTA pairs whose range
// held 1, 2 and 3 segments finished at ~186, ~198 and ~207 us on the
// DeepSeek-V2 batch), so each sequence start counts as 6 positions of the
// balanced split; positions that are no tile carry no work.
constexpr int kSegCost = 6;

// Exclusive prefix sums of split positions per sequence: its tiles plus
// kSegCost (whole CTA participates).
__device__ inline void scan_tiles(const int32_t* lens, int B, int bs, int max_blocks, int* s_scan) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    int run = 0;
    for (int base = 0; base < B; base += 32) {
      const int b = base + tid;
      const int nt = b < B ? seq_tiles(lens, b, bs, max_blocks) : 0;
      const int v = nt > 0 ? nt + kSegCost : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += u;
      }
      if (b < B) s_scan[b] = run + x - v;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (tid == 0) s_scan[B] = run;
  }
  __syncthreads();
}

__device__ __forceinline__ int64_t range_start(int64_t c, int64_t G, int64_t N) { return c * N / G; }
__device__ __forceinline__ int64_t pair_of(int64_t t, int64_t G, int64_t N) { return ((t + 1) * G - 1) / N; }

// A contiguous run of tiles of one sequence handled by this CTA.
struct Segment {
  int seq, t0, t1, ntiles;  // tiles [t0, t1) of the sequence's ntiles
  int64_t u0;               // split position of the sequence's first tile
  int which;                // record slot (0: segment starts the CTA range)
};

// Walks this CTA's segments: returns false when the range is exhausted.
struct Walker {
  int64_t pos, hi;
  int64_t lo;
  __device__ bool next(const Params& p, const int* s_scan, Segment& sg) {
    if (p.unit_mode) {
      if (pos >= hi) return false;
      sg.seq = static_cast<int>(pos);
      sg.ntiles = seq_tiles(p.context_lens, sg.seq, p.block_size, p.max_blocks);
      sg.t0 = 0;
      sg.t1 = sg.ntiles;
      sg.u0 = 0;
      sg.which = 0;
      pos = hi;
      return true;
    }
    if (pos >= hi) return false;
    int a = 0, b = p.batch - 1;
    while (a < b) {
      const int mid = (a + b + 1) >> 1;
      if (s_scan[mid] <= pos) a = mid; else b = mid - 1;
    }
    sg.seq = a;
    sg.u0 = s_scan[a] + kSegCost;  // the positions before it are no tiles
    sg.ntiles = static_cast<int>(s_scan[a + 1] - sg.u0);
    if (pos < sg.u0) {
      pos = sg.u0;
      if (pos >= hi) return false;
    }
    sg.t0 = static_cast<int>(pos - sg.u0);
    const int64_t end = sg.u0 + sg.ntiles < hi ? sg.u0 + sg.ntiles : hi;
    sg.t1 = static_cast<int>(end - sg.u0);
    sg.which = (pos == lo) ? 0 : 1;
    pos = end;
    return true;
  }
};

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                      const Params p) {
  // 1024-byte alignment (the 128B swizzle atom of TMA and UMMA) is declared,
  // so the whole dynamic allocation is usable; a misplaced window is
  // refused before any copy or TMEM allocation.
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t base = smem_addr(smem_raw);
  if ((base & 1023u) != 0) {
    if (threadIdx.x == 0) set_flag(p.err, 0x8u);
    return;
  }
  unsigned char* sm = smem_raw;
  const uint32_t sQ = base + kOffQ, sC = base + kOffC;
  const uint32_t bar0 = base + kOffBar;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(sm + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + kOffMisc + 4);
  int* s_scan = reinterpret_cast<int*>(sm + kOffScan);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hf = blockIdx.x & 1;  // output half of this CTA
  const int64_t pair = blockIdx.x >> 1;
  const int64_t G = gridDim.x >> 1;

  if (tid == 0) {
    *s_abort = 0;
    for (int i = 0; i < B_COUNT; ++i) {
      // Q~ full: the producer's copy plus the four softmax warps' TMEM stores;
      // P full and O free: the four softmax warps; all others: one.
      uint32_t c = 1;
      if (i == B_QFULL) c = 5;
      if ((i >= B_PFULL0 && i < B_PFULL0 + kSPBufs) || i == B_OFREE) c = 4;
      mbar_init(&bars[i], c);
    }
    fence_barrier_init();
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + kOffMisc),
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
      if (n < 1 || n > p.block_size * p.max_blocks) set_flag(p.err, 0x2u);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *s_tmem;

  Walker walk;
  if (p.unit_mode) {
    walk.lo = walk.pos = pair;
    walk.hi = pair + 1;
  } else {
    scan_tiles(p.context_lens, p.batch, p.block_size, p.max_blocks, s_scan);
    const int64_t N = s_scan[p.batch];
    walk.lo = walk.pos = range_start(pair, G, N);
    walk.hi = range_start(pair + 1, G, N);
  }
  // zero outputs of sequences with an invalid length (no CTA visits them);
  // the lengths are checked in parallel first, so the common case costs one pass
  bool any_bad = false;
  if (blockIdx.x < 2) {
    int bad = 0;
    for (int b = tid; b < p.batch; b += blockDim.x) bad |= (__ldg(p.context_lens + b) < 1) ? 1 : 0;
    any_bad = __syncthreads_or(bad) != 0;
  }
  if (any_bad) {
    for (int b = 0; b < p.batch; ++b) {
      if (__ldg(p.context_lens + b) >= 1) continue;
      if (!p.unit_mode && tid == 0) p.unit_lists[static_cast<int64_t>(b * 2 + hf) * (1 + p.list_cap)] = 0;
      for (int idx = tid; idx < kHeads * kHalf; idx += blockDim.x) {
        const int h = idx / kHalf, d = idx % kHalf;
        store_out(p.out, (static_cast<int64_t>(b) * kHeads + h) * kDc + hf * kHalf + d, 0.f, p.out_dtype);
      }
    }
  }
  __syncthreads();

  const int64_t N_all = p.unit_mode ? 0 : s_scan[p.batch];

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the segments; lane 0 waits and issues. A tile may
    // straddle two cache blocks, so it arrives as 16-row boxes that each lie
    // in one block; the source row of every box is read from the block table
    // 32 boxes (about ten tiles) at a time, one box per lane, so a table read
    // never sits between two tiles' copies.
    uint32_t g = 0, seg_i = 0;
    uint32_t issued[kStages] = {};
    bool q_pending = false;
    Segment sg;
    Walker w = walk;
    bool ok = true;
    for (;;) {
      // every decision below is uniform over the warp (lane 0's view of the abort flag)
      if (__shfl_sync(0xffffffffu, *s_abort ? 1 : 0, 0) != 0 || !w.next(p, s_scan, sg)) break;
      if (sg.ntiles == 0) continue;
      if (lane == 0) {
        ok = seg_i == 0 || wait_phase_yield(bar(B_QEMPTY), (seg_i - 1) & 1u, s_abort, p.err);
        if (ok) {
          arrive_expect(bar(B_QFULL), kQBytes);
          for (int kb = kQSmemKB0; kb < kKB; ++kb)
            tma_load_3d(sQ + (kb - kQSmemKB0) * kQSub, &tm_q, kb * 64, 0, sg.seq, bar(B_QFULL));
          q_pending = true;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const int32_t* bt = p.block_tables + static_cast<int64_t>(sg.seq) * p.max_blocks;
      const int last_blk = (seq_rows(p.context_lens, sg.seq, p.block_size, p.max_blocks) - 1) / p.block_size;
      int win = -1 << 30;  // first box of the window the lanes hold
      int my_row = 0;      // source row (pool row of the box's first token) of box win + lane
      for (int t = sg.t0; t < sg.t1; ++t, ++g) {
        const int b0 = t * kBoxes;
        if (b0 + kBoxes > win + 32) {
          win = b0;
          // Rows past the end of the sequence read its last block (they are
          // masked out of the softmax and zeroed before PV).
          const int tok = (win + lane) * kBoxRows;
          const int j = min(tok / p.block_size, last_blk);
          int phys = __ldg(bt + j);
          if (phys < 0 || phys >= p.num_blocks) {
            set_flag(p.err, 0x1u);
            phys = 0;  // keep the pipeline moving on valid memory; the output is flagged
          }
          my_row = phys * p.block_size + tok % p.block_size;
        }
        int rows[kBoxes];
#pragma unroll
        for (int c = 0; c < kBoxes; ++c) rows[c] = __shfl_sync(0xffffffffu, my_row, b0 - win + c);
        const int st = g % kStages;
        if (lane == 0) {
          ok = g < kStages || wait_phase_yield(bar(B_CEMPTY0 + st), (g / kStages - 1) & 1u, s_abort, p.err);
          if (ok) {
            arrive_expect(bar(B_CFULL0 + st), kTileBytes);
#pragma unroll
            for (int c = 0; c < kBoxes; ++c)
              for (int kb = 0; kb < kKB; ++kb)
                tma_load_2d(sC + st * kTileBytes + kb * kTileSub + c * kBoxBytes, &tm_c, kb * 64, rows[c],
                            bar(B_CFULL0 + st));
            ++issued[st];
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      if (!ok) break;
      ++seg_i;
    }
    if (lane == 0 && *s_abort) {
      // Copies still in flight must land before this shared memory goes away:
      // wait (bounded) for the last phase of every barrier this warp armed.
      for (int st = 0; st < kStages; ++st) {
        if (issued[st] == 0) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!try_wait(bar(B_CFULL0 + st), (issued[st] - 1) & 1u) && globaltimer_ns() - t0 < kWaitNs) {
        }
      }
      if (q_pending && seg_i > 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!try_wait(bar(B_QFULL), (seg_i - 1) & 1u) && globaltimer_ns() - t0 < kWaitNs) {
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issuer
    // Tensor-pipe order per segment: S(t0), S(t0+1), PV(t0), S(t0+2), PV(t0+1),
    // ...: S of the next tile is always queued before PV of the tile whose
    // weights the softmax warps are computing, and both S and P are double
    // buffered, so the tensor core works while the softmax runs.
    if (lane == 0) {
      const uint32_t id_s = instr_desc(kHeads, kTile, 0, 0);
      const uint32_t id_pv = instr_desc(kHeads, kHalf, 0, 1);
      const uint64_t a_q0 = smem_desc(sQ, 16, 1024, 2);
      uint32_t g = 0, seg_i = 0;  // g: tiles issued so far (all segments)
      Segment sg;
      Walker w = walk;
      bool ok = true;
      while (ok && !*s_abort && w.next(p, s_scan, sg)) {
        if (sg.ntiles == 0) continue;
        if (!wait_phase_yield(bar(B_QFULL), seg_i & 1u, s_abort, p.err)) break;
        fence_after();
        const uint32_t g_first = g;
        // PV of global tile gi: O (+)= P_hi V + P_lo V with A = P from TMEM and
        // B = this CTA's half of the tile's first 512 columns, read MN-major.
        auto issue_pv = [&](uint32_t gi) -> bool {
          const uint32_t pb = gi % kSPBufs;
          if (!wait_phase_yield(bar(B_PFULL0 + pb), (gi / kSPBufs) & 1u, s_abort, p.err)) return false;
          const bool first = (gi == g_first);
          if (first && seg_i > 0 && !wait_phase_yield(bar(B_OFREE), (seg_i - 1) & 1u, s_abort, p.err)) return false;
          fence_after();
          const uint32_t st = gi % kStages;
          const uint64_t bv0 = smem_desc(sC + st * kTileBytes + (4 * hf) * kTileSub, kTileSub, 1024, 2);
#pragma unroll
          for (int part = 0; part < 2; ++part) {  // P_hi, then P_lo, against the same V rows
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks) {
              mma_bf16_ts(tmem + kColO, tmem + kColSP + pb * kTile + part * (kTile / 2) + ks * 8,
                          bv0 + ((ks * 2048) >> 4), id_pv, (first && part == 0 && ks == 0) ? 0u : 1u);
            }
          }
          mma_commit(bar(B_CEMPTY0 + st));
          mma_commit(bar(B_PEMPTY0 + pb));
          return true;
        };
        for (int t = sg.t0; t < sg.t1 && ok; ++t, ++g) {
          const uint32_t st = g % kStages;  // latent stage
          const uint32_t sb = g % kSPBufs;  // S/P buffer
          if (!wait_phase_yield(bar(B_CFULL0 + st), (g / kStages) & 1u, s_abort, p.err)) { ok = false; break; }
          // S(g) overwrites the buffer that held P(g - 2): PV(g - 2) must be done
          if (g >= kSPBufs && !wait_phase_yield(bar(B_PEMPTY0 + sb), (g / kSPBufs - 1) & 1u, s_abort, p.err)) {
            ok = false;
            break;
          }
          fence_after();
          {
            // Descriptors advance by constant offsets (in 16-byte units) from
            // one base per operand, so each K step costs one add.
            const uint64_t b0 = smem_desc(sC + st * kTileBytes, 16, 1024, 2);
            const uint32_t d_s = tmem + kColSP + sb * kTile;
#pragma unroll
            for (int ks = 0; ks < kW / 16; ++ks) {
              const int kb = ks >> 2, kin = ks & 3;
              const uint64_t b = b0 + static_cast<uint64_t>((kb * kTileSub + kin * 32) >> 4);
              if (ks < kQTmemK / 16) {
                mma_bf16_ts(d_s, tmem + kColQ + ks * 8, b, id_s, ks == 0 ? 0u : 1u);
              } else {
                const uint64_t a = a_q0 + static_cast<uint64_t>(((kb - kQSmemKB0) * kQSub + kin * 32) >> 4);
                mma_bf16(d_s, a, b, id_s, 1u);
              }
            }
          }
          mma_commit(bar(B_SFULL0 + sb));
          if (t == sg.t1 - 1) mma_commit(bar(B_QEMPTY));
          if (t > sg.t0 && !issue_pv(g - 1)) { ok = false; break; }
        }
        if (ok && !issue_pv(g - 1)) ok = false;
        ++seg_i;
      }
      // all MMAs of this CTA complete before TMEM is released
      mma_commit(bar(B_FINAL));
      const uint64_t t0 = globaltimer_ns();
      while (!try_wait(bar(B_FINAL), 0) && globaltimer_ns() - t0 < kWaitNs) {
      }
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int h = warp * 32 + lane;  // head = TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // The four warps meet at named barriers (the record count and the merge),
    // so they leave together: a failed wait ends only the tile loop, and a
    // barrier vote before each shared step turns any failure into a common exit.
    uint32_t g = 0, seg_i = 0;
    Segment sg;
    Walker w = walk;
    bool ok = true;
    // Columns [0, 320) of this head's Q~ row for segment number si (sequence
    // seq) go to TMEM (the A operand of the first 20 K steps of S), once the
    // previous segment's S MMAs are done: 40 16-byte loads issued in two
    // batches (one round trip each) before the TMEM stores. Returns false on
    // a failed wait (every warp of the group sees the same result).
    auto load_q = [&](uint32_t si, int seq) -> bool {
      const bool got = si == 0 || __all_sync(0xffffffffu, wait_phase(bar(B_QEMPTY), (si - 1) & 1u, s_abort, p.err));
      if (block_any128(!got || *s_abort)) return false;
      fence_after();
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(seq) * kHeads + h) * kW);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[80];
#pragma unroll
        for (int i = 0; i < 20; ++i) {
          const uint4 x = __ldg(qrow + half * 20 + i);
          r[4 * i] = x.x;
          r[4 * i + 1] = x.y;
          r[4 * i + 2] = x.z;
          r[4 * i + 3] = x.w;
        }
        tmem_st32u(lane_addr + kColQ + half * 80, r);
        tmem_st32u(lane_addr + kColQ + half * 80 + 32, r + 32);
        tmem_st16u(lane_addr + kColQ + half * 80 + 64, r + 64);
      }
      fence_before();
      __syncwarp();
      if (lane == 0) arrive(bar(B_QFULL));
      return true;
    };
    bool have_q = false;  // this segment's Q~ was loaded during the previous segment's epilogue
    while (ok && w.next(p, s_scan, sg)) {
      if (sg.ntiles == 0) continue;
      const int n_rows = seq_rows(p.context_lens, sg.seq, p.block_size, p.max_blocks);
      if (!have_q && !load_q(seg_i, sg.seq)) {
        ok = false;
        break;
      }
      have_q = false;
      // the segment after this one (this CTA's walk is known)
      Walker wn = w;
      Segment sn;
      bool has_next = false;
      while (wn.next(p, s_scan, sn)) {
        if (sn.ntiles > 0) {
          has_next = true;
          break;
        }
      }
      if (has_next) {
        // warm L2 with its rows, so that its Q~ load costs L2 round trips
        const char* nrow = reinterpret_cast<const char*>(p.q + (static_cast<int64_t>(sn.seq) * kHeads + h) * kW);
#pragma unroll
        for (int i = 0; i < 5; ++i) prefetch_l2(nrow + 128 * i);
      }
      float m = -__builtin_huge_valf(), l = 0.f;
      const uint32_t g_first = g;
      for (int t = sg.t0; t < sg.t1; ++t, ++g) {
        const uint32_t sb = g % kSPBufs, pb = sb;
        if (!__all_sync(0xffffffffu, wait_phase(bar(B_SFULL0 + sb), (g / kSPBufs) & 1u, s_abort, p.err))) {
          ok = false;
          break;
        }
        fence_after();
        float s[kTile];
        tmem_ld32(lane_addr + kColSP + sb * kTile, s);
        tmem_ld16(lane_addr + kColSP + sb * kTile + 32, s + 32);
        const int valid = n_rows - t * kTile;
        float mt = -__builtin_huge_valf();
#pragma unroll
        for (int i = 0; i < kTile; ++i) {
          s[i] = (i < valid) ? s[i] * p.qscale : -__builtin_huge_valf();
          mt = fmaxf(mt, s[i]);
        }
        // This buffer's previous P was read by PV(g - 2), done before S(g) was issued.
        if (g >= kSPBufs &&
            !__all_sync(0xffffffffu, wait_phase(bar(B_PEMPTY0 + pb), (g / kSPBufs - 1) & 1u, s_abort, p.err))) {
          ok = false;
          break;
        }
        // Lazy rescale, decided per warp: the TMEM accesses below are warp-wide.
        if (__any_sync(0xffffffffu, mt > m + 8.0f)) {
          const float m_new = fmaxf(m, mt);
          const float alpha = fast_exp2(m - m_new);  // 0 on the first tile of a segment
          if (g > g_first) {
            // O must hold PV(g - 1) before it is rescaled (rare: the running
            // max grew by more than 2^8)
            const uint32_t gp = g - 1;
            if (!__all_sync(0xffffffffu,
                            wait_phase(bar(B_PEMPTY0 + gp % kSPBufs), (gp / kSPBufs) & 1u, s_abort, p.err))) {
              ok = false;
              break;
            }
            fence_after();
            for (int c = 0; c < kHalf; c += 32) {
              float v[32];
              tmem_ld32(lane_addr + kColO + c, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= alpha;
              tmem_st32(lane_addr + kColO + c, v);
            }
          }
          l *= alpha;
          m = m_new;
        }
        // Row h of P in TMEM, over the S it was computed from: kTile / 2
        // columns of bf16 pairs (hi), then kTile / 2 (lo).
        uint32_t pk[kTile];
#pragma unroll
        for (int i = 0; i < kTile / 2; ++i) {
          const float p0 = fast_exp2(s[2 * i] - m), p1 = fast_exp2(s[2 * i + 1] - m);
          l += p0 + p1;
          const uint32_t hi = pack_bf16(p0, p1);
          pk[i] = hi;
          pk[kTile / 2 + i] = pack_bf16(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xffff0000u));
        }
        tmem_st32u(lane_addr + kColSP + pb * kTile, pk);
        tmem_st16u(lane_addr + kColSP + pb * kTile + 32, pk + 32);
        if (valid < kTile) {
          // Rows past the end of the sequence (the rest of its last block) may
          // hold anything, NaN included; their weight is 0, but 0 x NaN is NaN,
          // so this CTA's value columns of those rows are zeroed before PV
          // reads them (whole 128-byte rows: the swizzle only permutes within
          // a row). The proxy fence hands the writes to the tensor core.
          const int r0 = valid > 0 ? valid : 0;
          const int n16 = (kTile - r0) * 4 * 8;  // 16-byte chunks: rows x 4 value blocks x 8
          unsigned char* stg = sm + kOffC + (g % kStages) * kTileBytes + (4 * hf) * kTileSub;
          for (int i = tid; i < n16; i += 128) {
            const int row = r0 + i / 32, blk = (i / 8) % 4, c = i % 8;
            *reinterpret_cast<uint4*>(stg + blk * kTileSub + row * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        fence_before();
        __syncwarp();
        if (lane == 0) arrive(bar(B_PFULL0 + pb));
      }
      // The next segment's Q~ goes to TMEM before this epilogue, so that its
      // first S products run while the output is read out and stored.
      if (ok && has_next) {
        if (!load_q(seg_i + 1, sn.seq)) {
          ok = false;
          break;
        }
        have_q = true;
      }
      // ---- epilogue: wait for the last PV, read O, write output or record
      {
        const uint32_t gl = g - 1;
        const bool got = ok && __all_sync(0xffffffffu, wait_phase(bar(B_PEMPTY0 + gl % kSPBufs), (gl / kSPBufs) & 1u,
                                                                  s_abort, p.err));
        if (block_any128(!got || *s_abort)) {
          ok = false;
          break;
        }
      }
      fence_after();
      const bool whole = (sg.t0 == 0 && sg.t1 == sg.ntiles);
      const int64_t rec = (static_cast<int64_t>(blockIdx.x) * 2 + sg.which) * kHeads + h;
      const float inv = 1.0f / l;
      for (int c = 0; c < kHalf; c += 32) {
        float v[32];
        tmem_ld32(lane_addr + kColO + c, v);
        if (whole) {
          // this head's 32 consecutive output dims: 16-byte stores
          const int64_t o = (static_cast<int64_t>(sg.seq) * kHeads + h) * kDc + hf * kHalf + c;
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= inv;
#pragma unroll
          for (int i = 0; i < 32; i += 8) store_out_vec<8>(p.out, o + i, v + i, p.out_dtype);
        } else {
          float4* dst = reinterpret_cast<float4*>(p.rec_o + rec * kHalf + c);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
      if (!whole) {
        p.rec_ml[rec * 2] = m;
        p.rec_ml[rec * 2 + 1] = l;
      }
      fence_before();
      __syncwarp();
      if (lane == 0) arrive(bar(B_OFREE));
      if (!p.unit_mode && sg.t0 == 0) {
        // the CTA holding the unit's first tile lists its records for the merge kernel
        const int64_t c0 = pair_of(sg.u0, G, N_all), c1 = pair_of(sg.u0 + sg.ntiles - 1, G, N_all);
        int* lst = p.unit_lists + (static_cast<int64_t>(sg.seq) * 2 + hf) * (1 + p.list_cap);
        const int64_t span = c1 - c0 + 1;
        const int R = whole ? 0 : static_cast<int>(span < p.list_cap ? span : p.list_cap);
        for (int r = tid; r < R; r += 128) {
          const int64_t c = c0 + r;
          const int64_t f0 = range_start(c, G, N_all);
          lst[1 + r] = (f0 == range_start(c + 1, G, N_all)) ? -1
                                                              : static_cast<int>((c * 2 + hf) * 2 + ((sg.u0 > f0) ? 1 : 0));
        }
        if (tid == 0) lst[0] = R;
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

// ------------------------------------------------------------------ merge
//
// One CTA per (sequence, half, group of 8 heads), launched behind the decode
// kernel: thread t takes dims 16 (t & 15) .. + 15 of head 8 g + t / 16 of the
// half and folds the unit's records, listed by the CTA that held its first
// tile, with the log-sum-exp rule (the count and the first list entries are
// read together, then kMergeBatch records at a time; a sequence has only a
// few contributors).
constexpr int kMergeBatch = 4;
constexpr int kMergeGroups = kHeads / 8;

__global__ void __launch_bounds__(128) mla_merge_kernel(const Params p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int unit = static_cast<int>(blockIdx.x / kMergeGroups), hg = static_cast<int>(blockIdx.x % kMergeGroups);
  const int seq = unit >> 1, hf = unit & 1;
  const int t = threadIdx.x;
  const int* lst = p.unit_lists + static_cast<int64_t>(unit) * (1 + p.list_cap);
  const int first = (t < kMergeBatch && t < p.list_cap) ? __ldcg(lst + 1 + t) : -1;
  int R = __ldcg(lst);
  if (R <= 0) return;
  R = R < p.list_cap ? R : p.list_cap;
  __shared__ int s_rec[kMergeBatch];
  const int h = hg * 8 + (t >> 4), q = t & 15;
  float M = -__builtin_huge_valf(), L = 0.f;
  float4 O[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) O[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < R; base += kMergeBatch) {
    if (base > 0) __syncthreads();
    if (t < kMergeBatch) {
      const int e = base == 0 ? first : (base + t < R ? __ldcg(lst + 1 + base + t) : -1);
      s_rec[t] = (base + t < R && e >= 0 && e < p.rec_slots) ? e : -1;
    }
    __syncthreads();
    float mr[kMergeBatch], lr[kMergeBatch];
    float4 x[kMergeBatch][4];
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      const int rs = s_rec[i];
      mr[i] = -__builtin_huge_valf();
      lr[i] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) x[i][k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rs >= 0) {
        const int64_t r = static_cast<int64_t>(rs) * kHeads + h;
        mr[i] = __ldcg(p.rec_ml + r * 2);
        lr[i] = __ldcg(p.rec_ml + r * 2 + 1);
        const float4* src = reinterpret_cast<const float4*>(p.rec_o + r * kHalf) + 4 * q;
#pragma unroll
        for (int k = 0; k < 4; ++k) x[i][k] = __ldcg(src + k);
      }
    }
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      if (mr[i] == -__builtin_huge_valf()) continue;
      if (mr[i] > M) {
        const float sc = M == -__builtin_huge_valf() ? 0.f : fast_exp2(M - mr[i]);
        L *= sc;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          O[k].x *= sc;
          O[k].y *= sc;
          O[k].z *= sc;
          O[k].w *= sc;
        }
        M = mr[i];
      }
      const float f = fast_exp2(mr[i] - M);
      L += f * lr[i];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        O[k].x += f * x[i][k].x;
        O[k].y += f * x[i][k].y;
        O[k].z += f * x[i][k].z;
        O[k].w += f * x[i][k].w;
      }
    }
  }
  const float inv = 1.0f / L;
  float v[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[4 * k] = O[k].x * inv;
    v[4 * k + 1] = O[k].y * inv;
    v[4 * k + 2] = O[k].z * inv;
    v[4 * k + 3] = O[k].w * inv;
  }
  const int64_t o = (static_cast<int64_t>(seq) * kHeads + h) * kDc + hf * kHalf + 16 * q;
  store_out_vec<8>(p.out, o, v, p.out_dtype);
  store_out_vec<8>(p.out, o + 8, v + 8, p.out_dtype);
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

int plan_pairs(const DeviceInfo* dev, int batch, int max_blocks, int block_size) {
  const int64_t tiles_upper = static_cast<int64_t>(batch) * ((static_cast<int64_t>(max_blocks) * block_size + kTile - 1) / kTile);
  int64_t G2 = dev->num_sms / 2;
  const int64_t forced = option(KVC_OPT_BLOCKS_PER_CTA);
  if (forced > 0) G2 = (tiles_upper * kTile / block_size + forced - 1) / forced;
  const int64_t cap = option(KVC_OPT_MAX_CTAS);
  if (cap > 0) G2 = std::min<int64_t>(G2, std::max<int64_t>(1, cap / 2));
  G2 = std::min<int64_t>(G2, std::max<int64_t>(1, tiles_upper));
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(G2, 1 << 20)));
}

// Per (sequence, half): the record count and up to G2 record slots.
size_t list_bytes(int batch, int G2) {
  return (static_cast<size_t>(batch) * 2 * (1 + static_cast<size_t>(G2)) * 4 + 255) / 256 * 256;
}
size_t record_bytes_per_pair() { return 2ull * 2 * kHeads * (kHalf + 2) * sizeof(float); }

kvc_status check(int batch, int n_q_heads, int d_c, int d_r, int block_size, int max_blocks) {
  if (batch < 1 || max_blocks < 1 || block_size < 1) return fail(KVC_ERR_INVALID_ARG, "sizes must be >= 1");
  if (n_q_heads != kHeads || d_c != kDc || d_r != kW - kDc)
    return fail(KVC_ERR_UNSUPPORTED, "MLA decode supports n_q_heads 128, d_c 512, d_r 64 (got %d, %d, %d)",
                n_q_heads, d_c, d_r);
  if (block_size % kBoxRows != 0 || block_size > 256)
    return fail(KVC_ERR_UNSUPPORTED, "MLA block_size must be a multiple of 16 up to 256 (got %d)", block_size);
  if (batch > kMaxBatch) return fail(KVC_ERR_UNSUPPORTED, "MLA batch %d > %d", batch, kMaxBatch);
  return KVC_OK;
}

}  // namespace mla
}  // namespace kvc

extern "C" {

kvc_status kvc_decode_mla_workspace_size(int batch, int n_q_heads, int d_c, int d_r, int block_size,
                                         int max_blocks_per_seq, size_t* bytes) {
  using namespace kvc;
  clear_error();
  if (bytes == nullptr) return fail(KVC_ERR_INVALID_ARG, "bytes is NULL");
  kvc_status s = mla::check(batch, n_q_heads, d_c, d_r, block_size, max_blocks_per_seq);
  if (s != KVC_OK) return s;
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != KVC_OK) return s;
  const int G2 = mla::plan_pairs(dev, batch, max_blocks_per_seq, block_size);
  *bytes = mla::list_bytes(batch, G2) + static_cast<size_t>(G2) * mla::record_bytes_per_pair();
  return KVC_OK;
}

kvc_status kvc_decode_attention_mla(const void* q_absorbed, const void* latent_cache, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens, int batch, float scale,
                                    int n_q_heads, int d_c, int d_r, int block_size, int64_t num_blocks,
                                    kvc_dtype dtype, void* out, kvc_dtype out_dtype, void* workspace,
                                    size_t workspace_bytes, kvc_stream stream) {
  using namespace kvc;
  clear_error();
  kvc_status s = mla::check(batch, n_q_heads, d_c, d_r, block_size, max_blocks_per_seq);
  if (s != KVC_OK) return s;
  if (dtype != KVC_BF16) return fail(KVC_ERR_UNSUPPORTED, "MLA decode reads bf16 caches only");
  if (!dtype_ok(out_dtype)) return fail(KVC_ERR_INVALID_ARG, "unknown out dtype");
  if (num_blocks < 1) return fail(KVC_ERR_INVALID_ARG, "num_blocks must be >= 1");
  if (num_blocks * block_size > (1ll << 31) - 1) return fail(KVC_ERR_UNSUPPORTED, "latent pool too large");
  if (q_absorbed == nullptr || latent_cache == nullptr || block_tables == nullptr || context_lens == nullptr ||
      out == nullptr)
    return fail(KVC_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(q_absorbed) || !aligned16(latent_cache)) return fail(KVC_ERR_INVALID_ARG, "16-byte alignment");
  if (!std::isfinite(scale)) return fail(KVC_ERR_INVALID_ARG, "scale must be finite");
  if (workspace_bytes > 0 && workspace == nullptr) return fail(KVC_ERR_INVALID_ARG, "workspace is NULL");
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(KVC_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != KVC_OK) return s;
  const uint32_t smem = mla::smem_bytes(batch);
  if (smem > static_cast<uint32_t>(dev->max_smem_optin))
    return fail(KVC_ERR_UNSUPPORTED, "MLA kernel needs %u bytes of shared memory (device max %d)", smem,
                dev->max_smem_optin);
  auto encode = mla::encode_fn();
  if (encode == nullptr) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");

  CUtensorMap tq, tc;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(mla::kW), static_cast<cuuint64_t>(mla::kHeads),
                                static_cast<cuuint64_t>(batch)};
    const cuuint64_t strides[2] = {mla::kW * 2ull, static_cast<cuuint64_t>(mla::kW) * 2 * mla::kHeads};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(mla::kHeads), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q_absorbed), dims, strides, box,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "tensor map for q_absorbed: CUresult %d", static_cast<int>(r));
  }
  {
    // the latent pool as [num_blocks * block_size rows, 576] in boxes of 16
    // rows x 64 columns (measured faster than 32- or 48-row boxes where a
    // tile lies in one block: 248 against 276 us on the DeepSeek-V2 batch)
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(mla::kW), static_cast<cuuint64_t>(num_blocks * block_size)};
    const cuuint64_t strides[1] = {mla::kW * 2ull};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(mla::kBoxRows)};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = encode(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(latent_cache), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "tensor map for latent_cache: CUresult %d", static_cast<int>(r));
  }

  mla::Params p{};
  p.q = static_cast<const __nv_bfloat16*>(q_absorbed);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.err = dev->error_word;
  p.num_blocks = num_blocks;
  p.batch = batch;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = block_size;
  p.out_dtype = static_cast<int>(out_dtype);
  p.qscale = scale * 1.4426950408889634f;
  int G2 = mla::plan_pairs(dev, batch, max_blocks_per_seq, block_size);
  const size_t cb = mla::list_bytes(batch, G2);
  const int64_t fit = workspace_bytes > cb ? static_cast<int64_t>((workspace_bytes - cb) / mla::record_bytes_per_pair()) : 0;
  if (fit >= 1) {
    p.list_cap = G2;
    G2 = static_cast<int>(std::min<int64_t>(G2, fit));
    p.unit_mode = 0;
    p.unit_lists = static_cast<int*>(workspace);
    p.rec_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + cb);
    p.rec_ml = p.rec_o + static_cast<size_t>(G2) * 2 * 2 * mla::kHeads * mla::kHalf;
    p.rec_slots = static_cast<int64_t>(G2) * 4;
  } else {
    p.unit_mode = 1;
    G2 = batch;
  }
  cudaError_t e = cudaFuncSetAttribute(mla::mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(mla)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // may start while the append of this step still runs (it waits before reading the cache)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * G2);
  cfg.blockDim = dim3(mla::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mla::mla_decode_kernel, tq, tc, p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(mla)");
  if (!p.unit_mode) {
    // the merge of split sequences, right behind (it waits for the decode grid)
    cudaLaunchConfig_t mcfg = {};
    mcfg.gridDim = dim3(static_cast<unsigned int>(batch) * 2 * mla::kMergeGroups);
    mcfg.blockDim = dim3(128);
    mcfg.stream = st;
    mcfg.attrs = attr;
    mcfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&mcfg, mla::mla_merge_kernel, p);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(mla merge)");
  }
  return finish_call(st);
}

}  // extern "C"
