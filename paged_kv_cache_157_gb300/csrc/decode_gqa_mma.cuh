// Paged decode attention for MHA / GQA / MQA with the two products of each
// 16-row tile on warp-level MMAs (bf16 or f16 caches, head_dim 128).
//
// What is computed is the paged decode of knowledge point 2 of "KV缓存原理与
// 显存估算" with the head grouping of "KV-Cache——为什么AI回复越来越快"
// section 03: every query head attends its kv head's rows gathered through the
// block table ("KV Cache（键值缓存）" section 2.3), softmax(scale * q . k)
// weighting v, in fp32.
//
// Why MMAs for a bandwidth-bound product: on CUDA cores every cached element
// costs a conversion and a share of an FMA per query, ~650 warp instructions
// per 16 rows of one kv head, and two 4-warp CTAs per SM could not issue them
// fast enough to keep HBM busy. As m16n8k16 MMAs the same tile is 8 matrix
// loads + 8 MMAs for the scores and 8 transposing loads + 16 MMAs for the
// output (~100 instructions), so one CTA per SM keeps a deep ring of copies in
// flight and every SM streams at the same rate.
//
// Per warp and tile (16 rows of one kv head, up to 8 of its query heads):
//   S^T [16 rows x 8 queries]  = K [16 x 128] . Q^T [128 x 8]     (8 k-steps)
//   O^T [128 dims x 8 queries] += V^T [128 x 16 rows] . P^T [16 x 8]
// Q^T stays in registers for a whole segment; the accumulators are fp32; P is
// split into hi + lo parts of the cache's 16-bit type (two PV products) so the
// weights keep ~2^-17 relative accuracy. The scores' C fragment becomes the B
// fragment of P^T by one 8x8 transpose (movmatrix) per half. Softmax runs in
// the log2 domain with a lazy rescale (the reference maximum only moves when a
// score exceeds it by more than 8, a factor 256).
//
// Pages reach shared memory by TMA tensor copies (a 2-D map over the pool as
// [num_blocks * n_kv_heads * block_size rows, 128]) in [hc * block_size rows x
// 64 dims] boxes with the 128-byte swizzle, so every 8x8 matrix load touches
// eight different bank groups. Work split, split-K records, the last-arriver
// merge and the bounded waits are those of the CUDA-core kernel.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "decode_gqa_impl.cuh"

namespace kvc {
namespace wmma16 {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// d += a . b for one m16n8k16 tile, fp32 accumulate; BF: bf16 operands, else f16.
template <bool BF>
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BF) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Transpose of an 8x8 matrix of 16-bit elements held in the standard
// fragment layout (lane 4g + c holds row g, columns 2c and 2c + 1).
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Two fp32 values rounded (nearest even) to the 16-bit type, `lo` in the low half.
template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (BF)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool BF>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
}

__device__ __forceinline__ void tma2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Byte offset of 16-byte chunk q (0..7) of row r in a box of 128-byte rows
// written by TMA with the 128-byte swizzle (box base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int r, int q) {
  return static_cast<uint32_t>(r * 128 + ((q ^ (r & 7)) << 4));
}

}  // namespace wmma16

// Per-warp state of a segment. Lane 4g + c holds, for query heads 2c and
// 2c + 1 of the warp (n-columns of the MMAs), the output dims 16i + g and
// 16i + g + 8 of every 16-dim tile i.
struct MmaWarpState {
  uint32_t qb[8][2];  // Q^T B fragments per k-step (query g, dims 16ks + 2c (+1) and + 8)
  float o[8][4];      // O^T C fragments: (dim 16i+g, q 2c), (16i+g, 2c+1), (16i+g+8, 2c), (16i+g+8, 2c+1)
  float m[2];         // reference maxima (log2 units) of queries 2c, 2c+1; equal over g
  float l[2];         // this lane's partial sums of the weights of queries 2c, 2c+1
};

// One 16-row tile of one kv head for the warp's GW query heads. kb / vb: the
// stage's K / V box (64-dim half 0; half 1 follows at + box_bytes); row0: the
// tile's first row in the box. PARTIAL tiles attend only rows [lo_valid,
// valid) and query column q only rows below vis[q & 1] of its lane.
template <bool BF, int GW, bool PARTIAL>
__device__ __forceinline__ void mma_tile(uint32_t kb, uint32_t vb, uint32_t box_bytes, int row0, int lo_valid,
                                         int valid, int vis0, int vis1, float qscale, MmaWarpState& st, int lane) {
  using namespace wmma16;
  const int g = lane >> 2, c = lane & 3;
  // ---- S^T = K . Q^T: lane l addresses row (l & 7) + 8 ((l >> 3) & 1) of
  // the tile in dims chunk 2 (ks & 3) + (l >> 4) of half ks >> 2.
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t rowk = kb + static_cast<uint32_t>(r * 128);
    const int sw = r & 7;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int q = ((ks & 3) << 1) + (lane >> 4);
      uint32_t a[4];
      ldsm_x4(rowk + (ks >> 2) * box_bytes + static_cast<uint32_t>((q ^ sw) << 4), a);
      if (ks & 1)
        mma<BF>(sb, a, st.qb[ks][0], st.qb[ks][1]);
      else
        mma<BF>(sa, a, st.qb[ks][0], st.qb[ks][1]);
    }
  }
  // scores in log2 units: x0 (row g, q 2c), x1 (row g, q 2c+1), x2 (row g+8, q 2c), x3 (row g+8, q 2c+1)
  float x[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = (sa[e] + sb[e]) * qscale;
  const bool q0 = 2 * c < GW, q1 = 2 * c + 1 < GW;
  if (!q0) {
    x[0] = kNegInf;
    x[2] = kNegInf;
  }
  if (!q1) {
    x[1] = kNegInf;
    x[3] = kNegInf;
  }
  if (PARTIAL) {
    const bool ra = g >= lo_valid, rb = g + 8 >= lo_valid;
    if (!ra || g >= vis0) x[0] = kNegInf;
    if (!ra || g >= vis1) x[1] = kNegInf;
    if (!rb || g + 8 >= vis0) x[2] = kNegInf;
    if (!rb || g + 8 >= vis1) x[3] = kNegInf;
  }
  // ---- online softmax (lazy rescale)
  const bool need = x[0] > st.m[0] + 8.0f || x[2] > st.m[0] + 8.0f || x[1] > st.m[1] + 8.0f || x[3] > st.m[1] + 8.0f;
  if (__any_sync(0xffffffffu, need)) {
    float t0 = fmaxf(x[0], x[2]), t1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int msk = 4; msk < 32; msk <<= 1) {
      t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, msk));
      t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, msk));
    }
    const float n0 = fmaxf(st.m[0], t0), n1 = fmaxf(st.m[1], t1);
    const float a0 = fast_exp2(st.m[0] - n0), a1 = fast_exp2(st.m[1] - n1);
    const float2 a2 = make_float2(a0, a1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 u = fmul2(make_float2(st.o[i][0], st.o[i][1]), a2);
      const float2 v = fmul2(make_float2(st.o[i][2], st.o[i][3]), a2);
      st.o[i][0] = u.x;
      st.o[i][1] = u.y;
      st.o[i][2] = v.x;
      st.o[i][3] = v.y;
    }
    st.l[0] *= a0;
    st.l[1] *= a1;
    st.m[0] = n0;
    st.m[1] = n1;
  }
  const float p0 = fast_exp2(x[0] - st.m[0]), p1 = fast_exp2(x[1] - st.m[1]);
  const float p2 = fast_exp2(x[2] - st.m[0]), p3 = fast_exp2(x[3] - st.m[1]);
  st.l[0] += p0 + p2;
  st.l[1] += p1 + p3;
  // ---- P^T as hi + lo parts: the C fragment [rows][queries] of each 8-row
  // half is one 8x8 matrix; its transpose is the B fragment [rows = k][queries = n].
  const uint32_t h01 = pack2<BF>(p0, p1), h23 = pack2<BF>(p2, p3);
  const float2 f01 = unpack2<BF>(h01), f23 = unpack2<BF>(h23);
  const uint32_t l01 = pack2<BF>(p0 - f01.x, p1 - f01.y), l23 = pack2<BF>(p2 - f23.x, p3 - f23.y);
  const uint32_t bh0 = movm_t(h01), bh1 = movm_t(h23), bl0 = movm_t(l01), bl1 = movm_t(l23);
  // ---- O^T += V^T . P^T: lane l addresses row (l & 7) + 8 (l >> 4) of the
  // tile in dims chunk 2i + ((l >> 3) & 1); the transposing load gives lane
  // 4g + c the rows 2c, 2c + 1 (+ 8) of dims 16i + g (+ 8).
  uint32_t keep01 = 0xffffffffu, keep89 = 0xffffffffu;
  if (PARTIAL) {
    // rows outside [lo_valid, valid) may hold anything (even NaN): their weight
    // is 0, but 0 x NaN is NaN, so their values are cleared
    const int ra = 2 * c, rb = 2 * c + 8;
    keep01 = ((ra >= lo_valid && ra < valid) ? 0x0000ffffu : 0u) | ((ra + 1 >= lo_valid && ra + 1 < valid) ? 0xffff0000u : 0u);
    keep89 = ((rb >= lo_valid && rb < valid) ? 0x0000ffffu : 0u) | ((rb + 1 >= lo_valid && rb + 1 < valid) ? 0xffff0000u : 0u);
  }
  {
    const int r = row0 + (lane & 7) + (lane >> 4) * 8;
    const uint32_t rowv = vb + static_cast<uint32_t>(r * 128);
    const int sw = r & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int chunk = 2 * i + ((lane >> 3) & 1);
      uint32_t a[4];
      ldsm_x4_t(rowv + (chunk >> 3) * box_bytes + static_cast<uint32_t>(((chunk & 7) ^ sw) << 4), a);
      if (PARTIAL) {
        a[0] &= keep01;
        a[1] &= keep01;
        a[2] &= keep89;
        a[3] &= keep89;
      }
      mma<BF>(st.o[i], a, bh0, bh1);
      mma<BF>(st.o[i], a, bl0, bl1);
    }
  }
}

// Shared-memory carve-up of the MMA kernel (offsets from a 1024-byte aligned
// base; the host adds 1024 bytes of slack for the alignment). A stage is
// [K half 0][K half 1][V half 0][V half 1] (each hc * block_size rows of 128
// bytes, swizzled) followed by the unit's query rows [hc][GH][128].
struct GqaMmaSmem {
  size_t box_bytes, stage_bytes, q_off, bar_off, rel_off, misc_off, scan_off, total;
};

__host__ __device__ inline GqaMmaSmem gqa_mma_smem_layout(int q_elt, int GH, int block_size, int hc, int stages,
                                                          int batch) {
  GqaMmaSmem s;
  s.box_bytes = static_cast<size_t>(hc) * block_size * 128;
  s.q_off = 4 * s.box_bytes;
  s.stage_bytes = align_up(s.q_off + static_cast<size_t>(hc) * GH * 128 * q_elt, 1024);
  s.bar_off = static_cast<size_t>(stages) * s.stage_bytes;
  s.rel_off = s.bar_off + static_cast<size_t>(stages) * 8;
  s.misc_off = align_up(s.rel_off + static_cast<size_t>(stages) * 8, 16);
  s.scan_off = s.misc_off + 16;
  s.total = s.scan_off + static_cast<size_t>(batch + 1 + 32) * 4 + 1024;
  return s;
}

__host__ __device__ constexpr int mma_warps_per_kvhead(int GH) { return GH > 8 ? GH / 8 : 1; }
__host__ __device__ constexpr int mma_max_chunk(int GH) { return kGqaWarps / mma_warps_per_kvhead(GH); }

template <typename T, int GH, bool EXT>
__global__ void __launch_bounds__(kGqaWarps * 32, 1)
    gqa_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const GqaParams p) {
  using namespace wmma16;
  constexpr int D = 128;
  constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
  constexpr int HW = mma_warps_per_kvhead(GH);  // warps per kv head
  constexpr int GW = GH / HW;                   // query heads per warp (MMA columns)
  constexpr int HCM = kGqaWarps / HW;           // kv heads per CTA at most
  constexpr int HS = HCM * GH;                  // query heads per record
  static_assert(GW <= 8 && GW * HW == GH, "at most 8 query heads per warp");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw_addr);
  const int hc = p.hc;
  const int wnd = EXT ? p.window : 0;
  const int n_tok = EXT ? p.n_tok : 1;
  const bool causal = !EXT || p.causal != 0;
  const int tm = causal ? n_tok - 1 : 0;
  const int min_len = causal ? n_tok : 1;
  const bool multi = EXT && n_tok > 1;
  const int32_t* row_start = EXT ? p.row_start : nullptr;
  const int row_div = EXT ? p.row_div : 0;
  const int bs = p.block_size, S = p.stages;
  const GqaMmaSmem L = gqa_mma_smem_layout(sizeof(T), GH, bs, hc, S, p.batch);
  uint64_t* fbar = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  unsigned int* s_rel = reinterpret_cast<unsigned int*>(smem + L.rel_off);
  unsigned int* s_iss = s_rel + S;
  volatile int* s_misc = reinterpret_cast<volatile int*>(smem + L.misc_off);
  int* s_scan = reinterpret_cast<int*>(smem + L.scan_off);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int kh = w / HW, hw = w % HW;
  const int nact = hc * HW;
  const bool active = w < nact;
  const int B = p.batch;
  const int tiles_per_page = bs / 16;
  const uint32_t box_bytes = static_cast<uint32_t>(L.box_bytes);
  const uint32_t q_bytes = static_cast<uint32_t>(hc * GH * D * sizeof(T));
  const T* qg = static_cast<const T*>(p.q);
  const uint32_t full = 0xffffffffu;
  const int HN = p.n_chunks * p.n_hsub;
  const bool q_contig = (GH == p.group);

  if (tid < S) {
    mbar_init(fbar + tid, 1);
    s_rel[tid] = 0u;
    s_iss[tid] = 0u;
  }
  if (tid == 0) {
    s_misc[0] = 0;
    s_misc[1] = 0;
    s_misc[2] = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  fence_barrier_init();
  // Launched right behind the previous kernel of the stream (programmatic
  // stream serialisation), the kernel sets up its barriers while that grid
  // runs; every thread then waits for it (its writes become visible) before it
  // reads or writes any caller buffer.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  scan_blocks(p.context_lens, B, bs, p.max_blocks, wnd, min_len, row_start, row_div, s_scan);  // ends with a CTA barrier
  const int64_t N = static_cast<int64_t>(HN) * s_scan[B];
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;

  if (blockIdx.x == 0) {
    int empty = 0;
    for (int b = tid; b < B; b += blockDim.x) {
      const int n = __ldg(p.context_lens + b);
      if (n < min_len || n > bs * p.max_blocks) set_flag(p.err, 0x2u);
      if (row_div > 0 && __ldg(row_start + b / row_div) > n) set_flag(p.err, 0x2u);
      empty |= (s_scan[b + 1] == s_scan[b]) ? 1 : 0;
    }
    if (__syncthreads_or(empty) && !p.unit_mode) {
      const int rows = n_tok * p.n_q_heads * D;
      for (int b = 0; b < B; ++b) {
        if (s_scan[b + 1] != s_scan[b]) continue;
        for (int idx = tid; idx < rows; idx += blockDim.x)
          store_out(p.out, static_cast<int64_t>(b) * rows + idx, 0.f, p.out_dtype);
        if (EXT && p.lse != nullptr)
          for (int idx = tid; idx < n_tok * p.n_q_heads; idx += blockDim.x)
            p.lse[static_cast<int64_t>(b) * n_tok * p.n_q_heads + idx] = kNegInf;
      }
    }
  }

  int64_t lo, hi;
  if (p.unit_mode) {
    const int seq = static_cast<int>(c / HN);
    const int idx = static_cast<int>(c - static_cast<int64_t>(seq) * HN);
    const int nb = s_scan[seq + 1] - s_scan[seq];
    if (nb == 0) {
      if (active) {
        const int chunk = idx / p.n_hsub, hsub = idx - chunk * p.n_hsub;
        const int kvh = chunk * hc + kh, v0 = hsub * GH + hw * GW;
        for (int i = lane; i < GW * D; i += 32) {
          const int64_t o = EXT ? out_row(p, seq, kvh, v0 + i / D) * D + i % D
                                : (static_cast<int64_t>(seq) * p.n_q_heads + kvh * p.group + v0) * D + i;
          store_out(p.out, o, 0.f, p.out_dtype);
        }
        if (EXT && p.lse != nullptr && lane < GW) p.lse[out_row(p, seq, kvh, v0 + lane)] = kNegInf;
      }
      return;
    }
    lo = static_cast<int64_t>(HN) * s_scan[seq] + static_cast<int64_t>(idx) * nb;
    hi = lo + nb;
  } else {
    lo = cta_range_start(c, G, N);
    hi = cta_range_start(c + 1, G, N);
  }
  const int total = static_cast<int>(hi - lo);
  if (total <= 0) return;  // uniform over the CTA

  const uint64_t pol = policy_evict_first();
  const uint32_t stage0 = base;  // stage s at base + s * stage_bytes
  const uint32_t stage_bytes = static_cast<uint32_t>(L.stage_bytes);

  // Positions lo + 32*win + lane, one per lane: the first row of the chunk's
  // pages in the pool viewed as rows ((block * n_kv_heads + first kv head of
  // the chunk) * block_size; -1 if the table entry is out of range) and, for
  // the first block of a segment, the element offset of the unit's first
  // query row (with several new tokens: the unit's index; -1 otherwise).
  auto window = [&](int win, int& src, int& qoff) {
    const int64_t pos = lo + static_cast<int64_t>(win) * 32 + lane;
    src = -1;
    qoff = -1;
    if (pos < hi) {
      const BlockPos bp = locate_block(pos, HN, s_scan, B, p.n_hsub);
      const int j0 =
          start_row(seq_rows(p.context_lens, bp.seq, bs, p.max_blocks, min_len), wnd, row_start, row_div, bp.seq) /
          bs;
      const int phys = __ldg(p.block_tables + static_cast<int64_t>(bp.seq) * p.max_blocks + j0 + bp.j);
      if (phys >= 0 && phys < p.num_blocks) src = (phys * p.n_kv_heads + bp.chunk * hc) * bs;
      if (pos == lo || bp.j == 0)
        qoff = multi ? (bp.seq * p.n_chunks + bp.chunk) * p.n_hsub + bp.hsub
                     : (bp.seq * p.n_q_heads + bp.chunk * hc * p.group + bp.hsub * GH) * D;
    }
  };
  auto issue = [&](int slot, int src, int qoff) {
    const uint32_t bytes = (src >= 0 ? 4 * box_bytes : 0u) + (qoff >= 0 ? q_bytes : 0u);
    if (src < 0) set_flag(p.err, 0x1u);
    atomicAdd(s_iss + slot, 1u);
    if (bytes == 0) {
      mbar_arrive(fbar + slot);
      return;
    }
    const uint32_t dst = stage0 + static_cast<uint32_t>(slot) * stage_bytes;
    const uint32_t bar = smem_addr(fbar + slot);
    mbar_arrive_expect_tx(fbar + slot, bytes);
    if (src >= 0) {
      tma2d(dst, &tm_k, 0, src, bar, pol);
      tma2d(dst + box_bytes, &tm_k, 64, src, bar, pol);
      tma2d(dst + 2 * box_bytes, &tm_v, 0, src, bar, pol);
      tma2d(dst + 3 * box_bytes, &tm_v, 64, src, bar, pol);
    }
    if (qoff >= 0) {
      unsigned char* qdst = smem + static_cast<size_t>(slot) * stage_bytes + L.q_off;
      if (multi) {
        const int hs = qoff % p.n_hsub, rest = qoff / p.n_hsub;
        const int ch = rest % p.n_chunks, sq = rest / p.n_chunks;
        const uint32_t rowb = static_cast<uint32_t>(D * sizeof(T));
        for (int h = 0; h < hc; ++h) {
          const int kvh = ch * hc + h;
          for (int v = hs * GH, ve = v + GH; v < ve;) {
            const int t = v / p.group, j = v - t * p.group;
            const int len = min(p.group - j, ve - v);
            const int64_t row = (static_cast<int64_t>(sq) * n_tok + t) * p.n_q_heads + kvh * p.group + j;
            bulk_g2s(qdst + (h * GH + v - hs * GH) * rowb, qg + row * D, len * rowb, fbar + slot, pol);
            v += len;
          }
        }
      } else if (q_contig) {
        bulk_g2s(qdst, qg + qoff, q_bytes, fbar + slot, pol);
      } else {
        const uint32_t rb = static_cast<uint32_t>(GH * D * sizeof(T));
        for (int h = 0; h < hc; ++h) bulk_g2s(qdst + h * rb, qg + qoff + h * p.group * D, rb, fbar + slot, pol);
      }
    }
  };

  int w_src0, w_src1 = -1, w_q0, w_q1 = -1;
  window(0, w_src0, w_q0);
  if (total > 32) window(1, w_src1, w_q1);

  const int n_first = total < S ? total : S;
  if (w == 0) {
    for (int i = 0; i < n_first; ++i) {
      const int src = __shfl_sync(full, w_src0, i);
      const int qo = __shfl_sync(full, w_q0, i);
      if (lane == 0) issue(i, src, qo);
    }
  }
  __syncwarp();

  bool pend0 = false, pend1 = false;
  unsigned int old0 = 0, old1 = 0;
  bool aborted = false;
  const int g8 = lane >> 2, c4 = lane & 3;

  if (active) {
    int slot = 0;
    uint32_t par = 0, fill = 0;
    int cpos = 0;
    int64_t gb = lo;
    while (gb < hi) {
      const BlockPos sg = locate_block(gb, HN, s_scan, B, p.n_hsub);
      const int seg_len = static_cast<int>(((sg.nb - sg.j) < (hi - gb)) ? (sg.nb - sg.j) : (hi - gb));
      const int n_rows = seq_rows(p.context_lens, sg.seq, bs, p.max_blocks, min_len);
      const int r0 = start_row(n_rows, wnd, row_start, row_div, sg.seq);
      const int j0 = r0 / bs;
      const int kvh = sg.chunk * hc + kh;
      const int v0 = sg.hsub * GH + hw * GW;
      const int hq0 = kvh * p.group + v0;
      // rows at the end each of the lane's two query columns may not see (multi-token causality)
      const int dh0 = (EXT && causal) ? tm - (v0 + 2 * c4) / p.group : 0;
      const int dh1 = (EXT && causal) ? tm - (v0 + 2 * c4 + 1) / p.group : 0;

      MmaWarpState st;
      for (int t = 0; t < seg_len; ++t, ++cpos) {
        if (cpos > 0 && (cpos & 31) == 0) {
          w_src0 = w_src1;
          w_q0 = w_q1;
          w_src1 = -1;
          w_q1 = -1;
          if (cpos + 32 < total) window((cpos >> 5) + 1, w_src1, w_q1);
        }
        const int src = __shfl_sync(full, w_src0, cpos & 31);
        const int cn = cpos + S;
        const bool in_cur = (cn >> 5) == (cpos >> 5);
        const int src_n = __shfl_sync(full, in_cur ? w_src0 : w_src1, cn & 31);
        const int q_n = __shfl_sync(full, in_cur ? w_q0 : w_q1, cn & 31);
        const bool ok = mbar_wait_bounded(fbar + slot, par);
        if (__any_sync(full, !ok) || s_misc[0]) {
          if (lane == 0) {
            set_flag(p.err, 0x8u);
            s_misc[0] = 1;
          }
          aborted = true;
          break;
        }
        const uint32_t stg = stage0 + static_cast<uint32_t>(slot) * stage_bytes;
        if (t == 0) {
          // Q^T fragments of the warp's query heads (query g of the warp, dims
          // 16 ks + 2c (+1) and + 8 (+9)); columns beyond GW are zero.
          const unsigned char* qs = smem + static_cast<size_t>(slot) * stage_bytes + L.q_off +
                                    static_cast<size_t>(kh * GH + hw * GW) * D * sizeof(T);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            if (g8 < GW) {
              const uint32_t* qr = reinterpret_cast<const uint32_t*>(qs + (g8 * D + 16 * ks + 2 * c4) * sizeof(T));
              st.qb[ks][0] = qr[0];
              st.qb[ks][1] = qr[4];
            } else {
              st.qb[ks][0] = 0u;
              st.qb[ks][1] = 0u;
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int e = 0; e < 4; ++e) st.o[i][e] = 0.f;
          }
          // a finite start: a column that meets only masked rows keeps weight 0
          st.m[0] = st.m[1] = -1e30f;
          st.l[0] = st.l[1] = 0.f;
        }
        if (src >= 0) {
          const uint32_t kb = stg, vb = stg + 2 * box_bytes;
          const int jb = j0 + sg.j + t;
          const int rb = n_rows - jb * bs;
          const int vr = min(bs, rb);
          const int lr = (jb == j0) ? r0 - j0 * bs : 0;
          const int rowk = kh * bs;
          if (rb - tm >= bs && lr == 0) {
            for (int tt = 0; tt < tiles_per_page; ++tt)
              mma_tile<BF, GW, false>(kb, vb, box_bytes, rowk + tt * 16, 0, 16, 16, 16, p.qscale, st, lane);
          } else {
            for (int tt = 0; tt < tiles_per_page; ++tt) {
              const int valid = vr - tt * 16, lo_valid = lr - tt * 16;
              const int rt = rb - tt * 16;
              if (valid <= 0) break;
              if (lo_valid >= 16) continue;
              if (rt - tm >= 16 && lo_valid <= 0)
                mma_tile<BF, GW, false>(kb, vb, box_bytes, rowk + tt * 16, 0, 16, 16, 16, p.qscale, st, lane);
              else
                mma_tile<BF, GW, true>(kb, vb, box_bytes, rowk + tt * 16, lo_valid, valid,
                                       EXT ? min(valid, rt - dh0) : valid, EXT ? min(valid, rt - dh1) : valid,
                                       p.qscale, st, lane);
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          const unsigned int old = atomic_add_acq_rel_cta_smem(s_rel + slot, 1u);
          if (old + 1 == static_cast<unsigned int>(nact) * (fill + 1) && cn < total) issue(slot, src_n, q_n);
        }
        __syncwarp();
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
          ++fill;
        }
      }
      if (aborted) break;

      // ---- finish the segment
      float lw0 = st.l[0], lw1 = st.l[1];
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1) {
        lw0 += __shfl_xor_sync(full, lw0, msk);
        lw1 += __shfl_xor_sync(full, lw1, msk);
      }
      const bool qv0 = 2 * c4 < GW, qv1 = 2 * c4 + 1 < GW;
      const bool whole = (sg.j == 0 && seg_len == sg.nb);
      if (whole) {
        const float i0 = 1.0f / lw0, i1 = 1.0f / lw1;
        const int64_t ob0 = (EXT ? out_row(p, sg.seq, kvh, v0 + 2 * c4)
                                 : static_cast<int64_t>(sg.seq) * p.n_q_heads + hq0 + 2 * c4) * D;
        const int64_t ob1 = (EXT ? out_row(p, sg.seq, kvh, v0 + 2 * c4 + 1) : ob0 / D + 1) * D;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d0 = 16 * i + g8;
          if (qv0) {
            store_out(p.out, ob0 + d0, st.o[i][0] * i0, p.out_dtype);
            store_out(p.out, ob0 + d0 + 8, st.o[i][2] * i0, p.out_dtype);
          }
          if (qv1) {
            store_out(p.out, ob1 + d0, st.o[i][1] * i1, p.out_dtype);
            store_out(p.out, ob1 + d0 + 8, st.o[i][3] * i1, p.out_dtype);
          }
        }
        if (EXT && p.lse != nullptr && g8 == 0) {
          if (qv0) p.lse[out_row(p, sg.seq, kvh, v0 + 2 * c4)] = st.m[0] + __log2f(lw0);
          if (qv1) p.lse[out_row(p, sg.seq, kvh, v0 + 2 * c4 + 1)] = st.m[1] + __log2f(lw1);
        }
      } else {
        const int64_t rec = c * 2 + (gb == lo ? 0 : 1);
        const int hr = kh * GH + hw * GW;
        float* ro0 = p.rec_o + (rec * HS + hr + 2 * c4) * D;
        float* ro1 = ro0 + D;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d0 = 16 * i + g8;
          if (qv0) {
            ro0[d0] = st.o[i][0];
            ro0[d0 + 8] = st.o[i][2];
          }
          if (qv1) {
            ro1[d0] = st.o[i][1];
            ro1[d0 + 8] = st.o[i][3];
          }
        }
        if (g8 == 0) {
          if (qv0) {
            p.rec_ml[(rec * HS + hr + 2 * c4) * 2] = st.m[0];
            p.rec_ml[(rec * HS + hr + 2 * c4) * 2 + 1] = lw0;
          }
          if (qv1) {
            p.rec_ml[(rec * HS + hr + 2 * c4 + 1) * 2] = st.m[1];
            p.rec_ml[(rec * HS + hr + 2 * c4 + 1) * 2 + 1] = lw1;
          }
        }
        __syncwarp();
        if (lane == 0) {
          const int64_t unit = (static_cast<int64_t>(sg.seq) * p.n_chunks + sg.chunk) * p.n_hsub + sg.hsub;
          const unsigned int old = atomic_add_acq_rel_gpu(p.counters + unit * nact + w, 1u);
          if (gb == lo) old0 = old; else old1 = old;
        }
        if (gb == lo) pend0 = true; else pend1 = true;
      }
      gb += seg_len;
    }
  }

  __syncthreads();
  const bool any_abort = s_misc[0] != 0;
  if (active && !any_abort && (pend0 || pend1)) {
    const BlockPos q0 = locate_block(lo, HN, s_scan, B, p.n_hsub);
    const BlockPos q1 = locate_block(hi - 1, HN, s_scan, B, p.n_hsub);
    const int64_t p0_u0 = lo - q0.j, p1_u0 = hi - 1 - q1.j;
    int last = 0;
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (!(k == 0 ? pend0 : pend1)) continue;
        const BlockPos& qq = k == 0 ? q0 : q1;
        const int64_t u0 = k == 0 ? p0_u0 : p1_u0;
        const int64_t c0 = worker_of_block(u0, G, N), c1 = worker_of_block(u0 + qq.nb - 1, G, N);
        int64_t contributors = c1 - c0 + 1;
        if (N < G) {
          contributors = 0;
          for (int64_t x = c0; x <= c1; ++x)
            contributors += (worker_range_start(x, G, N) != worker_range_start(x + 1, G, N)) ? 1 : 0;
        }
        const int64_t unit = (static_cast<int64_t>(qq.seq) * p.n_chunks + qq.chunk) * p.n_hsub + qq.hsub;
        unsigned int* ctr = p.counters + unit * nact + w;
        const unsigned int old = k == 0 ? old0 : old1;
        if (old + 1 == static_cast<unsigned int>(contributors)) {
          last |= 1 << k;
          *ctr = 0u;
        } else if (old + 1 > static_cast<unsigned int>(contributors)) {
          set_flag(p.err, 0x10u);
          atomicExch(ctr, 0u);
        }
      }
    }
    last = __shfl_sync(full, last, 0);
    if (last & 1)
      merge_unit_warp<D, HS, GW, EXT>(p, p0_u0, q0.nb, G, N, q0.seq, q0.chunk * hc + kh, q0.hsub * GH + hw * GW,
                                      kh * GH + hw * GW, lane);
    if (last & 2)
      merge_unit_warp<D, HS, GW, EXT>(p, p1_u0, q1.nb, G, N, q1.seq, q1.chunk * hc + kh, q1.hsub * GH + hw * GW,
                                      kh * GH + hw * GW, lane);
  }
  if (any_abort && tid == 0) {
    for (int x = 0; x < S; ++x) {
      const unsigned int n = s_iss[x];
      if (n > 0) (void)mbar_wait_bounded(fbar + x, (n - 1) & 1u);
    }
  }
}

}  // namespace kvc
