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
// eight different bank groups. Positions are split over the CTAs in static
// ranges (optionally with claimed chunks at every unit's tail); segments that
// cover part of a unit leave fp32 records, which a merge kernel launched
// behind this one combines, all units in parallel. Every wait is bounded.
//
// One-byte caches (e4m3 or int8 codes with per-channel K scales and per-token
// V scales, bf16 queries) use the same loop on f16 MMAs: every code is an f16
// value, so each lane converts the codes it needs straight into its MMA
// fragments (one conversion per pair of codes, no staging copy). The K scales
// are folded into the query (q * k_scale split into f16 hi + lo), the V
// scales into the weights; see mma_tile_q8.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "decode_gqa_impl.cuh"

namespace kvc {

#ifndef KVC_MMA_CTAS_PER_SM
#define KVC_MMA_CTAS_PER_SM 1
#endif
#ifndef KVC_MMA_WARPS
#define KVC_MMA_WARPS 8
#endif
// Resident CTAs per SM the register and shared-memory budgets aim at, and the
// consumer warps of a CTA (one kv head of the stage's block each).
constexpr int kMmaCtasPerSm = KVC_MMA_CTAS_PER_SM;
constexpr int kMmaWarps = KVC_MMA_WARPS;
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;  // consumer warps + one producer warp


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

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// The four one-byte codes of w as two f16 pairs: bytes 0, 1 into lo (byte 0
// in its low half), bytes 2, 3 into hi. Q8 = 1: e4m3 codes (hardware
// conversion, exact); Q8 = 2: int8 codes c, placed as c + 128 in the low
// mantissa byte of the f16 1024 (1024 + c + 128, exact) minus 1152.
template <int Q8>
__device__ __forceinline__ void codes_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (Q8 == 1) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  } else {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u), b = __byte_perm(u, 0x64646464u, 0x4342u);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
  }
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
// tile's first row in the box. The boxes are 1024-byte aligned and written by
// TMA with the 128-byte swizzle: 16-byte chunk q of row r sits at
// r * 128 + ((q ^ (r & 7)) << 4). PARTIAL tiles attend only rows [lo_valid,
// valid) and query column q only rows below vis[q & 1] of its lane.
template <bool BF, int GW, bool PARTIAL>
__device__ __forceinline__ void mma_tile(uint32_t kb, uint32_t vb, uint32_t box_bytes, int row0, int lo_valid,
                                         int valid, int vis0, int vis1, float qscale, MmaWarpState& st, int lane) {
  using namespace wmma16;
  const int g = lane >> 2, c = lane & 3;
  // Swizzled chunk offsets: row r of the tile sits at r * 128 and its 16-byte
  // chunk q at ((q ^ (r & 7)) << 4); every row a lane addresses has r & 7 =
  // lane & 7, so for q = 2k + h the offset is 32 (k ^ s2) + 16 ((h ^ sw) & 1).
  const int sw = lane & 7, s2 = sw >> 1;
  // ---- S^T = K . Q^T: lane l addresses row (l & 7) + 8 ((l >> 3) & 1) of
  // the tile in dims chunk 2 (ks & 3) + (l >> 4) of half ks >> 2; four
  // independent accumulator chains.
  float sc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[j][e] = 0.f;
  }
  {
    const uint32_t rowk = kb + static_cast<uint32_t>((row0 + (lane & 7) + ((lane >> 3) & 1) * 8) * 128) +
                          static_cast<uint32_t>((((lane >> 4) ^ sw) & 1) << 4);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[4];
      ldsm_x4(rowk + (ks >> 2) * box_bytes + static_cast<uint32_t>(((ks & 3) ^ s2) << 5), a);
      mma<BF>(sc[ks & 3], a, st.qb[ks][0], st.qb[ks][1]);
    }
  }
  // scores in log2 units: x0 (row g, q 2c), x1 (row g, q 2c+1), x2 (row g+8, q 2c), x3 (row g+8, q 2c+1)
  float x[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = ((sc[0][e] + sc[1][e]) + (sc[2][e] + sc[3][e])) * qscale;
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
    const uint32_t rowv = vb + static_cast<uint32_t>((row0 + (lane & 7) + (lane >> 4) * 8) * 128) +
                          static_cast<uint32_t>(((((lane >> 3) & 1) ^ sw) & 1) << 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t a[4];
      ldsm_x4_t(rowv + (i >> 2) * box_bytes + static_cast<uint32_t>(((i & 3) ^ s2) << 5), a);
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

// Per-warp state of a segment over a one-byte cache. As MmaWarpState, but the
// query is q * k_scale * 2^t in f16 hi + lo parts (t per segment and warp,
// so that the largest entry lies in [2^14, 2^15)), and the output dims of
// lane 4g + c in tile i are 16g + 2i (o[i][0], o[i][1]) and 16g + 2i + 1
// (o[i][2], o[i][3]).
struct Q8WarpState {
  uint32_t qh[8][2];  // B fragments per k-step: query g, dims 32c + 4ks + {0, 1} and + {2, 3}
  uint32_t ql[8][2];
  float o[8][4];
  float m[2];
  float l[2];
  float f;  // the weights' factor (a power of two); 0 before the segment's first tile
};

// One 16-row tile of one kv head over a one-byte cache. kb / vb: the stage's
// K / V code boxes (128 codes per 128-byte row, 1024-byte aligned, 128-byte
// swizzle: 16-byte chunk q of row r at r * 128 + ((q ^ (r & 7)) << 4)); row0:
// the tile's first row (a multiple of 16); vsp: the V scales of the box's rows.
//
// The order of the dims inside a product is free (Q uses the same order), so
// each lane takes whole 16-byte chunks: for S, lane 4g + c reads dims 32c ..
// 32c + 31 of rows g and g + 8 and k-step ks uses its bytes 4ks .. 4ks + 3
// (the MMA's k-columns 2c, 2c + 1 and 2c + 8, 2c + 9); for PV, it reads dims
// 16g .. 16g + 15 of rows 2c, 2c + 1, 2c + 8, 2c + 9, and a byte permute
// pairs rows 2c and 2c + 1 (and 2c + 8, 2c + 9) of one dim, the A fragment
// V^T wants, so output tile i holds dims 16g + 2i and 16g + 2i + 1. All
// loads of a quarter warp hit eight different bank groups.
//
// Weights: p * v_scale * f with f a power of two that keeps every weight
// below 2^15, an f16 value: the lazily rescaled p reaches 2^8, so f puts the
// largest scale of the segment's first tile in [2^6, 2^7) and drops (with a
// rescale of O) when a later tile's largest scale reaches 2^7 / f; the sum l
// takes the unscaled p, the segment's end divides O by f.
template <int Q8, int GW, bool PARTIAL>
__device__ __forceinline__ void mma_tile_q8(uint32_t kb, uint32_t vb, int row0, const float* vsp, int lo_valid,
                                            int valid, int vis0, int vis1, float qscale, Q8WarpState& st, int lane) {
  using namespace wmma16;
  const int g = lane >> 2, c = lane & 3;
  // ---- S^T = K . Q^T (hi and lo parts of Q, two accumulator chains each)
  uint32_t kw[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t row = kb + static_cast<uint32_t>((row0 + g + 8 * h) * 128);
    const uint4 u0 = lds128(row + static_cast<uint32_t>(((2 * c) ^ g) << 4));
    const uint4 u1 = lds128(row + static_cast<uint32_t>(((2 * c + 1) ^ g) << 4));
    kw[h][0] = u0.x;
    kw[h][1] = u0.y;
    kw[h][2] = u0.z;
    kw[h][3] = u0.w;
    kw[h][4] = u1.x;
    kw[h][5] = u1.y;
    kw[h][6] = u1.z;
    kw[h][7] = u1.w;
  }
  // the V codes: rows 2c, 2c + 1, 2c + 8, 2c + 9, dims 16g .. 16g + 15 (read
  // before the scores where registers allow, to hide the load latency)
  constexpr bool kEarlyV = GW <= 4;
  uint4 vr[4];
  auto load_v = [&]() {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = row0 + 2 * c + (j & 1) + 8 * (j >> 1);
      vr[j] = lds128(vb + static_cast<uint32_t>(r * 128) + static_cast<uint32_t>((g ^ (r & 7)) << 4));
    }
  };
  if constexpr (kEarlyV) load_v();
  float sc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[j][e] = 0.f;
  }
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t a[4];
    codes_to_f16x2<Q8>(kw[0][ks], a[0], a[2]);
    codes_to_f16x2<Q8>(kw[1][ks], a[1], a[3]);
    mma<false>(sc[ks & 1], a, st.qh[ks][0], st.qh[ks][1]);
    mma<false>(sc[2 + (ks & 1)], a, st.ql[ks][0], st.ql[ks][1]);
  }
  if constexpr (!kEarlyV) load_v();
  float x[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = ((sc[0][e] + sc[1][e]) + (sc[2][e] + sc[3][e])) * qscale;
  const bool q0 = 2 * c < GW, q1 = 2 * c + 1 < GW;
  if (!q0) {
    x[0] = kNegInf;
    x[2] = kNegInf;
  }
  if (!q1) {
    x[1] = kNegInf;
    x[3] = kNegInf;
  }
  float vs0, vs1;
  if (PARTIAL) {
    const bool ra = g >= lo_valid && g < valid, rb = g + 8 >= lo_valid && g + 8 < valid;
    if (!ra || g >= vis0) x[0] = kNegInf;
    if (!ra || g >= vis1) x[1] = kNegInf;
    if (!rb || g + 8 >= vis0) x[2] = kNegInf;
    if (!rb || g + 8 >= vis1) x[3] = kNegInf;
    // rows outside the range may hold anything: their scale is not used
    vs0 = ra ? vsp[row0 + g] : 0.f;
    vs1 = rb ? vsp[row0 + g + 8] : 0.f;
  } else {
    vs0 = vsp[row0 + g];
    vs1 = vsp[row0 + g + 8];
  }
  // ---- the weights' factor
  {
    float vmax = fmaxf(vs0, vs1);
#pragma unroll
    for (int msk = 4; msk < 32; msk <<= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, msk));
    if (st.f == 0.f || vmax * st.f >= 128.f) {
      // 2^(133 - E) for vmax in [2^(E - 127), 2^(E - 126)): vmax * f in [2^6, 2^7)
      const int e = static_cast<int>((__float_as_uint(vmax) >> 23) & 0xffu);
      const int field = min(254, max(1, 260 - e));
      const float nf = __uint_as_float(static_cast<uint32_t>(field) << 23);
      if (st.f != 0.f) {
        const float r = nf / st.f;  // both powers of two: exact
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
          for (int k = 0; k < 4; ++k) st.o[i][k] *= r;
        }
      }
      st.f = nf;
    }
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
  const float w0 = vs0 * st.f, w1 = vs1 * st.f;
  const float r0 = p0 * w0, r1 = p1 * w0, r2 = p2 * w1, r3 = p3 * w1;
  const uint32_t h01 = pack2<false>(r0, r1), h23 = pack2<false>(r2, r3);
  const float2 f01 = unpack2<false>(h01), f23 = unpack2<false>(h23);
  const uint32_t l01 = pack2<false>(r0 - f01.x, r1 - f01.y), l23 = pack2<false>(r2 - f23.x, r3 - f23.y);
  const uint32_t bh0 = movm_t(h01), bh1 = movm_t(h23), bl0 = movm_t(l01), bl1 = movm_t(l23);
  // ---- O^T += V^T . P^T
  uint32_t keep01 = 0xffffffffu, keep89 = 0xffffffffu;
  if (PARTIAL) {
    const int ra = 2 * c, rb = 2 * c + 8;
    keep01 = ((ra >= lo_valid && ra < valid) ? 0x0000ffffu : 0u) | ((ra + 1 >= lo_valid && ra + 1 < valid) ? 0xffff0000u : 0u);
    keep89 = ((rb >= lo_valid && rb < valid) ? 0x0000ffffu : 0u) | ((rb + 1 >= lo_valid && rb + 1 < valid) ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // bytes 2 (i & 1) and 2 (i & 1) + 1 of word i >> 1: dims 16g + 2i, + 1; rows interleaved
    const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
    const uint32_t e01 = __byte_perm(word(vr[0], i >> 1), word(vr[1], i >> 1), sel);
    const uint32_t e89 = __byte_perm(word(vr[2], i >> 1), word(vr[3], i >> 1), sel);
    uint32_t a[4];
    codes_to_f16x2<Q8>(e01, a[0], a[1]);
    codes_to_f16x2<Q8>(e89, a[2], a[3]);
    if (PARTIAL) {
      a[0] &= keep01;
      a[1] &= keep01;
      a[2] &= keep89;
      a[3] &= keep89;
    }
    mma<false>(st.o[i], a, bh0, bh1);
    mma<false>(st.o[i], a, bl0, bl1);
  }
}

// ------------------------------------------------------------------ work split
//
// A unit (sequence, kv-head chunk, head subgroup) has nb cache blocks. Its
// first nb - d blocks are static positions and its last d = nb * share / 256
// dynamic positions; each kind is laid end to end over the units (sequence
// major, then chunk, then subgroup): static positions 0 .. N0-1, dynamic
// positions 0 .. Nd-1. Workers 0 .. G-1 are the CTAs' static ranges
// [w N0 / G, (w+1) N0 / G); workers G .. G+K-1 are the chunks [k C, (k+1) C)
// of the dynamic positions, claimed at run time from a counter in the
// workspace by whichever CTA runs out of work first, so CTAs on SMs that
// stream faster take more of them. With the dynamic share spread over every
// unit's tail, a unit has a handful of contributors (the merge reads one
// record from each). Every segment of a unit that is not the whole unit
// leaves one fp32 record, which the merge kernel combines: worker w's slot
// 2w holds the segment at its range start, slot 2w + 1 the one that runs
// past its range end, and a part that lies strictly inside a range (a unit
// whose static or dynamic blocks one worker covers, but not all its blocks)
// goes to the unit's own slot, 2 (G + K) + 2 unit (+ 1 for the dynamic part).
struct MmaSplit {
  int64_t N0, Nd, G, K;
  int C, share;  // share 0: static ranges only
  __device__ __forceinline__ int dyn(int nb) const {
    return static_cast<int>((static_cast<int64_t>(nb) * share) >> 8);
  }
  // a / b for a, b >= 0, b > 0, with a 32-bit division when both fit
  __device__ __forceinline__ static int64_t div(int64_t a, int64_t b) {
    return (static_cast<uint64_t>(a | b) >> 32) == 0 ? static_cast<int64_t>(static_cast<uint32_t>(a) /
                                                                             static_cast<uint32_t>(b))
                                                     : a / b;
  }
  __device__ __forceinline__ int64_t start(int64_t w) const {
    if (w < G) return div(w * N0, G);
    const int64_t s = (w - G) * C;
    return s < Nd ? s : Nd;
  }
  __device__ __forceinline__ int64_t end(int64_t w) const {
    if (w < G) return div((w + 1) * N0, G);
    const int64_t e = (w - G + 1) * C;
    return e < Nd ? e : Nd;
  }
  // the static worker whose range holds static position b (N0 > 0)
  __device__ __forceinline__ int64_t static_worker(int64_t b) const { return div((b + 1) * G - 1, N0); }
  // record slot of worker w for the unit part that starts at u0 (in w's space)
  // and does not lie strictly inside w's range
  __device__ __forceinline__ int64_t record(int64_t w, int64_t u0) const { return 2 * w + (u0 > start(w) ? 1 : 0); }
  // record slot of a unit's static (dyn = false) or dynamic part that lies
  // strictly inside one worker's range
  __device__ __forceinline__ int64_t interior(int64_t unit, bool dyn) const {
    return 2 * (G + K) + 2 * unit + (dyn ? 1 : 0);
  }
};

// scan_blocks for a batch of at most 32 sequences: warp 0 computes the
// exclusive prefix sums s_scan[0..B] with shuffles, and one CTA barrier
// publishes them.
__device__ inline void scan_blocks_warp(const int32_t* lens, int B, int bs, int max_blocks, int window, int min_len,
                                        const int32_t* row_start, int row_div, int* s_scan) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int x = lane < B ? seq_blocks(lens, lane, bs, max_blocks, window, min_len, row_start, row_div) : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += u;
    }
    if (lane < B) s_scan[lane + 1] = x;
    if (lane == 0) s_scan[0] = 0;
  }
  __syncthreads();
}

// N: all positions, Nd: the dynamic ones under `share`. The dynamic share is
// kept only when every CTA still gets at least min_static static positions;
// every CTA computes the same split.
__device__ __forceinline__ MmaSplit make_mma_split(int64_t N, int64_t Nd, int64_t G, int share, int chunk,
                                                   int min_static) {
  MmaSplit s;
  s.G = G;
  s.C = chunk > 0 ? chunk : 1;
  s.share = chunk > 0 ? share : 0;
  s.Nd = s.share > 0 ? Nd : 0;
  if (s.Nd > 0 && N - s.Nd < G * static_cast<int64_t>(min_static)) {
    s.share = 0;
    s.Nd = 0;
  }
  s.N0 = N - s.Nd;
  s.K = (s.Nd + s.C - 1) / s.C;
  return s;
}

// Exclusive prefix sums over the batch of d = nb * share / 256 (nb from the
// block prefix s_scan) into s_dscan[0..B]; the whole CTA participates.
// s_dscan needs B + 1 + 32 ints.
__device__ inline void scan_dyn(int B, int share, const int* s_scan, int* s_dscan) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (B + nt - 1) / nt;
  const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
  auto d_of = [&](int b) {
    return static_cast<int>((static_cast<int64_t>(s_scan[b + 1] - s_scan[b]) * share) >> 8);
  };
  int local = 0;
  for (int b = b0; b < b1; ++b) local += d_of(b);
  const int lane = tid & 31, wid = tid >> 5;
  int v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  int* wsum = s_dscan + B + 1;
  if (lane == 31) wsum[wid] = v;
  __syncthreads();
  if (wid == 0) {
    const int nw = (nt + 31) >> 5;
    int x = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += u;
    }
    if (lane < nw) wsum[lane] = x;
  }
  __syncthreads();
  int run = v - local + (wid > 0 ? wsum[wid - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    s_dscan[b] = run;
    run += d_of(b);
  }
  if (b1 == B && b0 < B) s_dscan[B] = run;
  if (B == 0 && tid == 0) s_dscan[0] = 0;
  __syncthreads();
}

// Where static (dyn = false) or dynamic position pos lies: the unit, the
// block index j within the unit, the unit's total blocks nb, its blocks in
// this space cnt, and u0, the space's first position of the unit.
struct SplitPos {
  int64_t u0;
  int seq, chunk, hsub, j, nb, cnt;
};

__device__ __forceinline__ SplitPos locate_split(int64_t pos, bool dyn, const MmaSplit& sp, int HN,
                                                 const int* s_scan, const int* s_dscan, int B, int n_hsub) {
  auto prefix = [&](int b) -> int64_t {
    const int d = sp.share > 0 ? s_dscan[b] : 0;
    return static_cast<int64_t>(HN) * (dyn ? d : s_scan[b] - d);
  };
  int a = 0, hi = B - 1;  // the last sequence whose prefix is <= pos (skips empty ones)
  while (a < hi) {
    const int mid = (a + hi + 1) >> 1;
    if (prefix(mid) <= pos) a = mid; else hi = mid - 1;
  }
  SplitPos r;
  r.seq = a;
  r.nb = s_scan[a + 1] - s_scan[a];
  const int d = sp.dyn(r.nb);
  r.cnt = dyn ? d : r.nb - d;
  const int r2 = static_cast<int>(pos - prefix(a));
  const int idx = r2 / r.cnt;
  const int jsp = r2 - idx * r.cnt;
  r.chunk = idx / n_hsub;
  r.hsub = idx - r.chunk * n_hsub;
  r.j = dyn ? r.nb - d + jsp : jsp;
  r.u0 = pos - jsp;
  return r;
}

// The records of one unit: its static part [su0, su0 + s) spans static
// workers c0 .. c1, its dynamic part [du0, du0 + d) chunks k0 .. k1.
struct UnitRecs {
  int64_t su0, du0, c0, c1, k0, k1, ns, R;
  bool whole;  // one worker covered the unit: no records
};

__device__ __forceinline__ UnitRecs unit_recs(int seq, int idx, const MmaSplit& sp, int HN, const int* s_scan,
                                              const int* s_dscan) {
  UnitRecs u;
  const int nb = s_scan[seq + 1] - s_scan[seq];
  const int d = sp.dyn(nb), s = nb - d;
  const int dpre = sp.share > 0 ? s_dscan[seq] : 0;
  u.su0 = static_cast<int64_t>(HN) * (s_scan[seq] - dpre) + static_cast<int64_t>(idx) * s;
  u.c0 = sp.static_worker(u.su0);
  u.c1 = sp.static_worker(u.su0 + s - 1);
  u.du0 = static_cast<int64_t>(HN) * dpre + static_cast<int64_t>(idx) * d;
  u.k0 = MmaSplit::div(u.du0, sp.C);
  u.k1 = d > 0 ? MmaSplit::div(u.du0 + d - 1, sp.C) : u.k0 - 1;
  u.ns = u.c1 - u.c0 + 1;
  u.R = u.ns + (u.k1 - u.k0 + 1);
  u.whole = d == 0 && u.c0 == u.c1;
  return u;
}

// Record slot of contributor r of the unit (-1: an empty static range). Every
// static range after c0 starts inside the unit (slot 2w) and, when N0 >= G,
// is non-empty; dynamic chunk k starts at k C.
__device__ __forceinline__ int64_t unit_record(const UnitRecs& u, int64_t unit, const MmaSplit& sp, int64_t r) {
  if (r < u.ns) {
    if (r == 0) {
      const int64_t s0 = sp.start(u.c0);
      return u.c0 == u.c1 && u.su0 > s0 ? sp.interior(unit, false) : 2 * u.c0 + (u.su0 > s0 ? 1 : 0);
    }
    const int64_t wk = u.c0 + r;
    return (sp.N0 >= sp.G || sp.start(wk) != sp.end(wk)) ? 2 * wk : -1;
  }
  const int64_t k = u.k0 + (r - u.ns);
  const bool after = u.du0 > k * sp.C;
  return u.k0 == u.k1 && after ? sp.interior(unit, true) : 2 * (sp.G + k) + (after ? 1 : 0);
}

// ------------------------------------------------------------ shared memory
//
// Offsets from a 1024-byte aligned base (the host adds 1024 bytes of slack
// for the alignment). A stage is [K half 0][K half 1][V half 0][V half 1]
// (each hc * block_size rows of 128 bytes, swizzled); each stage has a
// 64-byte descriptor written by the producer warp, a "full" barrier (the
// copies landed) and an "empty" barrier (every consumer warp released it).
// A segment's query rows [hc][GH][128] arrive with its first stage (same
// "full" barrier) in one of two query slots.

struct GqaMmaSmem {
  size_t box_bytes, stage_bytes, vbox_off, vs_off, q_off, q_slot_bytes, meta_off, full_off, empty_off, iss_off,
      misc_off, scan_off, dscan_off, total;
};

// q8: one-byte caches, whose stage holds one K and one V box (128 codes per
// row) and the block's V scales [hc * block_size]; with pair, two blocks of
// one segment (K boxes, then V boxes, then the two scale arrays, so that the
// second block's rows follow the first's). The query rows of a segment go to
// one of two query slots after the ring (a segment's consumers copy them into
// registers at its first stage).
__host__ __device__ inline GqaMmaSmem gqa_mma_smem_layout(int q_elt, int GH, int block_size, int hc, int stages,
                                                          int batch, bool q8 = false, bool pair = false) {
  GqaMmaSmem s;
  const size_t np = (q8 && pair) ? 2 : 1;  // cache blocks per stage
  s.box_bytes = static_cast<size_t>(hc) * block_size * 128;
  s.vbox_off = (q8 ? np : 2) * s.box_bytes;
  s.vs_off = (q8 ? 2 * np : 4) * s.box_bytes;
  s.stage_bytes = align_up(s.vs_off + (q8 ? np * hc * block_size * 4 : 0), 1024);
  s.q_slot_bytes = static_cast<size_t>(hc) * GH * 128 * q_elt;
  s.q_off = static_cast<size_t>(stages) * s.stage_bytes;
  s.meta_off = s.q_off + 2 * s.q_slot_bytes;
  s.full_off = s.meta_off + static_cast<size_t>(stages) * 64;
  s.empty_off = s.full_off + static_cast<size_t>(stages) * 8;
  s.iss_off = s.empty_off + static_cast<size_t>(stages) * 8;
  s.misc_off = align_up(s.iss_off + static_cast<size_t>(stages) * 4, 16);
  s.scan_off = s.misc_off + 16;
  s.dscan_off = s.scan_off + static_cast<size_t>(batch + 1 + 32) * 4;
  s.total = s.dscan_off + static_cast<size_t>(batch + 1 + 32) * 4 + 1024;
  return s;
}


__host__ __device__ constexpr int mma_warps_per_kvhead(int GH) { return GH > 8 ? GH / 8 : 1; }
__host__ __device__ constexpr int mma_max_chunk(int GH) { return kMmaWarps / mma_warps_per_kvhead(GH); }

// Descriptor of the position a stage holds (written by the producer before it
// arms the stage's "full" barrier).
struct StageMeta {
  int64_t u0;      // first global position of the unit
  int seq;         // -1: no more work
  int chunk, hsub, nb;
  int jb;          // table index of the block
  int n_rows, r0;  // cached rows of the sequence, its first visible row
  int flags;
  int rec;         // record index of the segment (partial segments)
  int qslot;       // query slot holding the segment's query rows
  int npos;        // cache blocks in the stage (2: blocks jb and jb + 1)
};
static_assert(sizeof(StageMeta) <= 64, "stage descriptor slot");
constexpr int kFirst = 1, kLast = 2, kSrc = 4, kWhole = 8;

// Q8 = 0: T is the cache and query type; Q8 = 1 (e4m3) or 2 (int8): one-byte
// caches with T (bf16) queries.
template <typename T, int GH, bool EXT, int Q8 = 0>
__global__ void __launch_bounds__(kMmaThreads, kMmaCtasPerSm)
    gqa_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const GqaParams p) {
  using namespace wmma16;
  constexpr int D = 128;
  constexpr bool BF = Q8 == 0 && std::is_same<T, __nv_bfloat16>::value;
  static_assert(Q8 == 0 || (!EXT && std::is_same<T, __nv_bfloat16>::value), "one-byte caches: bf16 queries");
  constexpr int HW = mma_warps_per_kvhead(GH);  // warps per kv head
  constexpr int GW = GH / HW;                   // query heads per warp (MMA columns)
  constexpr int HCM = kMmaWarps / HW;           // kv heads per CTA at most
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
  const bool paired = Q8 != 0 && p.pair != 0;  // two cache blocks per stage
  const GqaMmaSmem L = gqa_mma_smem_layout(sizeof(T), GH, bs, hc, S, p.batch, Q8 != 0, paired);
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + L.meta_off);
  uint64_t* fbar = reinterpret_cast<uint64_t*>(smem + L.full_off);
  uint64_t* ebar = reinterpret_cast<uint64_t*>(smem + L.empty_off);
  unsigned int* s_iss = reinterpret_cast<unsigned int*>(smem + L.iss_off);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc_off);
  int* s_scan = reinterpret_cast<int*>(smem + L.scan_off);
  int* s_dscan = reinterpret_cast<int*>(smem + L.dscan_off);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int kh = w / HW, hw = w % HW;
  const int nact = hc * HW;  // consumer warps with work
  const int B = p.batch;
  const uint32_t full = 0xffffffffu;
  const int HN = p.n_chunks * p.n_hsub;

  if (tid < S) {
    mbar_init(fbar + tid, 1);     // the producer's arrive (with the copy bytes)
    mbar_init(ebar + tid, nact);  // one release per consumer warp
    s_iss[tid] = 0u;
  }
  if (tid == 0) {
    *s_abort = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  fence_barrier_init();
  // Launched right behind the previous kernel of the stream (programmatic
  // stream serialisation), the kernel sets up its barriers while that grid
  // runs; every thread then waits for it (its writes become visible) before it
  // reads or writes any caller buffer.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (w == kMmaWarps && !p.unit_mode) {
    // Warm L2 with the block-table lines this CTA reads first, which only the
    // scan below decides: the whole table when it is small (up to 64 KB), else
    // a guess that assumes full-length sequences. Either overlaps the scan.
    const int64_t entries = static_cast<int64_t>(B) * p.max_blocks;
    if (entries <= 16384) {
      for (int64_t e = 32 * static_cast<int64_t>(lane); e < entries; e += 32 * 32) prefetch_l2(p.block_tables + e);
      if (lane == 0) prefetch_l2(p.block_tables + entries - 1);
    } else {
      const int64_t per_seq = static_cast<int64_t>(HN) * p.max_blocks;
      const int64_t pos = static_cast<int64_t>(blockIdx.x) * B * per_seq / gridDim.x + 32 * lane;
      const int64_t seq = pos / per_seq;
      const int j = static_cast<int>((pos - seq * per_seq) % p.max_blocks);
      if (lane < 4 && seq < B) prefetch_l2(p.block_tables + seq * p.max_blocks + j);
    }
  }
  // ends with a CTA barrier; a batch of up to 32 sequences is scanned by one warp
  if (B <= 32)
    scan_blocks_warp(p.context_lens, B, bs, p.max_blocks, wnd, min_len, row_start, row_div, s_scan);
  else
    scan_blocks(p.context_lens, B, bs, p.max_blocks, wnd, min_len, row_start, row_div, s_scan);
  const int64_t N = static_cast<int64_t>(HN) * s_scan[B];
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;

  if (blockIdx.x == 0) {
    int empty = 0;
    for (int b = tid; b < B; b += blockDim.x) {
      const int n = __ldg(p.context_lens + b);
      if (n < min_len || n > bs * p.max_blocks) set_flag(p.err, 0x2u);
      if (row_div > 0 && __ldg(row_start + b / (row_div > 0 ? row_div : 1)) > n) set_flag(p.err, 0x2u);
      empty |= (s_scan[b + 1] == s_scan[b]) ? 1 : 0;
    }
    if (__syncthreads_or(empty) && !p.unit_mode) {
      const int rows = n_tok * p.n_q_heads * D;
      for (int b = 0; b < B; ++b) {
        if (s_scan[b + 1] != s_scan[b]) continue;
        for (int idx = tid; idx < HN; idx += blockDim.x)  // nothing to merge
          p.unit_lists[static_cast<int64_t>(b * HN + idx) * (1 + p.list_cap)] = 0;
        for (int idx = tid; idx < rows; idx += blockDim.x)
          store_out(p.out, static_cast<int64_t>(b) * rows + idx, 0.f, p.out_dtype);
        if (EXT && p.lse != nullptr)
          for (int idx = tid; idx < n_tok * p.n_q_heads; idx += blockDim.x)
            p.lse[static_cast<int64_t>(b) * n_tok * p.n_q_heads + idx] = kNegInf;
      }
    }
  }

  // The work split (every CTA computes the same one). In the unit mode CTA u
  // takes unit u whole and nothing is claimed.
  const int dshare = (!p.unit_mode && p.dyn_chunk > 0) ? p.dyn_share : 0;
  if (dshare > 0) scan_dyn(B, dshare, s_scan, s_dscan);  // ends with a CTA barrier; unused without a share
  MmaSplit sp;
  int64_t lo, hi;
  if (p.unit_mode) {
    sp = make_mma_split(N, 0, G, 0, 0, 1);
    const int seq = static_cast<int>(c / HN);
    const int idx = static_cast<int>(c - static_cast<int64_t>(seq) * HN);
    const int nb = s_scan[seq + 1] - s_scan[seq];
    if (nb == 0) {
      if (w < nact) {
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
    sp = make_mma_split(N, dshare > 0 ? static_cast<int64_t>(HN) * s_dscan[B] : 0, G, dshare, p.dyn_chunk,
                        p.dyn_min_static);
    lo = sp.start(c);
    hi = sp.end(c);
  }

  if (w == kMmaWarps) {
    // ============================================================== producer
    // Walks its static range, then the chunks it claims, position by
    // position: lane i describes position base + i of a window of 32 (block
    // table entry, segment flags, record), lane 0 waits for the stage to be
    // released, writes its descriptor and issues the copies.
    const T* qg = static_cast<const T*>(p.q);
    const uint64_t pol = policy_evict_first();
    const uint32_t box_bytes = static_cast<uint32_t>(L.box_bytes);
    const uint32_t q_bytes = static_cast<uint32_t>(hc * GH * D * sizeof(T));
    const uint32_t vs_bytes = static_cast<uint32_t>(hc * bs * 4);
    const bool q_contig = (GH == p.group);
    unsigned int claim = 0;
    if (!p.unit_mode && sp.K > 0 && lane == 0) claim = atomicAdd(p.sched, 1u);  // for after the static range
    int64_t wk = c;
    uint32_t slot = 0, ph = 0;
    bool ok = true;
    // Query slots: slot j was last filled with the first stage of the
    // segment issued as position qpos_j (ring slot and phase in qsp_j).
    // Reusing it for a new segment waits until that stage was released (its
    // rows are in the consumers' registers by then); when S positions have
    // been issued since, the ring order already guarantees it.
    int64_t icount = 0;
    int nseg = 0;
    int64_t qpos0 = -(1ll << 40), qpos1 = -(1ll << 40);
    uint32_t qsp0 = 0u, qsp1 = 0u;  // ring slot | phase << 16
    for (;;) {
      for (int64_t bpos = lo; ok && bpos < hi; bpos += 32) {
        const int64_t pos = bpos + lane;
        StageMeta m{};
        int src = -1, qoff = -1;
        if (pos < hi) {
          const SplitPos bp = locate_split(pos, wk >= G, sp, HN, s_scan, s_dscan, B, p.n_hsub);
          m.seq = bp.seq;
          m.chunk = bp.chunk;
          m.hsub = bp.hsub;
          m.nb = bp.nb;
          m.u0 = bp.u0;
          m.n_rows = seq_rows(p.context_lens, bp.seq, bs, p.max_blocks, min_len);
          m.r0 = start_row(m.n_rows, wnd, row_start, row_div, bp.seq);
          m.jb = m.r0 / bs + bp.j;
          const int phys = __ldg(p.block_tables + static_cast<int64_t>(bp.seq) * p.max_blocks + m.jb);
          if (phys >= 0 && phys < p.num_blocks) src = (phys * p.n_kv_heads + bp.chunk * hc) * bs;
          const bool first = (pos == lo) || (pos == bp.u0);
          const bool whole = bp.cnt == bp.nb && bp.u0 >= lo && bp.u0 + bp.cnt <= hi;
          m.flags = (first ? kFirst : 0) | ((pos == hi - 1 || pos - bp.u0 == bp.cnt - 1) ? kLast : 0) |
                    (src >= 0 ? kSrc : 0) | (whole ? kWhole : 0);
          const int64_t unit = static_cast<int64_t>(bp.seq) * HN + bp.chunk * p.n_hsub + bp.hsub;
          m.rec = static_cast<int>((bp.u0 > lo && bp.u0 + bp.cnt <= hi) ? sp.interior(unit, wk >= G)
                                                                        : sp.record(wk, bp.u0));
          if (first)
            qoff = multi ? (bp.seq * p.n_chunks + bp.chunk) * p.n_hsub + bp.hsub
                         : (bp.seq * p.n_q_heads + bp.chunk * hc * p.group + bp.hsub * GH) * D;
        }
        const int n = static_cast<int>(hi - bpos < 32 ? hi - bpos : 32);
        for (int i = 0; i < n;) {
          StageMeta mi;
          mi.u0 = __shfl_sync(full, m.u0, i);
          mi.seq = __shfl_sync(full, m.seq, i);
          mi.chunk = __shfl_sync(full, m.chunk, i);
          mi.hsub = __shfl_sync(full, m.hsub, i);
          mi.nb = __shfl_sync(full, m.nb, i);
          mi.jb = __shfl_sync(full, m.jb, i);
          mi.n_rows = __shfl_sync(full, m.n_rows, i);
          mi.r0 = __shfl_sync(full, m.r0, i);
          mi.flags = __shfl_sync(full, m.flags, i);
          mi.rec = __shfl_sync(full, m.rec, i);
          mi.qslot = 0;
          mi.npos = 1;
          const int srci = __shfl_sync(full, src, i);
          const int qo = __shfl_sync(full, qoff, i);
          // paired stages: the segment's next block (held by lane i + 1 of this
          // window) shares the stage when both blocks are valid
          int srcj = -1;
          if (paired) {
            const int nx = (i + 1) & 31;
            const int srcn = __shfl_sync(full, src, nx);
            const int fln = __shfl_sync(full, m.flags, nx);
            if (i + 1 < n && !(mi.flags & kLast) && srci >= 0 && srcn >= 0) {
              srcj = srcn;
              mi.npos = 2;
              mi.flags |= fln & kLast;
            }
          }
          if (lane == 0) {
            ok = mbar_wait_data(ebar + slot, ph ^ 1u, p.wait_polls) && !*s_abort;
            const int qj = nseg & 1;
            const int64_t qp = qj ? qpos1 : qpos0;
            const uint32_t qsp = qj ? qsp1 : qsp0;
            if (ok && qo >= 0 && icount - qp < S)
              ok = mbar_wait_data(ebar + (qsp & 0xffffu), qsp >> 16, p.wait_polls) && !*s_abort;
            if (ok) {
              if (qo >= 0) {
                ++nseg;
                if (qj) {
                  qpos1 = icount;
                  qsp1 = slot | (ph << 16);
                } else {
                  qpos0 = icount;
                  qsp0 = slot | (ph << 16);
                }
                mi.qslot = qj;
              }
              ++icount;
              if (srci < 0) set_flag(p.err, 0x1u);
              meta[slot] = mi;
              const uint32_t bytes =
                  (srci >= 0 ? (Q8 ? static_cast<uint32_t>(mi.npos) * (2 * box_bytes + vs_bytes) : 4 * box_bytes) : 0u) +
                  (qo >= 0 ? q_bytes : 0u);
              s_iss[slot] += 1u;
              if (bytes == 0) {
                mbar_arrive(fbar + slot);
              } else {
                const uint32_t dst = base + static_cast<uint32_t>(slot * L.stage_bytes);
                const uint32_t bar = smem_addr(fbar + slot);
                mbar_arrive_expect_tx(fbar + slot, bytes);
                if (srci >= 0) {
                  if constexpr (Q8 != 0) {
                    const uint32_t vdst = dst + static_cast<uint32_t>(L.vbox_off);
                    unsigned char* vsd = smem + slot * L.stage_bytes + L.vs_off;
                    tma2d(dst, &tm_k, 0, srci, bar, pol);
                    tma2d(vdst, &tm_v, 0, srci, bar, pol);
                    bulk_g2s(vsd, p.v_scale + srci, vs_bytes, fbar + slot, pol);
                    if (srcj >= 0) {
                      tma2d(dst + box_bytes, &tm_k, 0, srcj, bar, pol);
                      tma2d(vdst + box_bytes, &tm_v, 0, srcj, bar, pol);
                      bulk_g2s(vsd + vs_bytes, p.v_scale + srcj, vs_bytes, fbar + slot, pol);
                    }
                  } else {
                    tma2d(dst, &tm_k, 0, srci, bar, pol);
                    tma2d(dst + box_bytes, &tm_k, 64, srci, bar, pol);
                    tma2d(dst + 2 * box_bytes, &tm_v, 0, srci, bar, pol);
                    tma2d(dst + 3 * box_bytes, &tm_v, 64, srci, bar, pol);
                  }
                }
                if (qo >= 0) {
                  unsigned char* qdst = smem + L.q_off + qj * L.q_slot_bytes;
                  if (multi) {
                    const int hs = qo % p.n_hsub, rest = qo / p.n_hsub;
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
                    bulk_g2s(qdst, qg + qo, q_bytes, fbar + slot, pol);
                  } else {
                    const uint32_t rb = static_cast<uint32_t>(GH * D * sizeof(T));
                    for (int h = 0; h < hc; ++h) bulk_g2s(qdst + h * rb, qg + qo + h * p.group * D, rb, fbar + slot, pol);
                  }
                }
              }
            } else {
              set_flag(p.err, 0x8u);
              *s_abort = 1;
            }
          }
          ok = __shfl_sync(full, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (!p.unit_mode && wk < G && mi.u0 == bpos + i) {
            // the unit's first block: publish its record list for the merge
            // (after the copies are on their way)
            const int uidx = mi.chunk * p.n_hsub + mi.hsub;
            const int64_t unit = static_cast<int64_t>(mi.seq) * HN + uidx;
            const UnitRecs u = unit_recs(mi.seq, uidx, sp, HN, s_scan, s_dscan);
            int* lst = p.unit_lists + unit * (1 + p.list_cap);
            const int R = u.whole ? 0 : static_cast<int>(u.R < p.list_cap ? u.R : p.list_cap);
            for (int r = lane; r < R; r += 32) lst[1 + r] = static_cast<int>(unit_record(u, unit, sp, r));
            if (lane == 0) lst[0] = R;
          }
          if (++slot == static_cast<uint32_t>(S)) {
            slot = 0;
            ph ^= 1u;
          }
          i += mi.npos;
        }
      }
      if (!ok || p.unit_mode || sp.K == 0) break;
      // the next chunk: the claim made a range ago; claim the one after it now
      const int64_t k = static_cast<int64_t>(__shfl_sync(full, claim, 0));
      if (k >= sp.K) break;
      if (lane == 0) claim = atomicAdd(p.sched, 1u);
      wk = G + k;
      lo = sp.start(wk);
      hi = sp.end(wk);
    }
    if (lane == 0) {
      if (ok && mbar_wait_bounded(ebar + slot, ph ^ 1u)) {
        meta[slot].seq = -1;  // no more work
        mbar_arrive(fbar + slot);
      } else if (ok) {
        set_flag(p.err, 0x8u);
        *s_abort = 1;
      }
      // Every CTA makes exactly one failed claim; the last one to do so
      // resets the claim counter for the next call.
      if (!p.unit_mode && sp.K > 0 && atomicAdd(p.sched + 1, 1u) == static_cast<unsigned int>(G) - 1) {
        atomicExch(p.sched, 0u);
        atomicExch(p.sched + 1, 0u);
      }
    }
  } else if (w < nact) {
    // ============================================================== consumers
    const int g8 = lane >> 2, c4 = lane & 3;
    const uint32_t box_bytes = static_cast<uint32_t>(L.box_bytes);
    // One pass of the outer loop per segment (the positions of one unit in
    // one worker's range): the first position carries the unit's query rows,
    // the last one closes the segment.
    uint32_t slot = 0, ph = 0;
    bool abort_seen = false;
    for (;;) {
      if (!mbar_wait_data(fbar + slot, ph, p.wait_polls) || *s_abort) {
        abort_seen = true;
        break;
      }
      StageMeta m = meta[slot];
      if (m.seq < 0) break;
      const int kvh = m.chunk * hc + kh;
      const int v0 = m.hsub * GH + hw * GW;
      // rows at the end each of the lane's two query columns may not see
      const int dh0 = (EXT && causal) ? tm - (v0 + 2 * c4) / p.group : 0;
      const int dh1 = (EXT && causal) ? tm - (v0 + 2 * c4 + 1) / p.group : 0;
      std::conditional_t<Q8 != 0, Q8WarpState, MmaWarpState> st;
      float qsc = p.qscale;
      {
        const unsigned char* qs = smem + L.q_off + m.qslot * L.q_slot_bytes +
                                  static_cast<size_t>(kh * GH + hw * GW) * D * sizeof(T);
        if constexpr (Q8 == 0) {
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
        } else {
          // q * k_scale over dims 32c .. 32c + 31 of query g, scaled by 2^t
          // so that the warp's largest entry lies in [2^14, 2^15), as f16 hi + lo
          float y[32];
          if (g8 < GW) {
            const uint4* qv = reinterpret_cast<const uint4*>(qs + (g8 * D + 32 * c4) * 2);
            const float4* kv = reinterpret_cast<const float4*>(p.k_scale + static_cast<int64_t>(kvh) * D + 32 * c4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 u = qv[j];
              const float4 s0 = __ldg(kv + 2 * j), s1 = __ldg(kv + 2 * j + 1);
              const uint32_t wq[4] = {u.x, u.y, u.z, u.w};
              const float sk[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const uint32_t wv = wq[e >> 1];
                y[8 * j + e] = __uint_as_float((e & 1) ? (wv & 0xffff0000u) : (wv << 16)) * sk[e];
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) y[e] = 0.f;
          }
          float amax = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(y[e]));
#pragma unroll
          for (int msk = 1; msk < 32; msk <<= 1) amax = fmaxf(amax, __shfl_xor_sync(full, amax, msk));
          const int field = min(254, max(1, 268 - static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu)));
          const float fq = __uint_as_float(static_cast<uint32_t>(field) << 23);
          qsc = p.qscale * __uint_as_float(static_cast<uint32_t>(254 - field) << 23);  // / 2^t, exact
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float z0 = y[4 * ks + 2 * h] * fq, z1 = y[4 * ks + 2 * h + 1] * fq;
              const uint32_t hi = pack2<false>(z0, z1);
              const float2 fh = unpack2<false>(hi);
              st.qh[ks][h] = hi;
              st.ql[ks][h] = pack2<false>(z0 - fh.x, z1 - fh.y);
            }
          }
          st.f = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
          for (int e = 0; e < 4; ++e) st.o[i][e] = 0.f;
        }
        st.m[0] = st.m[1] = -1e30f;  // finite: a column that meets only masked rows keeps weight 0
        st.l[0] = st.l[1] = 0.f;
      }
      for (;;) {
        if (m.flags & kSrc) {
          const uint32_t stg = base + static_cast<uint32_t>(slot * L.stage_bytes);
          const float* vsp = reinterpret_cast<const float*>(smem + slot * L.stage_bytes + L.vs_off);
          // one tile (PT: partial) on the kernel's cache type
          auto tile = [&](auto pt, int row0, int lo_valid, int valid, int vis0, int vis1) {
            constexpr bool PT = decltype(pt)::value;
            if constexpr (Q8 == 0)
              mma_tile<BF, GW, PT>(stg, stg + 2 * box_bytes, box_bytes, row0, lo_valid, valid, vis0, vis1, qsc, st,
                                   lane);
            else
              mma_tile_q8<Q8, GW, PT>(stg, stg + static_cast<uint32_t>(L.vbox_off), row0, vsp, lo_valid, valid, vis0,
                                      vis1, qsc, st, lane);
          };
          using Full = std::integral_constant<bool, false>;
          using Part = std::integral_constant<bool, true>;
          const int j0 = m.r0 / bs;
          const int tiles = bs / 16;
          // block jb + j of a paired stage: its rows follow block jb's (hc * bs rows per block)
          for (int j = 0; j < (paired ? m.npos : 1); ++j) {
            const int jb = m.jb + j;
            const int rb = m.n_rows - jb * bs;  // rows from the block's first to the end
            const int vr = min(bs, rb);
            const int lr = (jb == j0) ? m.r0 - j0 * bs : 0;
            const int rowk = (j * hc + kh) * bs;
            if (rb - tm >= bs && lr == 0) {
              for (int tt = 0; tt < tiles; ++tt) tile(Full{}, rowk + tt * 16, 0, 16, 16, 16);
            } else {
              for (int tt = 0; tt < tiles; ++tt) {
                const int valid = vr - tt * 16, lo_valid = lr - tt * 16;
                const int rt = rb - tt * 16;
                if (valid <= 0) break;
                if (lo_valid >= 16) continue;
                if (rt - tm >= 16 && lo_valid <= 0)
                  tile(Full{}, rowk + tt * 16, 0, 16, 16, 16);
                else
                  tile(Part{}, rowk + tt * 16, lo_valid, valid, EXT ? min(valid, rt - dh0) : valid,
                       EXT ? min(valid, rt - dh1) : valid);
              }
            }
          }
        }
        // release the stage: every read of it fed an instruction issued before this barrier
        __syncwarp();
        if (lane == 0) mbar_arrive(ebar + slot);
        if (++slot == static_cast<uint32_t>(S)) {
          slot = 0;
          ph ^= 1u;
        }
        if (m.flags & kLast) break;
        if (!mbar_wait_data(fbar + slot, ph, p.wait_polls) || *s_abort) {
          abort_seen = true;
          break;
        }
        m = meta[slot];
      }
      if (abort_seen) break;

      // ---- close the segment
      float lw0 = st.l[0], lw1 = st.l[1];
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1) {
        lw0 += __shfl_xor_sync(full, lw0, msk);
        lw1 += __shfl_xor_sync(full, lw1, msk);
      }
      const bool qv0 = 2 * c4 < GW, qv1 = 2 * c4 + 1 < GW;
      // output dims of o[i][0..1] and o[i][2..3], and the one-byte path's weight factor
      float fo = 1.f;
      if constexpr (Q8 != 0) fo = st.f > 0.f ? 1.0f / st.f : 0.f;
      auto dim_a = [&](int i) { return Q8 != 0 ? 16 * g8 + 2 * i : 16 * i + g8; };
      constexpr int kDimB = Q8 != 0 ? 1 : 8;
      if (m.flags & kWhole) {
        const float i0 = fo / lw0, i1 = fo / lw1;
        const int64_t ob0 = (EXT ? out_row(p, m.seq, kvh, v0 + 2 * c4)
                                 : static_cast<int64_t>(m.seq) * p.n_q_heads + kvh * p.group + v0 + 2 * c4) * D;
        const int64_t ob1 = EXT ? out_row(p, m.seq, kvh, v0 + 2 * c4 + 1) * D : ob0 + D;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d0 = dim_a(i);
          if (qv0) {
            store_out(p.out, ob0 + d0, st.o[i][0] * i0, p.out_dtype);
            store_out(p.out, ob0 + d0 + kDimB, st.o[i][2] * i0, p.out_dtype);
          }
          if (qv1) {
            store_out(p.out, ob1 + d0, st.o[i][1] * i1, p.out_dtype);
            store_out(p.out, ob1 + d0 + kDimB, st.o[i][3] * i1, p.out_dtype);
          }
        }
        if (EXT && p.lse != nullptr && g8 == 0) {
          if (qv0) p.lse[out_row(p, m.seq, kvh, v0 + 2 * c4)] = st.m[0] + __log2f(lw0);
          if (qv1) p.lse[out_row(p, m.seq, kvh, v0 + 2 * c4 + 1)] = st.m[1] + __log2f(lw1);
        }
      } else {
        // record (max, sum, unnormalised output) of this warp's heads
        const int64_t rec = m.rec;
        const int hr = kh * GH + hw * GW;
        float* ro0 = p.rec_o + (rec * HS + hr + 2 * c4) * D;
        float* ro1 = ro0 + D;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d0 = dim_a(i);
          if (qv0) {
            ro0[d0] = st.o[i][0] * fo;
            ro0[d0 + kDimB] = st.o[i][2] * fo;
          }
          if (qv1) {
            ro1[d0] = st.o[i][1] * fo;
            ro1[d0 + kDimB] = st.o[i][3] * fo;
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
      }
    }
    if (abort_seen && lane == 0) {
      set_flag(p.err, 0x8u);
      *s_abort = 1;
    }
  }

  __syncthreads();
  if (*s_abort && tid == 0) {
    // Copies that may still be in flight must land before the CTA exits and
    // its shared memory is reused: wait (bounded) for the latest issued fill
    // of every stage.
    for (int x = 0; x < S; ++x) {
      const unsigned int n = s_iss[x];
      if (n > 0) (void)mbar_wait_bounded(fbar + x, (n - 1) & 1u);
    }
  }
}

// ------------------------------------------------------------------ merge
//
// Runs after the decode kernel (launched behind it on the same stream). For
// one unit and one head group (the GW query heads a consumer warp owns) it
// combines the records listed for the unit (by the worker that held its
// first block) with the log-sum-exp rule, O = sum_r 2^(m_r - M) O_r /
// sum_r 2^(m_r - M) l_r, and writes the normalised output (and the LSE row).
// The list is read together with its count, the records in one batch: two
// dependent rounds of loads. The CTA's threads form NG groups of 32 GW, a
// thread owning dims 4 (t & 31) .. + 3 of head (t mod 32 GW) / 32; group g
// folds records g, g + NG, ..., then the groups' results are combined. All
// merges run in parallel, one small CTA each (several fit on an SM).
constexpr int kMergeBatch = 16;
__host__ __device__ constexpr int merge_threads(int GH) {
  return 32 * (GH / mma_warps_per_kvhead(GH)) > 128 ? 32 * (GH / mma_warps_per_kvhead(GH)) : 128;
}

template <int GH, bool EXT>
__global__ void __launch_bounds__(merge_threads(GH)) gqa_mma_merge_kernel(const GqaParams p) {
  constexpr int D = 128;
  constexpr int HW = mma_warps_per_kvhead(GH);
  constexpr int GW = GH / HW;
  constexpr int HS = (kMmaWarps / HW) * GH;  // query heads per record
  constexpr int TG = 32 * GW;                // threads per group
  constexpr int NG = merge_threads(GH) / TG; // groups
  constexpr int RR = NG * kMergeBatch;       // records per round
  static_assert(RR <= merge_threads(GH), "one list entry per thread");
  __shared__ int64_t s_rec[RR];
  __shared__ float s_pm[NG][GW], s_pl[NG][GW];
  __shared__ float4 s_po[NG][TG];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int HN = p.n_chunks * p.n_hsub;
  const int nact = p.hc * HW;
  const int unit = static_cast<int>(blockIdx.x / nact), wi = static_cast<int>(blockIdx.x % nact);
  const int kh = wi / HW, hw = wi % HW;
  const int seq = unit / HN, idx = unit - seq * HN;
  const int chunk = idx / p.n_hsub, hsub = idx - chunk * p.n_hsub;
  const int* lst = p.unit_lists + static_cast<int64_t>(unit) * (1 + p.list_cap);
  const int t = threadIdx.x;
  // the count and the first round's entries together (entries past the count are ignored)
  const int first = (t < RR && t < p.list_cap) ? __ldcg(lst + 1 + t) : -1;
  int R = __ldcg(lst);
  if (R <= 0) return;  // nothing to merge: the decode kernel wrote the output
  R = R < p.list_cap ? R : p.list_cap;
  const int g = t / TG, q = t - g * TG, h = q >> 5, q4 = q & 31;
  const int hr = kh * GH + hw * GW + h;  // the head's slot in a record
  float M = kNegInf, Ls = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < R; base += RR) {
    if (base > 0) __syncthreads();
    if (t < RR) {
      const int e = base == 0 ? first : (base + t < R ? __ldcg(lst + 1 + base + t) : -1);
      // a slot outside the workspace (a list left by a call that gave up) is skipped
      s_rec[t] = (base + t < R && e >= 0 && e < p.rec_slots) ? e : -1;
    }
    __syncthreads();
    float mr[kMergeBatch], lr[kMergeBatch];
    float4 ov[kMergeBatch];
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      const int64_t rec = s_rec[i * NG + g];
      mr[i] = kNegInf;
      lr[i] = 0.f;
      ov[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rec >= 0) {
        const float* ml = p.rec_ml + (rec * HS + hr) * 2;
        mr[i] = __ldcg(ml);
        lr[i] = __ldcg(ml + 1);
        ov[i] = __ldcg(reinterpret_cast<const float4*>(p.rec_o + (rec * HS + hr) * D) + q4);
      }
    }
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      if (mr[i] == kNegInf) continue;
      if (mr[i] > M) {
        const float a = M == kNegInf ? 0.f : fast_exp2(M - mr[i]);
        Ls *= a;
        O.x *= a;
        O.y *= a;
        O.z *= a;
        O.w *= a;
        M = mr[i];
      }
      const float f = fast_exp2(mr[i] - M);
      Ls += f * lr[i];
      O.x += f * ov[i].x;
      O.y += f * ov[i].y;
      O.z += f * ov[i].z;
      O.w += f * ov[i].w;
    }
  }
  if (NG > 1) {
    if (q4 == 0) {
      s_pm[g][h] = M;
      s_pl[g][h] = Ls;
    }
    s_po[g][q] = O;
    __syncthreads();
    if (g != 0) return;
    float Mx = kNegInf;
#pragma unroll
    for (int j = 0; j < NG; ++j) Mx = fmaxf(Mx, s_pm[j][h]);
    Ls = 0.f;
    O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const float mj = s_pm[j][h];
      if (mj == kNegInf) continue;
      const float f = fast_exp2(mj - Mx);
      const float4 oj = s_po[j][q];
      Ls += f * s_pl[j][h];
      O.x += f * oj.x;
      O.y += f * oj.y;
      O.z += f * oj.z;
      O.w += f * oj.w;
    }
    M = Mx;
  }
  const int kvh = chunk * p.hc + kh, v = hsub * GH + hw * GW + h;
  const int64_t row = EXT ? out_row(p, seq, kvh, v) : static_cast<int64_t>(seq) * p.n_q_heads + kvh * p.group + v;
  const float inv = 1.0f / Ls;
  const float vals[4] = {O.x * inv, O.y * inv, O.z * inv, O.w * inv};
  store_out_vec<4>(p.out, row * D + 4 * q4, vals, p.out_dtype);
  if (EXT && p.lse != nullptr && q4 == 0) p.lse[row] = M + __log2f(Ls);
}

}  // namespace kvc
