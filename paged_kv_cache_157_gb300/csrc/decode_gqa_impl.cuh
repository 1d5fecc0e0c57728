// Paged decode attention for MHA / GQA / MQA on CUDA cores.
//
// What is computed (knowledge point 2 of "KV缓存原理与显存估算"): for each
// sequence i and query head h, with kv head h / g,
//     z_t = scale * q . k_t,   a = softmax(z) (max subtracted),   o = sum_t a_t v_t
// over the context_lens[i] rows gathered in logical order through the block
// table (PagedAttention, "KV Cache（键值缓存）" section 2.3).
//
// How (sm_103a):
// * Work unit = (kv head, sequence, head subgroup of GH <= 16 query heads).
//   All GH query heads of a unit share every K/V page that is loaded. A
//   stream of pages is consumed by one warp holding up to 4 heads; 8 or 16
//   heads split over 2 or 4 warps that consume the same stream (as a build
//   option, 2 or 4 heads split over a warp pair too).
// * Balanced split: the cache blocks of all units are laid end to end
//   (kv head major, then sequence, then subgroup, so units that read the
//   same pages sit next to each other) and CTA c takes blocks
//   [c*N/G, (c+1)*N/G). A CTA finishes whole units itself. A unit cut by a
//   range boundary leaves one fp32 record (max, sum, unnormalised output) per
//   CTA that touched it; the last of those CTAs to finish (a counter per unit
//   in the workspace, reset to zero by that CTA) merges the records with the
//   log-sum-exp rule. No CTA ever waits for another.
// * Each stream has its own ring of shared-memory stages: lane 0 of its
//   first warp issues 1-D bulk copies (TMA) of the K page and V page of a
//   block, completion counted on a "full" mbarrier (with a warp pair, both
//   warps release a stage on an "empty" mbarrier before it is refilled);
//   every wait is bounded. Stage and phase advance incrementally per tile.
// * Per 16-row tile a lane owns 16 (or 8) head dimensions of TL-strided rows.
//   Products use the packed fp32x2 FMA of sm_100+ (two fp32 lanes per
//   instruction, an IEEE fma in each). Partial dot products are reduced across
//   the lanes of a row with a reduce-scatter (each lane ends holding whole
//   scores of one head), softmax runs online in the log2 domain with a lazy
//   rescale (the reference maximum moves only when a score exceeds it by more
//   than 8, i.e. a factor 256), and the weights are gathered back for the V
//   accumulation in fp32.
#pragma once

#include <type_traits>

#include "decode_gqa.h"
#include "kvc_device.cuh"

namespace kvc {

template <typename T, int D, int GW>
struct GqaCfg {
  // Scores: a lane owns DPL head dimensions of RT rows of a 16-row tile.
  static constexpr int DPL = (D >= 64) ? 16 : 8;   // dims per lane
  static constexpr int DP2 = DPL / 2;               // fp32 pairs per lane
  static constexpr int DL = D / DPL;                // lanes per row
  static constexpr int TL = 32 / DL;                // row groups per warp
  static constexpr int RT = 16 / TL;                // rows per lane per tile
  static constexpr int VEC = Elem<T>::kVec;         // elements per 16-byte chunk
  static constexpr int NCH = DPL / VEC;             // chunks per lane per row
  // The RT rows are reduced in NS sets of SR rows: SR * GW partial scores
  // per set are reduce-scattered over the DL lanes of a row group.
  static constexpr int SR0 = DL / GW > 2 ? DL / GW : 2;
  static constexpr int SR = SR0 < RT ? SR0 : RT;    // rows per set
  static constexpr int NS = RT / SR;                // sets per tile
  static constexpr int NV = SR * GW;                // partial scores per set
  static constexpr int NVF = NV >= DL ? NV / DL : 1;  // whole scores per lane per set
  static constexpr int DUP = NV >= DL ? 1 : DL / NV;  // lanes holding the same score
  // Weighted sum of V: a lane owns VD dims of every row of its row group.
  static constexpr int VL = D >= 64 ? 32 : D / 2;   // lanes per V row
  static constexpr int VG = 32 / VL;                // V row groups
  static constexpr int VD = D / VL;                 // dims per lane: 2, 4 or 8
  static constexpr int NPAIR = 8 / VG;              // row pairs per lane per tile
  static_assert(DL * DPL == D && TL * DL == 32 && RT * TL == 16, "lane layout");
  static_assert(NCH * VEC == DPL, "chunking");
  static_assert(NS * SR == RT && SR % NVF == 0, "a lane's scores must belong to one head");
  static_assert(VL * VD == D && VG * VL == 32, "V lane layout");
};

// Rows of sequence b that are cached (capped by the table width; 0 if its
// length is invalid, i.e. below min_len: 1, or the number of new query tokens).
__device__ __forceinline__ int seq_rows(const int32_t* lens, int b, int bs, int max_blocks, int min_len = 1) {
  const int n = __ldg(lens + b);
  if (n < min_len || n < 1) return 0;
  const int cap = bs * max_blocks;
  return n < cap ? n : cap;
}

// First visible row of a sequence of `rows` cached rows: with a sliding
// window of W rows (W > 0) the newest W rows, [rows - W, rows), are attended.
__device__ __forceinline__ int first_row(int rows, int window) {
  return (window > 0 && rows > window) ? rows - window : 0;
}

// First visible row of sequence b: from the window, or, when row_div > 0,
// the start row row_start[b / row_div] (a shared prefix that another pass
// covers), capped at `rows`.
__device__ __forceinline__ int start_row(int rows, int window, const int32_t* row_start, int row_div, int b) {
  if (row_div > 0) {
    const int r = __ldg(row_start + b / row_div);
    return r < 0 ? 0 : (r < rows ? r : rows);
  }
  return first_row(rows, window);
}

// Number of cache blocks sequence b contributes: the blocks holding visible
// rows (0 if its length is invalid or no row is visible).
__device__ __forceinline__ int seq_blocks(const int32_t* lens, int b, int bs, int max_blocks, int window,
                                          int min_len, const int32_t* row_start, int row_div) {
  const int rows = seq_rows(lens, b, bs, max_blocks, min_len);
  if (rows == 0) return 0;
  const int r0 = start_row(rows, window, row_start, row_div, b);
  if (r0 >= rows) return 0;
  return (rows + bs - 1) / bs - r0 / bs;
}

// Exclusive prefix sums of seq_blocks over the batch into s_scan[0..B];
// the whole CTA participates. s_scan needs B + 1 + 32 ints.
__device__ inline void scan_blocks(const int32_t* lens, int B, int bs, int max_blocks, int window, int min_len,
                                   const int32_t* row_start, int row_div, int* s_scan) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (B + nt - 1) / nt;
  const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += seq_blocks(lens, b, bs, max_blocks, window, min_len, row_start, row_div);
  const int lane = tid & 31, wid = tid >> 5;
  int v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  int* wsum = s_scan + B + 1;
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
    if (lane < nw) wsum[lane] = x;  // inclusive
  }
  __syncthreads();
  int run = v - local + (wid > 0 ? wsum[wid - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    s_scan[b] = run;
    run += seq_blocks(lens, b, bs, max_blocks, window, min_len, row_start, row_div);
  }
  if (b1 == B && b0 < B) s_scan[B] = run;
  if (B == 0 && tid == 0) s_scan[0] = 0;
  __syncthreads();
}

// CTA whose block range [c*N/G, (c+1)*N/G) contains global block b.
__device__ __forceinline__ int64_t cta_of_block(int64_t b, int64_t G, int64_t N) { return ((b + 1) * G - 1) / N; }
__device__ __forceinline__ int64_t cta_range_start(int64_t c, int64_t G, int64_t N) { return c * N / G; }

// Reduce-scatter of CUR partial values across the lanes of a row group
// (xor masks B, B/2, ..., 1) without selects: every lane keeps the lower
// half of its registers and sends the upper half. This is correct because a
// lane whose mask bit is set stores its partial values with the two halves
// swapped at that level (register slot p holds logical value p ^ (NVF * dq)),
// so the partner's upper half is exactly the logical half this lane keeps.
// Once one value is left the remaining steps all-reduce it.
template <int CUR, int B>
struct ReduceScatter {
  __device__ __forceinline__ static void run(float* s) {
    if constexpr (B >= 1) {
      if constexpr (CUR > 1) {
        constexpr int H = CUR / 2;
#pragma unroll
        for (int t = 0; t < H; ++t) s[t] += __shfl_xor_sync(0xffffffffu, s[t + H], B);
        ReduceScatter<H, B / 2>::run(s);
      } else {
        s[0] += __shfl_xor_sync(0xffffffffu, s[0], B);
        ReduceScatter<1, B / 2>::run(s);
      }
    }
  }
};

// Per-lane geometry of the tile loops, fixed for the whole kernel.
template <typename T, int D, int GW>
struct LaneGeo {
  using C = GqaCfg<T, D, GW>;
  int kofs[C::SR];  // element offset of the K row held in register slot r (set 0), plus the lane's dims
  int mh;           // query-head permutation: register slot h holds head h ^ mh
  int h_lane;       // head of the whole scores this lane holds after the reduction
  int prow[C::NVF]; // tile row of score k of set 0 (set s adds s)
  int vofs;         // element offset of the lane's V dims in row 0 of its row group
  int vg;           // V row group
  __device__ __forceinline__ void init(int lane) {
    const int tq = lane / C::DL, dq = lane % C::DL;
    const int M = C::NVF * (dq / C::DUP);  // logical index of register slot p is p ^ M
    const int mr = M % C::SR;
    mh = M / C::SR;
    h_lane = mh;
#pragma unroll
    for (int r = 0; r < C::SR; ++r) kofs[r] = (tq * C::RT + (r ^ mr) * C::NS) * D + dq * C::VEC;
#pragma unroll
    for (int k = 0; k < C::NVF; ++k) prow[k] = tq * C::RT + (mr + k) * C::NS;
    vg = lane / C::VL;
    vofs = (lane % C::VL) * C::VD;
  }
};

template <typename T, int D, int GW>
struct WarpState {
  using C = GqaCfg<T, D, GW>;
  float2 q[GW][C::DP2];      // query slot h = head h ^ mh, pre-scaled by scale*log2(e)
  float2 o[GW][C::VD];       // unnormalised output of head h, dim vofs+d: (even rows, odd rows)
  float m[GW];               // reference maximum (log2 units), warp-uniform
  float l;                   // partial sum of this lane's weights (head h_lane)
};

template <int GW>
__device__ __forceinline__ float select_head(const float (&v)[GW], int h) {
  float r = v[0];
#pragma unroll
  for (int i = 1; i < GW; ++i) r = (h == i) ? v[i] : r;
  return r;
}

// VD consecutive elements of T (VD even) as raw words; pair(i) returns
// elements 2i and 2i+1 as fp32.
template <typename T, int VD>
struct VRow {
  static constexpr int BYTES = VD * static_cast<int>(sizeof(T));
  static constexpr int NW = (BYTES + 3) / 4;
  uint32_t w[NW];
  __device__ __forceinline__ void load(const T* p) {
    if constexpr (BYTES == 2) {
      w[0] = *reinterpret_cast<const unsigned short*>(p);
    } else if constexpr (NW == 1) {
      w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else if constexpr (NW == 2) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      w[0] = u.x;
      w[1] = u.y;
    } else {
#pragma unroll
      for (int i = 0; i < NW; i += 4) {
        const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(p) + i);
        w[i] = u.x;
        w[i + 1] = u.y;
        w[i + 2] = u.z;
        w[i + 3] = u.w;
      }
    }
  }
  __device__ __forceinline__ float2 pair(int i) const {
    if constexpr (sizeof(T) == 4) {
      return make_float2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
    } else if constexpr (sizeof(T) == 2) {
      return make_float2(Elem<T>::half_to_float(w[i], 0), Elem<T>::half_to_float(w[i], 1));
    } else if constexpr (std::is_same<T, s8q>::value) {
      return s8x2_to_float2(w[i >> 1] >> (16 * (i & 1)));
    } else {
      return fp8x2_to_float2(w[i >> 1] >> (16 * (i & 1)));
    }
  }
  // INT8 codes: element d of this row and of row o as an fp32 pair, built
  // straight from the two rows' bytes (no repacking of same-row pairs; 4 %
  // faster. The same for e4m3, through a byte permute ahead of the hardware
  // conversion, was 3 % slower than converting same-row pairs.)
  __device__ __forceinline__ float2 cross(const VRow& o, int d) const {
    static_assert(std::is_same<T, s8q>::value, "int8 codes");
    const int b = d & 3;
    return s8_unbias(make_float2(s8_biased(s8_flip(w[d >> 2]), b), s8_biased(s8_flip(o.w[d >> 2]), b)));
  }
};

// One 16-row tile of a page: scores, online softmax, V accumulation.
// sp is this warp's [GW][16] fp32 weight buffer.
// PARTIAL tiles attend only rows [lo_valid, valid) of the 16, and the lane's
// head only those below vis (<= valid: with several new tokens an earlier
// token does not see the later ones' rows). For FP8
// caches vsp holds the tile's 16 per-token V scales: they multiply the
// weights that feed the V accumulation (the sum l keeps the unscaled ones).
template <typename T, int D, int GW, bool PARTIAL>
__device__ __forceinline__ void gqa_tile(const T* __restrict__ kp, const T* __restrict__ vp, float* sp,
                                         const float* __restrict__ vsp, int lo_valid, int valid, int vis,
                                         WarpState<T, D, GW>& st, const LaneGeo<T, D, GW>& g) {
  using C = GqaCfg<T, D, GW>;
  float sc[C::NS][C::NVF];
#pragma unroll
  for (int set = 0; set < C::NS; ++set) {
    // The SR rows' raw K chunks first, then the SR*GW accumulators advance
    // together over the lane's dims (independent FMA chains).
    uint4 kr[C::SR][C::NCH];
#pragma unroll
    for (int r = 0; r < C::SR; ++r) {
#pragma unroll
      for (int j = 0; j < C::NCH; ++j) kr[r][j] = lds128(kp + g.kofs[r] + set * D + C::DL * j * C::VEC);
    }
    float2 acc[C::SR][GW];
#pragma unroll
    for (int j = 0; j < C::NCH; ++j) {
#pragma unroll
      for (int c = 0; c < C::VEC / 2; ++c) {
        const int i = j * (C::VEC / 2) + c;
#pragma unroll
        for (int r = 0; r < C::SR; ++r) {
          const float2 kf = Elem<T>::pair(kr[r][j], c);
#pragma unroll
          for (int h = 0; h < GW; ++h) acc[r][h] = (i == 0) ? fmul2(st.q[h][0], kf) : ffma2(st.q[h][i], kf, acc[r][h]);
        }
      }
    }
    float s[C::NV];
#pragma unroll
    for (int h = 0; h < GW; ++h) {
#pragma unroll
      for (int r = 0; r < C::SR; ++r) s[h * C::SR + r] = acc[r][h].x + acc[r][h].y;
    }
    ReduceScatter<C::NV, C::DL / 2>::run(s);
#pragma unroll
    for (int k = 0; k < C::NVF; ++k) sc[set][k] = s[k];
  }

  float m_l = select_head<GW>(st.m, g.h_lane);
  bool need = false;
#pragma unroll
  for (int set = 0; set < C::NS; ++set) {
#pragma unroll
    for (int k = 0; k < C::NVF; ++k) {
      if (PARTIAL && (g.prow[k] + set >= vis || g.prow[k] + set < lo_valid)) sc[set][k] = kNegInf;
      need |= sc[set][k] > m_l + 8.0f;
    }
  }
  if (__any_sync(0xffffffffu, need)) {
    float loc = kNegInf;
#pragma unroll
    for (int set = 0; set < C::NS; ++set) {
#pragma unroll
      for (int k = 0; k < C::NVF; ++k) loc = fmaxf(loc, sc[set][k]);
    }
#pragma unroll
    for (int hh = 0; hh < GW; ++hh) {
      const float tmax = warp_max(g.h_lane == hh ? loc : kNegInf);
      const float mn = fmaxf(st.m[hh], tmax);
      const float alpha = fast_exp2(st.m[hh] - mn);
      const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
      for (int d = 0; d < C::VD; ++d) st.o[hh][d] = fmul2(st.o[hh][d], a2);
      if (g.h_lane == hh) st.l *= alpha;
      st.m[hh] = mn;
    }
    m_l = select_head<GW>(st.m, g.h_lane);
  }
  __syncwarp();  // the previous tile's reads of sp are done
#pragma unroll
  for (int set = 0; set < C::NS; ++set) {
#pragma unroll
    for (int k = 0; k < C::NVF; ++k) {
      const float pv = fast_exp2(sc[set][k] - m_l);
      st.l += pv;
      sc[set][k] = pv;
      if constexpr (sizeof(T) == 1) sc[set][k] = pv * vsp[g.prow[k] + set];
    }
  }
  if constexpr (C::NVF == 1 && C::NS == 2) {
    // the lane's two weights are adjacent rows
    *reinterpret_cast<float2*>(sp + g.h_lane * 16 + g.prow[0]) = make_float2(sc[0][0], sc[1][0]);
  } else {
#pragma unroll
    for (int set = 0; set < C::NS; ++set) {
#pragma unroll
      for (int k = 0; k < C::NVF; ++k) sp[g.h_lane * 16 + g.prow[k] + set] = sc[set][k];
    }
  }
  __syncwarp();

  // o[h][d] += (p[h][2k], p[h][2k+1]) * (v[2k][d], v[2k+1][d]): one packed
  // FMA covers a row pair, so no weight or value needs duplicating.
  float4 p4[GW];
#pragma unroll
  for (int kk = 0; kk < C::NPAIR; ++kk) {
    const int k = kk * C::VG + g.vg;  // row pair
    VRow<T, C::VD> va, vb;
    va.load(vp + (2 * k) * D + g.vofs);
    vb.load(vp + (2 * k + 1) * D + g.vofs);
    float2 pp[GW];
    if constexpr (C::VG == 1) {
      // weights of row pairs k and k + 1 in one 16-byte load (sp is 16-byte aligned)
      if ((kk & 1) == 0) {
#pragma unroll
        for (int h = 0; h < GW; ++h) p4[h] = *reinterpret_cast<const float4*>(sp + h * 16 + 2 * k);
      }
#pragma unroll
      for (int h = 0; h < GW; ++h) pp[h] = (kk & 1) ? make_float2(p4[h].z, p4[h].w) : make_float2(p4[h].x, p4[h].y);
    } else {
#pragma unroll
      for (int h = 0; h < GW; ++h) pp[h] = *reinterpret_cast<const float2*>(sp + h * 16 + 2 * k);
    }
    const bool za = PARTIAL && (2 * k >= valid || 2 * k < lo_valid);
    const bool zb = PARTIAL && (2 * k + 1 >= valid || 2 * k + 1 < lo_valid);
#pragma unroll
    for (int dp = 0; dp < C::VD / 2; ++dp) {
      float2 a, b;
      if constexpr (!std::is_same<T, s8q>::value) {
        a = va.pair(dp);
        b = vb.pair(dp);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int d = 2 * dp + e;
        float2 v;
        if constexpr (std::is_same<T, s8q>::value)
          v = va.cross(vb, d);
        else
          v = e == 0 ? make_float2(a.x, b.x) : make_float2(a.y, b.y);
        if (PARTIAL) {
          // rows outside the attended range may hold anything (even NaN): their weight is 0
          if (za) v.x = 0.f;
          if (zb) v.y = 0.f;
        }
#pragma unroll
        for (int h = 0; h < GW; ++h) st.o[h][d] = ffma2(pp[h], v, st.o[h][d]);
      }
    }
  }
}

// Worker whose block range [w*N/W, (w+1)*N/W) contains global block b, and
// the first block of worker w's range.
__device__ __forceinline__ int64_t worker_of_block(int64_t b, int64_t W, int64_t N) { return ((b + 1) * W - 1) / N; }
__device__ __forceinline__ int64_t worker_range_start(int64_t w, int64_t W, int64_t N) { return w * N / W; }

// Global position -> (sequence, kv-head chunk, head subgroup, block of the
// sequence). Positions are numbered sequence major, then chunk, then
// subgroup, then block: gb = HN * scan[seq] + (chunk * n_hsub + hsub) * nb + j
// with HN = n_chunks * n_hsub; s_scan holds the exclusive prefix sums of the
// per-sequence block counts.
struct BlockPos {
  int chunk, seq, hsub, j, nb;
};

__device__ __forceinline__ BlockPos locate_block(int64_t gb, int HN, const int* s_scan, int B, int n_hsub) {
  BlockPos r;
  int a = 0, b = B - 1;  // largest sequence with HN * S[seq] <= gb (skips empty ones)
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (static_cast<int64_t>(HN) * s_scan[mid] <= gb) a = mid; else b = mid - 1;
  }
  r.seq = a;
  r.nb = s_scan[a + 1] - s_scan[a];
  const int r2 = static_cast<int>(gb - static_cast<int64_t>(HN) * s_scan[a]);
  const int idx = r2 / r.nb;
  r.chunk = idx / n_hsub;
  r.hsub = idx - r.chunk * n_hsub;
  r.j = r2 - idx * r.nb;
  return r;
}

// Row of `out` ([batch, n_tok, n_q_heads, D], flattened over rows) that holds
// virtual query head v of kv head kvh: with several new tokens per sequence
// the n_tok * group queries of a kv head are its virtual heads, v = t * group
// + j (token t, query head j of the group).
__device__ __forceinline__ int64_t out_row(const GqaParams& p, int seq, int kvh, int v) {
  const int t = v / p.group, j = v - t * p.group;
  return (static_cast<int64_t>(seq) * p.n_tok + t) * p.n_q_heads + kvh * p.group + j;
}

// Record slot that worker c left for the unit whose first block is u0: 2c
// if the unit's part in c starts at c's first block, else 2c + 1. Returns
// -1 for a worker with an empty range (only when N < W).
__device__ __forceinline__ int64_t record_of(int64_t c, int64_t c0, int64_t u0, int64_t f00, int64_t W, int64_t N) {
  if (N >= W) return 2 * c + ((c == c0 && u0 > f00) ? 1 : 0);
  const int64_t f0 = worker_range_start(c, W, N), f1 = worker_range_start(c + 1, W, N);
  if (f0 == f1) return -1;
  return 2 * c + (u0 > f0 ? 1 : 0);
}

// One warp merges, for its GW heads of a unit (first block u0, nb blocks),
// the records of every worker that touched the unit, with the log-sum-exp
// rule, and writes the normalised output. Records are taken RG at a time:
// lane r loads the (max, sum) pairs of record r while every lane loads its
// chunks of the group's output rows, so one round trip serves the group.
// Lane L owns the float4 chunks L + 32k of the warp's GW x D outputs.
template <int D, int HS, int GW, bool EXT>
__device__ void merge_unit_warp(const GqaParams& p, int64_t u0, int nb, int64_t W, int64_t N, int seq, int kvh, int v0,
                                int hoff, int lane) {
  constexpr int CH = D / 4;                  // float4 chunks per head
  constexpr int NCK = (GW * CH + 31) / 32;   // chunks per lane
  constexpr int RG = NCK <= 4 ? 8 : 4;       // records in flight together
  const int64_t c0 = worker_of_block(u0, W, N), c1 = worker_of_block(u0 + nb - 1, W, N);
  const int64_t f00 = worker_range_start(c0, W, N);
  const int span = static_cast<int>(c1 - c0 + 1);
  const float* rbase = p.rec_o + static_cast<int64_t>(hoff) * D + 4 * lane;
  float M[GW], Lp[GW];
  float4 O[NCK];
#pragma unroll
  for (int h = 0; h < GW; ++h) {
    M[h] = kNegInf;
    Lp[h] = 0.f;
  }
#pragma unroll
  for (int k = 0; k < NCK; ++k) O[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < span; base += RG) {
    const int n = min(RG, span - base);
    // lanes r < n: (max, sum) of record base + r
    const int64_t rec = (lane < n) ? record_of(c0 + base + lane, c0, u0, f00, W, N) : -1;
    float mr[GW], lr[GW];
#pragma unroll
    for (int h = 0; h < GW; ++h) {
      const float* ml = p.rec_ml + (rec * HS + hoff + h) * 2;
      mr[h] = rec >= 0 ? __ldcg(ml) : kNegInf;
      lr[h] = rec >= 0 ? __ldcg(ml + 1) : 0.f;
    }
    // every lane: its chunks of the group's output rows
    float4 ov[RG][NCK];
#pragma unroll
    for (int i = 0; i < RG; ++i) {
      const int64_t rr = __shfl_sync(0xffffffffu, rec, i);
#pragma unroll
      for (int k = 0; k < NCK; ++k) {
        const bool ok = i < n && rr >= 0 && lane + 32 * k < GW * CH;
        ov[i][k] = ok ? __ldcg(reinterpret_cast<const float4*>(rbase + rr * HS * D + 128 * k))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float fr[GW];
#pragma unroll
    for (int h = 0; h < GW; ++h) {
      const float mn = fmaxf(M[h], warp_max(mr[h]));
      if (mn != M[h]) {
        const float a = (M[h] == kNegInf) ? 0.f : fast_exp2(M[h] - mn);
        Lp[h] *= a;
#pragma unroll
        for (int k = 0; k < NCK; ++k) {
          if (((lane + 32 * k) / CH) == h) {
            O[k].x *= a;
            O[k].y *= a;
            O[k].z *= a;
            O[k].w *= a;
          }
        }
        M[h] = mn;
      }
      fr[h] = (mr[h] == kNegInf) ? 0.f : fast_exp2(mr[h] - M[h]);
      Lp[h] += fr[h] * lr[h];
    }
#pragma unroll
    for (int i = 0; i < RG; ++i) {
      float fh[GW];
#pragma unroll
      for (int h = 0; h < GW; ++h) fh[h] = __shfl_sync(0xffffffffu, fr[h], i);
#pragma unroll
      for (int k = 0; k < NCK; ++k) {
        float f = 0.f;
#pragma unroll
        for (int h = 0; h < GW; ++h) f = ((lane + 32 * k) / CH == h) ? fh[h] : f;
        O[k].x += f * ov[i][k].x;
        O[k].y += f * ov[i][k].y;
        O[k].z += f * ov[i][k].z;
        O[k].w += f * ov[i][k].w;
      }
    }
  }
  float inv[GW];
#pragma unroll
  for (int h = 0; h < GW; ++h) {
    const float lsum = warp_sum(Lp[h]);
    inv[h] = 1.0f / lsum;
    if (EXT && p.lse != nullptr && lane == 0) p.lse[out_row(p, seq, kvh, v0 + h)] = M[h] + __log2f(lsum);
  }
#pragma unroll
  for (int k = 0; k < NCK; ++k) {
    const int idx = lane + 32 * k;
    if (idx >= GW * CH) break;
    float iv = 0.f;
#pragma unroll
    for (int h = 0; h < GW; ++h) iv = (idx / CH == h) ? inv[h] : iv;
    const int64_t o = EXT ? out_row(p, seq, kvh, v0 + idx / CH) * D + 4 * (idx % CH)
                          : (static_cast<int64_t>(seq) * p.n_q_heads + kvh * p.group + v0) * D + 4 * idx;
    store_out(p.out, o, O[k].x * iv, p.out_dtype);
    store_out(p.out, o + 1, O[k].y * iv, p.out_dtype);
    store_out(p.out, o + 2, O[k].z * iv, p.out_dtype);
    store_out(p.out, o + 3, O[k].w * iv, p.out_dtype);
  }
}

// Shared-memory atomic add with acquire-release semantics at CTA scope: the
// reads of a stage that precede it (ordered by a warp barrier) happen before
// the refill that the last releasing warp issues after it.
__device__ __forceinline__ unsigned int atomic_add_acq_rel_cta_smem(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v) : "memory");
  return old;
}

// EXT: the extensions (sliding window, several new query tokens per
// sequence) are compiled in only where they are used, so the single-token
// full-attention kernel keeps no per-block bookkeeping for them.
//
// With n_tok new tokens the queries of a kv head are its n_tok * group
// "virtual heads" v = t * group + j; they share every page. Token t sits at
// position n - n_tok + t of a sequence of n cached rows and attends rows
// [0, n - n_tok + t], so virtual head v hides the last n_tok - 1 - t rows.
template <typename T, int D, int GH, typename TQ, bool EXT>
__global__ void __launch_bounds__(kGqaWarps * 32, kGqaCtasPerSm) gqa_decode_kernel(const GqaParams p) {
  constexpr int HW = gqa_warps_per_kvhead(GH);  // warps per kv head
  constexpr int GW = GH / HW;                    // query heads per warp
  constexpr int HCM = kGqaWarps / HW;            // kv heads per CTA at most
  constexpr int HS = HCM * GH;                   // query heads per record
  using C = GqaCfg<T, D, GW>;
  static_assert(GW * HW == GH && kGqaWarps % HW == 0, "head split over the warps of a kv head");
  static_assert(D % 32 == 0, "merge lanes own D / 32 dims");
  extern __shared__ __align__(128) unsigned char smem[];
  const int hc = p.hc;
  constexpr bool kFp8 = sizeof(T) == 1;
  const int wnd = EXT ? p.window : 0;   // sliding window rows (0: all)
  const int n_tok = EXT ? p.n_tok : 1;  // new query tokens per sequence
  const bool causal = !EXT || p.causal != 0;
  const int tm = causal ? n_tok - 1 : 0;  // rows hidden from the first of them
  const int min_len = causal ? n_tok : 1;  // shortest valid context
  const bool multi = EXT && n_tok > 1;
  const int32_t* row_start = EXT ? p.row_start : nullptr;
  const int row_div = EXT ? p.row_div : 0;
  constexpr int VSB = kFp8 ? 4 : 0;  // V-scale bytes per cached row
  const GqaSmem L = gqa_smem_layout(sizeof(T), sizeof(TQ), VSB, D, GH, p.block_size, hc, p.stages, p.batch);
  unsigned char* s_stage = smem + L.stage_off;
  uint64_t* fbar = reinterpret_cast<uint64_t*>(smem + L.bar_off);  // [S] full
  unsigned int* s_rel = reinterpret_cast<unsigned int*>(smem + L.rel_off);  // [S] releases seen
  unsigned int* s_iss = s_rel + p.stages;  // [S] fills issued
  volatile int* s_misc = reinterpret_cast<volatile int*>(smem + L.misc_off);  // [abort flag]
  int* s_scan = reinterpret_cast<int*>(smem + L.scan_off);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int kh = w / HW, hw = w % HW;  // kv head of the chunk and share of its query heads
  const int nact = hc * HW;            // warps with work
  const bool active = w < nact;
  LaneGeo<T, D, GW> geo;
  geo.init(lane);
  const int bs = p.block_size, S = p.stages;
  const int B = p.batch;
  const int tiles_per_page = bs / 16;
  const int page_elems = bs * D;
  const int chunk_elems = hc * page_elems;
  // stage: [K chunk][V chunk][the unit's query rows (TQ)][FP8: the chunk's V scales]
  const uint32_t page_bytes = static_cast<uint32_t>(page_elems * sizeof(T));
  const uint32_t chunk_bytes = static_cast<uint32_t>(chunk_elems * sizeof(T));
  const uint32_t q_bytes = static_cast<uint32_t>(hc * GH * D * sizeof(TQ));
  const uint32_t vs_bytes = static_cast<uint32_t>(hc * bs * VSB);
  const size_t stage_bytes = align_up(2 * chunk_bytes + q_bytes + vs_bytes, 16);
  const T* kc = static_cast<const T*>(p.k_cache);
  const T* vc = static_cast<const T*>(p.v_cache);
  const TQ* qg = static_cast<const TQ*>(p.q);
  const uint32_t full = 0xffffffffu;
  const int HN = p.n_chunks * p.n_hsub;
  const bool q_contig = (GH == p.group);  // the chunk's query rows are one contiguous run

  if (tid < S) {
    mbar_init(fbar + tid, 1);  // one arrive (with the copy bytes) per fill
    s_rel[tid] = 0u;
    s_iss[tid] = 0u;
  }
  if (tid == 0) {
    s_misc[0] = 0;
    s_misc[1] = 0;
    s_misc[2] = 0;
  }
  fence_barrier_init();
  // Launched right behind the previous kernel of the stream (programmatic
  // stream serialisation: the append of this step, or whatever wrote the
  // lengths, tables or queries on the device), the kernel becomes resident and
  // sets up its barriers while that grid runs. Every thread then waits for
  // the grid to finish (its writes become visible) before it reads or writes
  // any caller buffer.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid < 2 && !p.unit_mode) {
    // Warm L2 with the block-table line this CTA most likely reads first (a
    // guess that assumes equal lengths; it only overlaps the length scan).
    const int64_t Gc = gridDim.x;
    const int64_t per_seq = static_cast<int64_t>(HN) * p.max_blocks;
    const int64_t pos = static_cast<int64_t>(blockIdx.x) * B * per_seq / Gc;
    const int seq = static_cast<int>(pos / per_seq);
    const int j = static_cast<int>((pos - seq * per_seq) % p.max_blocks) + tid * 32;
    if (seq < B && j < p.max_blocks) prefetch_l2(p.block_tables + static_cast<int64_t>(seq) * p.max_blocks + j);
  }
  scan_blocks(p.context_lens, B, bs, p.max_blocks, wnd, min_len, row_start, row_div, s_scan);  // ends with a CTA barrier
  const int64_t N = static_cast<int64_t>(HN) * s_scan[B];
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;

  if (blockIdx.x == 0) {
    // Validate every length once; in the split mode CTA 0 also writes the
    // zero outputs of sequences with no visible row (an invalid length, or
    // every row before the start row): no CTA visits them.
    int empty = 0;
    for (int b = tid; b < B; b += blockDim.x) {
      const int n = __ldg(p.context_lens + b);
      if (n < min_len || n > bs * p.max_blocks) set_flag(p.err, 0x2u);
      if (row_div > 0 && __ldg(row_start + b / row_div) > n) set_flag(p.err, 0x2u);
      empty |= (s_scan[b + 1] == s_scan[b]) ? 1 : 0;
    }
    if (__syncthreads_or(empty) && !p.unit_mode) {
      const int rows = n_tok * p.n_q_heads * D;  // outputs of one sequence
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
    // CTA u takes unit u = (sequence, chunk, subgroup) whole
    const int seq = static_cast<int>(c / HN);
    const int idx = static_cast<int>(c - static_cast<int64_t>(seq) * HN);
    const int nb = s_scan[seq + 1] - s_scan[seq];
    if (nb == 0) {
      // no visible row (invalid length, or all before the start row): zero
      // output for this CTA's heads
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
  const int total = static_cast<int>(hi - lo);  // positions of this CTA
  if (total <= 0) return;                       // uniform over the CTA

  unsigned char* my_k = s_stage + kh * page_bytes;  // + slot * stage_bytes
  unsigned char* my_v = s_stage + chunk_bytes + kh * page_bytes;
  float* wp = reinterpret_cast<float*>(smem + L.p_off) + w * GW * 16;  // this warp's weights
  const uint64_t pol = policy_evict_first();

  // Positions lo + 32*win + lane, one per lane: the page index (block *
  // n_kv_heads + first kv head of the chunk; -1 if the table entry is out of
  // range) and, for the first block of a segment, the element offset of the
  // unit's first query row, or with several new tokens the unit's index
  // (-1 otherwise).
  auto window = [&](int win, int& src, int& qoff) {
    const int64_t pos = lo + static_cast<int64_t>(win) * 32 + lane;
    src = -1;
    qoff = -1;
    if (pos < hi) {
      const BlockPos bp = locate_block(pos, HN, s_scan, B, p.n_hsub);
      // bp.j counts the sequence's visible blocks; the table is indexed from block 0
      const int j0 =
          start_row(seq_rows(p.context_lens, bp.seq, bs, p.max_blocks, min_len), wnd, row_start, row_div, bp.seq) /
          bs;
      const int phys = __ldg(p.block_tables + static_cast<int64_t>(bp.seq) * p.max_blocks + j0 + bp.j);
      if (phys >= 0 && phys < p.num_blocks) src = phys * p.n_kv_heads + bp.chunk * hc;
      if (pos == lo || bp.j == 0)
        qoff = multi ? (bp.seq * p.n_chunks + bp.chunk) * p.n_hsub + bp.hsub
                     : (bp.seq * p.n_q_heads + bp.chunk * hc * p.group + bp.hsub * GH) * D;
    }
  };
  // Copies of one position into stage `slot` (one thread).
  auto issue = [&](int slot, int src, int qoff) {
    const uint32_t bytes = (src >= 0 ? 2 * chunk_bytes + vs_bytes : 0u) + (qoff >= 0 ? q_bytes : 0u);
    if (src < 0) set_flag(p.err, 0x1u);
    atomicAdd(s_iss + slot, 1u);
    if (bytes == 0) {
      mbar_arrive(fbar + slot);
      return;
    }
    unsigned char* dst = s_stage + static_cast<size_t>(slot) * stage_bytes;
    mbar_arrive_expect_tx(fbar + slot, bytes);
    if (src >= 0) {
      const int64_t e = static_cast<int64_t>(src) * page_elems;
      bulk_g2s(dst, kc + e, chunk_bytes, fbar + slot, pol);
      bulk_g2s(dst + chunk_bytes, vc + e, chunk_bytes, fbar + slot, pol);
      if constexpr (kFp8)  // the V scales of the chunk's rows: [hc heads][bs rows]
        bulk_g2s(dst + 2 * chunk_bytes + q_bytes, p.v_scale + static_cast<int64_t>(src) * bs, vs_bytes, fbar + slot,
                 pol);
    }
    if (qoff >= 0) {
      if (multi) {
        // The unit's GH virtual heads of each kv head, v = t * group + j, are
        // query rows (seq, t, kv head * group + j): one copy per run of one token.
        const int hs = qoff % p.n_hsub, rest = qoff / p.n_hsub;
        const int ch = rest % p.n_chunks, sq = rest / p.n_chunks;
        const uint32_t rowb = static_cast<uint32_t>(D * sizeof(TQ));
        for (int h = 0; h < hc; ++h) {
          const int kvh = ch * hc + h;
          for (int v = hs * GH, ve = v + GH; v < ve;) {
            const int t = v / p.group, j = v - t * p.group;
            const int len = min(p.group - j, ve - v);
            const int64_t row = (static_cast<int64_t>(sq) * n_tok + t) * p.n_q_heads + kvh * p.group + j;
            bulk_g2s(dst + 2 * chunk_bytes + (h * GH + v - hs * GH) * rowb, qg + row * D, len * rowb, fbar + slot,
                     pol);
            v += len;
          }
        }
      } else if (q_contig) {
        bulk_g2s(dst + 2 * chunk_bytes, qg + qoff, q_bytes, fbar + slot, pol);
      } else {
        const uint32_t rb = static_cast<uint32_t>(GH * D * sizeof(TQ));
        for (int h = 0; h < hc; ++h)
          bulk_g2s(dst + 2 * chunk_bytes + h * rb, qg + qoff + h * p.group * D, rb, fbar + slot, pol);
      }
    }
  };

  int w_src0, w_src1 = -1, w_q0, w_q1 = -1;
  window(0, w_src0, w_q0);
  if (total > 32) window(1, w_src1, w_q1);

  // Warp 0 fills the first S stages; after that the warp that releases a
  // stage last (its release count reaches nact per fill) refills it, so no
  // warp waits for another except through the "full" barriers.
  const int n_first = total < S ? total : S;
  if (w == 0) {
    for (int i = 0; i < n_first; ++i) {
      const int src = __shfl_sync(full, w_src0, i);
      const int qo = __shfl_sync(full, w_q0, i);
      if (lane == 0) issue(i, src, qo);
    }
  }
  __syncwarp();

  // Partial segments (at most two: the one starting at lo, the one ending
  // at hi) whose records wait to be counted.
  bool pend0 = false, pend1 = false;
  unsigned int old0 = 0, old1 = 0;  // the counts seen by this warp's adds (lane 0)
  bool aborted = false;

  if (active) {
    int slot = 0;
    uint32_t par = 0, fill = 0;  // phase parity and fill number of `slot`
    int cpos = 0;                // positions consumed
    int64_t gb = lo;
    while (gb < hi) {
      // ---- segment: the part of one unit inside [lo, hi)
      const BlockPos sg = locate_block(gb, HN, s_scan, B, p.n_hsub);
      const int seg_len = static_cast<int>(((sg.nb - sg.j) < (hi - gb)) ? (sg.nb - sg.j) : (hi - gb));
      const int n_rows = seq_rows(p.context_lens, sg.seq, bs, p.max_blocks, min_len);
      const int r0 = start_row(n_rows, wnd, row_start, row_div, sg.seq);  // first visible row
      const int j0 = r0 / bs;                      // table index of the first visible block
      const int kvh = sg.chunk * hc + kh;          // kv head of this warp
      const int v0 = sg.hsub * GH + hw * GW;       // first (virtual) query head of this warp
      const int hq0 = kvh * p.group + v0;          // its query head (single token)
      const int dh = (EXT && causal) ? tm - (v0 + geo.h_lane) / p.group : 0;  // last rows the lane's head may not see

      WarpState<T, D, GW> st;
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
        const bool ok = mbar_wait_data(fbar + slot, par, p.wait_polls);
        if (__any_sync(full, !ok) || s_misc[0]) {
          if (lane == 0) {
            set_flag(p.err, 0x8u);
            s_misc[0] = 1;
          }
          aborted = true;
          break;
        }
        const unsigned char* stg = s_stage + static_cast<size_t>(slot) * stage_bytes;
        if (t == 0) {
          // The unit's query rows came with its first position. Register slot
          // h holds head h ^ mh (the lane's reduction order); the lane's dims
          // are C::VEC-element runs at (dq + DL * j) * C::VEC. FP8 caches fold
          // the per-channel K scales into the query.
          const int d0 = geo.kofs[0] % D;  // first dim of the lane's first run
          const TQ* qs = reinterpret_cast<const TQ*>(stg + 2 * chunk_bytes) + (kh * GH + hw * GW) * D + d0;
          constexpr int QV = Elem<TQ>::kVec;  // query elements per 16-byte load
          float ksc[C::DPL];
#pragma unroll
          for (int i = 0; i < C::DPL; ++i) ksc[i] = p.qscale;
          if constexpr (kFp8) {
            const float* ks = p.k_scale + static_cast<int64_t>(sg.chunk * hc + kh) * D + d0;
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
#pragma unroll
              for (int e = 0; e < C::VEC; e += 4) {
                const float4 k4 = __ldg(reinterpret_cast<const float4*>(ks + C::DL * j * C::VEC + e));
                ksc[j * C::VEC + e] *= k4.x;
                ksc[j * C::VEC + e + 1] *= k4.y;
                ksc[j * C::VEC + e + 2] *= k4.z;
                ksc[j * C::VEC + e + 3] *= k4.w;
              }
            }
          }
#pragma unroll
          for (int h = 0; h < GW; ++h) {
            float f[C::DPL];
            const TQ* qh = qs + (h ^ geo.mh) * D;
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
#pragma unroll
              for (int e = 0; e < C::VEC; e += QV) Elem<TQ>::unpack(lds128(qh + C::DL * j * C::VEC + e), f + j * C::VEC + e);
            }
#pragma unroll
            for (int i = 0; i < C::DP2; ++i) st.q[h][i] = make_float2(f[2 * i] * ksc[2 * i], f[2 * i + 1] * ksc[2 * i + 1]);
#pragma unroll
            for (int d = 0; d < C::VD; ++d) st.o[h][d] = make_float2(0.f, 0.f);
            // With several tokens a head may meet only rows it may not see in
            // a segment; a finite start keeps exp2(score - max) at 0 there.
            st.m[h] = EXT ? -1e30f : kNegInf;
          }
          st.l = 0.f;
        }
        if (src >= 0) {
          const T* kp = reinterpret_cast<const T*>(my_k + static_cast<size_t>(slot) * stage_bytes);
          const T* vp = reinterpret_cast<const T*>(my_v + static_cast<size_t>(slot) * stage_bytes);
          const float* vsp = reinterpret_cast<const float*>(stg + 2 * chunk_bytes + q_bytes) + kh * bs;
          const int jb = j0 + sg.j + t;                          // table index of this block
          const int rb = n_rows - jb * bs;                       // rows from the block's first to the end
          const int vr = min(bs, rb);                            // rows of the block before the end
          const int lr = (jb == j0) ? r0 - j0 * bs : 0;          // rows of the block before the window
          if (rb - tm >= bs && lr == 0) {
            for (int tt = 0; tt < tiles_per_page; ++tt)
              gqa_tile<T, D, GW, false>(kp + tt * 16 * D, vp + tt * 16 * D, wp, vsp + tt * 16, 0, 16, 16, st, geo);
          } else {
            for (int tt = 0; tt < tiles_per_page; ++tt) {
              const int valid = vr - tt * 16, lo_valid = lr - tt * 16;
              const int rt = rb - tt * 16;  // rows from the tile's first to the end
              if (valid <= 0) break;
              if (lo_valid >= 16) continue;
              if (rt - tm >= 16 && lo_valid <= 0)
                gqa_tile<T, D, GW, false>(kp + tt * 16 * D, vp + tt * 16 * D, wp, vsp + tt * 16, 0, 16, 16, st, geo);
              else
                gqa_tile<T, D, GW, true>(kp + tt * 16 * D, vp + tt * 16 * D, wp, vsp + tt * 16, lo_valid, valid,
                                         EXT ? min(valid, rt - dh) : valid, st, geo);
            }
          }
        }
        // Every shared-memory read of this stage fed an instruction issued
        // before this barrier, so none is outstanding once it is released.
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

      // ---- finish the segment: this warp holds every row of it for its heads
      float ov[GW][C::VD];
#pragma unroll
      for (int h = 0; h < GW; ++h) {
#pragma unroll
        for (int d = 0; d < C::VD; ++d) {
          float v = st.o[h][d].x + st.o[h][d].y;
#pragma unroll
          for (int msk = C::VL; msk < 32; msk <<= 1) v += __shfl_xor_sync(full, v, msk);
          ov[h][d] = v;
        }
      }
      float lw[GW];
#pragma unroll
      for (int hh = 0; hh < GW; ++hh) lw[hh] = warp_sum(geo.h_lane == hh ? st.l : 0.f) * (1.0f / C::DUP);
      const bool whole = (sg.j == 0 && seg_len == sg.nb);
      if (whole) {
        if (geo.vg == 0) {
#pragma unroll
          for (int h = 0; h < GW; ++h) {
            const float inv = 1.0f / lw[h];
            const int64_t ob = (EXT ? out_row(p, sg.seq, kvh, v0 + h)
                                    : static_cast<int64_t>(sg.seq) * p.n_q_heads + hq0 + h) * D + geo.vofs;
#pragma unroll
            for (int d = 0; d < C::VD; ++d) ov[h][d] *= inv;
            store_out_vec<C::VD>(p.out, ob, ov[h], p.out_dtype);
          }
        }
        if (EXT && p.lse != nullptr && lane == 0) {
#pragma unroll
          for (int h = 0; h < GW; ++h) p.lse[out_row(p, sg.seq, kvh, v0 + h)] = st.m[h] + __log2f(lw[h]);
        }
      } else {
        // Record (max, sum, unnormalised output) for this warp's heads; the
        // last CTA of the unit to finish merges all of them.
        const int64_t rec = c * 2 + (gb == lo ? 0 : 1);
        const int hr = kh * GH + hw * GW;  // first head of this warp within the record
        if (geo.vg == 0) {
#pragma unroll
          for (int h = 0; h < GW; ++h) {
            float* ro = p.rec_o + (rec * HS + hr + h) * D + geo.vofs;
#pragma unroll
            for (int d = 0; d < C::VD; d += 2) *reinterpret_cast<float2*>(ro + d) = make_float2(ov[h][d], ov[h][d + 1]);
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < GW; ++h) {
            p.rec_ml[(rec * HS + hr + h) * 2] = st.m[h];
            p.rec_ml[(rec * HS + hr + h) * 2 + 1] = lw[h];
          }
        }
        // Count the record (one counter per unit and warp slot): the warp
        // barrier orders the lanes' record writes before lane 0's release.
        // The first segment is counted now and its result only read at the
        // end, so the add's round trip never stalls the stream.
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

  // The warp whose add completes a unit's count (one add per contributing
  // CTA) merges the records of its heads and resets the counter for the next
  // call. No warp waits for another warp or CTA.
  __syncthreads();
  const bool any_abort = s_misc[0] != 0;
  if (active && !any_abort && (pend0 || pend1)) {
    const BlockPos q0 = locate_block(lo, HN, s_scan, B, p.n_hsub);
    const BlockPos q1 = locate_block(hi - 1, HN, s_scan, B, p.n_hsub);
    const int64_t p0_u0 = lo - q0.j, p1_u0 = hi - 1 - q1.j;
    int last = 0;  // bit 0: the segment at lo, bit 1: the segment ending at hi
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
          set_flag(p.err, 0x10u);  // the workspace counters were not zero
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
    // Copies that may still be in flight must land before the CTA exits and
    // its shared memory is reused: wait (bounded) for the latest issued fill
    // of every stage.
    for (int x = 0; x < S; ++x) {
      const unsigned int n = s_iss[x];
      if (n > 0) (void)mbar_wait_bounded(fbar + x, (n - 1) & 1u);
    }
  }
}

}  // namespace kvc
