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

#include "decode_gqa.h"
#include "kvc_device.cuh"

namespace kvc {

template <typename T, int D, int GH>
struct GqaCfg {
  static constexpr int DPL = (D >= 64) ? 16 : 8;  // dims per lane
  static constexpr int DP2 = DPL / 2;               // fp32 pairs per lane
  static constexpr int DL = D / DPL;                // lanes per row
  static constexpr int TL = 32 / DL;                // row groups per warp
  static constexpr int RT = 16 / TL;                // rows per lane per 16-row tile
  static constexpr int VEC = Elem<T>::kVec;         // elements per 16-byte chunk
  static constexpr int NCH = DPL / VEC;             // chunks per lane per row
  static constexpr int NV = RT * GH;                // partial scores per lane per tile
  static constexpr int NVF = NV >= DL ? NV / DL : 1;  // whole scores per lane after reduce-scatter
  static constexpr int DUP = NV >= DL ? 1 : DL / NV;  // lanes holding the same score
  static_assert(DL * DPL == D && TL * DL == 32 && RT * TL == 16, "lane layout");
  static_assert(NCH * VEC == DPL, "chunking");
  static_assert(RT % NVF == 0, "a lane's scores must belong to one head");
};

// Number of cache blocks sequence b contributes (0 if its length is invalid).
__device__ __forceinline__ int seq_blocks(const int32_t* lens, int b, int bs, int max_blocks) {
  const int n = __ldg(lens + b);
  if (n < 1) return 0;
  const int nb = (n + bs - 1) / bs;
  return nb < max_blocks ? nb : max_blocks;
}

__device__ __forceinline__ int seq_rows(const int32_t* lens, int b, int bs, int max_blocks) {
  const int n = __ldg(lens + b);
  if (n < 1) return 0;
  const int cap = bs * max_blocks;
  return n < cap ? n : cap;
}

// Exclusive prefix sums of seq_blocks over the batch into s_scan[0..B];
// the whole CTA participates. s_scan needs B + 1 + 32 ints.
__device__ inline void scan_blocks(const int32_t* lens, int B, int bs, int max_blocks, int* s_scan) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (B + nt - 1) / nt;
  const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += seq_blocks(lens, b, bs, max_blocks);
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
    run += seq_blocks(lens, b, bs, max_blocks);
  }
  if (b1 == B && b0 < B) s_scan[B] = run;
  if (B == 0 && tid == 0) s_scan[0] = 0;
  __syncthreads();
}

// CTA whose block range [c*N/G, (c+1)*N/G) contains global block b.
__device__ __forceinline__ int64_t cta_of_block(int64_t b, int64_t G, int64_t N) { return ((b + 1) * G - 1) / N; }
__device__ __forceinline__ int64_t cta_range_start(int64_t c, int64_t G, int64_t N) { return c * N / G; }

// Reduce-scatter of CUR partial values across the lanes of a row group
// (xor masks B, B/2, ..., 1). Upper lanes keep the upper half at each step;
// once one value is left the remaining steps all-reduce it.
template <int CUR, int B>
struct ReduceScatter {
  __device__ __forceinline__ static void run(float* s, int dq) {
    if constexpr (B >= 1) {
      if constexpr (CUR > 1) {
        constexpr int H = CUR / 2;
        const bool up = (dq & B) != 0;
#pragma unroll
        for (int t = 0; t < H; ++t) {
          const float send = up ? s[t] : s[t + H];
          const float keep = up ? s[t + H] : s[t];
          s[t] = keep + __shfl_xor_sync(0xffffffffu, send, B);
        }
        ReduceScatter<H, B / 2>::run(s, dq);
      } else {
        s[0] += __shfl_xor_sync(0xffffffffu, s[0], B);
        ReduceScatter<1, B / 2>::run(s, dq);
      }
    }
  }
};

template <typename T, int D, int GH>
struct WarpState {
  using C = GqaCfg<T, D, GH>;
  float2 q[GH][C::DP2];  // query, pre-scaled by scale*log2(e)
  float2 o[GH][C::DP2];  // unnormalised output relative to m
  float m[GH];           // reference maximum (log2 units), warp-uniform
  float l;               // partial sum of this lane's weights (head h_lane)
};

template <int GH>
__device__ __forceinline__ float select_head(const float (&v)[GH], int h) {
  float r = v[0];
#pragma unroll
  for (int i = 1; i < GH; ++i) r = (h == i) ? v[i] : r;
  return r;
}

template <typename T, int NCH, int DL, int VEC>
__device__ __forceinline__ void load_pairs(const T* rp, int dq, float2* f) {
#pragma unroll
  for (int j = 0; j < NCH; ++j)
    Elem<T>::unpack(lds128(rp + (dq + DL * j) * VEC), reinterpret_cast<float*>(f) + j * VEC);
}

// One 16-row tile of a page: scores, online softmax, V accumulation.
template <typename T, int D, int GH, bool PARTIAL>
__device__ __forceinline__ void gqa_tile(const T* __restrict__ kp, const T* __restrict__ vp, int valid,
                                         WarpState<T, D, GH>& st, int tq, int dq, int lane, int h_lane) {
  using C = GqaCfg<T, D, GH>;
  float s[C::NV];
  {
    // All RT rows' raw K chunks first, then the RT*GH accumulators advance
    // together over the lane's dims (independent FMA chains, unpacked lazily).
    uint4 kr[C::RT][C::NCH];
#pragma unroll
    for (int r = 0; r < C::RT; ++r) {
#pragma unroll
      for (int j = 0; j < C::NCH; ++j) kr[r][j] = lds128(kp + (r * C::TL + tq) * D + (dq + C::DL * j) * C::VEC);
    }
    float2 acc[C::RT][GH];
#pragma unroll
    for (int j = 0; j < C::NCH; ++j) {
#pragma unroll
      for (int c = 0; c < C::VEC / 2; ++c) {
        const int i = j * (C::VEC / 2) + c;
#pragma unroll
        for (int r = 0; r < C::RT; ++r) {
          const float2 kf = Elem<T>::pair(kr[r][j], c);
#pragma unroll
          for (int h = 0; h < GH; ++h) acc[r][h] = (i == 0) ? fmul2(st.q[h][0], kf) : ffma2(st.q[h][i], kf, acc[r][h]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < C::RT; ++r) {
#pragma unroll
      for (int h = 0; h < GH; ++h) s[h * C::RT + r] = acc[r][h].x + acc[r][h].y;
    }
  }
  ReduceScatter<C::NV, C::DL / 2>::run(s, dq);

  // Score k of this lane has value index i = h*RT + r.
  const int base_i = C::NV >= C::DL ? C::NVF * dq : dq / C::DUP;
  float m_l = select_head<GH>(st.m, h_lane);
  bool need = false;
#pragma unroll
  for (int k = 0; k < C::NVF; ++k) {
    if (PARTIAL) {
      const int r = (base_i + k) % C::RT;
      if (r * C::TL + tq >= valid) s[k] = kNegInf;
    }
    need |= s[k] > m_l + 8.0f;
  }
  if (__any_sync(0xffffffffu, need)) {
    float loc = s[0];
#pragma unroll
    for (int k = 1; k < C::NVF; ++k) loc = fmaxf(loc, s[k]);
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
      const float tmax = warp_max(h_lane == hh ? loc : kNegInf);
      const float mn = fmaxf(st.m[hh], tmax);
      const float alpha = fast_exp2(st.m[hh] - mn);
      const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
      for (int i = 0; i < C::DP2; ++i) st.o[hh][i] = fmul2(st.o[hh][i], a2);
      if (h_lane == hh) st.l *= alpha;
      st.m[hh] = mn;
    }
    m_l = select_head<GH>(st.m, h_lane);
  }
  float p[C::NVF];
#pragma unroll
  for (int k = 0; k < C::NVF; ++k) {
    p[k] = fast_exp2(s[k] - m_l);
    st.l += p[k];
  }
  float pa[C::NV];
  const int grp = lane & ~(C::DL - 1);
#pragma unroll
  for (int i = 0; i < C::NV; ++i) {
    const int src = C::NV >= C::DL ? i / C::NVF : i * C::DUP;
    const int k = C::NV >= C::DL ? i % C::NVF : 0;
    pa[i] = __shfl_sync(0xffffffffu, p[k], grp | src);
  }
#pragma unroll
  for (int r = 0; r < C::RT; ++r) {
    float2 vf[C::DP2];
    load_pairs<T, C::NCH, C::DL, C::VEC>(vp + (r * C::TL + tq) * D, dq, vf);
    if (PARTIAL && r * C::TL + tq >= valid) {
#pragma unroll
      for (int i = 0; i < C::DP2; ++i) vf[i] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const float2 pp = make_float2(pa[h * C::RT + r], pa[h * C::RT + r]);
#pragma unroll
      for (int i = 0; i < C::DP2; ++i) st.o[h][i] = ffma2(pp, vf[i], st.o[h][i]);
    }
  }
}

// Worker whose block range [w*N/W, (w+1)*N/W) contains global block b, and
// the first block of worker w's range.
__device__ __forceinline__ int64_t worker_of_block(int64_t b, int64_t W, int64_t N) { return ((b + 1) * W - 1) / N; }
__device__ __forceinline__ int64_t worker_range_start(int64_t w, int64_t W, int64_t N) { return w * N / W; }

// Global block index -> (kv head, sequence, head subgroup, block of the
// sequence). Blocks are numbered kv head major, then sequence, then subgroup;
// s_scan holds the exclusive prefix sums of the per-sequence block counts.
struct BlockPos {
  int kvh, seq, hsub, j, nb;
};

__device__ __forceinline__ BlockPos locate_block(int64_t gb, int64_t slab, const int* s_scan, int B, int n_hsub) {
  BlockPos r;
  r.kvh = static_cast<int>(gb / slab);
  const int64_t rem = gb - r.kvh * slab;
  int a = 0, b = B - 1;  // largest sequence with n_hsub * S[seq] <= rem (skips empty ones)
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (static_cast<int64_t>(n_hsub) * s_scan[mid] <= rem) a = mid; else b = mid - 1;
  }
  r.seq = a;
  r.nb = s_scan[a + 1] - s_scan[a];
  const int r2 = static_cast<int>(rem - static_cast<int64_t>(n_hsub) * s_scan[a]);
  r.hsub = r2 / r.nb;
  r.j = r2 - r.hsub * r.nb;
  return r;
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
template <int D, int GH, int GW>
__device__ void merge_unit_warp(const GqaParams& p, int64_t u0, int nb, int64_t W, int64_t N, int seq, int hq0,
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
      const float* ml = p.rec_ml + (rec * GH + hoff + h) * 2;
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
        ov[i][k] = ok ? __ldcg(reinterpret_cast<const float4*>(rbase + rr * GH * D + 128 * k))
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
  for (int h = 0; h < GW; ++h) inv[h] = 1.0f / warp_sum(Lp[h]);
#pragma unroll
  for (int k = 0; k < NCK; ++k) {
    const int idx = lane + 32 * k;
    if (idx >= GW * CH) break;
    float iv = 0.f;
#pragma unroll
    for (int h = 0; h < GW; ++h) iv = (idx / CH == h) ? inv[h] : iv;
    const int64_t o = (static_cast<int64_t>(seq) * p.n_q_heads + hq0) * D + 4 * idx;
    store_out(p.out, o, O[k].x * iv, p.out_dtype);
    store_out(p.out, o + 1, O[k].y * iv, p.out_dtype);
    store_out(p.out, o + 2, O[k].z * iv, p.out_dtype);
    store_out(p.out, o + 3, O[k].w * iv, p.out_dtype);
  }
}

template <typename T, int D, int GH>
__global__ void __launch_bounds__(kGqaWarps * 32, 2) gqa_decode_kernel(const GqaParams p) {
  constexpr int HW = gqa_warps_per_stream(GH);  // warps sharing one page stream
  constexpr int GW = GH / HW;                    // query heads per warp
  constexpr int NP = kGqaWarps / HW;             // page streams (workers) per CTA
  using C = GqaCfg<T, D, GW>;
  static_assert(GW * HW == GH && kGqaWarps % HW == 0, "head split over the warps of a stream");
  static_assert(D % 32 == 0, "merge lanes own D / 32 dims");
  extern __shared__ __align__(128) unsigned char smem[];
  const GqaSmem L = gqa_smem_layout(sizeof(T), D, GH, p.block_size, p.stages, p.batch);
  T* s_stage = reinterpret_cast<T*>(smem + L.stage_off);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + L.bar_off);  // [NP * S] full, then [NP * S] empty
  int* s_scan = reinterpret_cast<int*>(smem + L.scan_off);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int sp = w / HW, hw = w % HW;  // stream (worker) of this warp, and its share of the heads
  const bool issuer = (hw == 0);       // lane 0 of the stream's first warp issues the copies
  const int tq = lane / C::DL, dq = lane % C::DL;
  const int base_i = C::NV >= C::DL ? C::NVF * dq : dq / C::DUP;
  const int h_lane = base_i / C::RT;
  const int bs = p.block_size, S = p.stages;
  const int B = p.batch;
  const int tiles_per_page = bs / 16;
  const int page_elems = bs * D;
  const int stage_elems = 2 * page_elems + GH * D;  // K page, V page, the unit's query rows
  const uint32_t page_bytes = static_cast<uint32_t>(page_elems * sizeof(T));
  const uint32_t q_bytes = static_cast<uint32_t>(GH * D * sizeof(T));
  const T* kc = static_cast<const T*>(p.k_cache);
  const T* vc = static_cast<const T*>(p.v_cache);
  const T* qg = static_cast<const T*>(p.q);
  const uint32_t full = 0xffffffffu;

  if (tid < NP * S) {
    mbar_init(s_bar + tid, 1);            // full: one arrive (with the copy bytes)
    mbar_init(s_bar + NP * S + tid, HW);  // empty: every warp of the stream releases
  }
  fence_barrier_init();
  scan_blocks(p.context_lens, B, bs, p.max_blocks, s_scan);  // ends with a CTA barrier
  const int64_t slab = static_cast<int64_t>(p.n_hsub) * s_scan[B];
  const int64_t N = slab * p.n_kv_heads;
  const int64_t W = static_cast<int64_t>(gridDim.x) * NP;
  const int64_t wk = static_cast<int64_t>(blockIdx.x) * NP + sp;

  if (blockIdx.x == 0) {
    // Validate every length once; in the split mode CTA 0 also writes the
    // zero outputs of sequences whose length is invalid (no worker visits them).
    for (int b = tid; b < B; b += blockDim.x) {
      const int n = __ldg(p.context_lens + b);
      if (n < 1 || n > bs * p.max_blocks) set_flag(p.err, 0x2u);
    }
    if (!p.unit_mode) {
      for (int b = 0; b < B; ++b) {
        if (__ldg(p.context_lens + b) >= 1) continue;
        for (int idx = tid; idx < p.n_q_heads * D; idx += blockDim.x)
          store_out(p.out, static_cast<int64_t>(b) * p.n_q_heads * D + idx, 0.f, p.out_dtype);
      }
    }
  }
  // No CTA-wide barrier below this point: every stream runs on its own.

  int64_t lo, hi;
  if (p.unit_mode) {
    // worker u takes unit u = (kv head, sequence, subgroup) whole
    const int64_t units = static_cast<int64_t>(p.n_kv_heads) * B * p.n_hsub;
    if (wk >= units) return;
    const int hsub = static_cast<int>(wk % p.n_hsub);
    const int seq = static_cast<int>((wk / p.n_hsub) % B);
    const int kvh = static_cast<int>(wk / (static_cast<int64_t>(p.n_hsub) * B));
    const int nb = s_scan[seq + 1] - s_scan[seq];
    if (nb == 0) {
      // invalid length: zero output for this warp's heads
      const int hq0 = kvh * p.group + hsub * GH + hw * GW;
      for (int idx = lane; idx < GW * D; idx += 32)
        store_out(p.out, (static_cast<int64_t>(seq) * p.n_q_heads + hq0) * D + idx, 0.f, p.out_dtype);
      return;
    }
    lo = kvh * slab + static_cast<int64_t>(p.n_hsub) * s_scan[seq] + static_cast<int64_t>(hsub) * nb;
    hi = lo + nb;
  } else {
    lo = worker_range_start(wk, W, N);
    hi = worker_range_start(wk + 1, W, N);
  }
  const int total = static_cast<int>(hi - lo);  // blocks (positions) of this worker
  if (total <= 0) return;

  T* wst = s_stage + static_cast<size_t>(sp) * S * stage_elems;
  uint64_t* fbar = s_bar + sp * S;
  uint64_t* ebar = s_bar + NP * S + sp * S;
  const uint64_t pol = policy_evict_first();

  // Positions lo + 32*win + lane, one per lane: the element offset of the
  // K/V page (-1 if the table entry is out of range) and, for the first
  // block of a segment, the element offset of the unit's query rows.
  auto window = [&](int win, int64_t& src, int& qoff) {
    const int64_t pos = lo + static_cast<int64_t>(win) * 32 + lane;
    src = -1;
    qoff = -1;
    if (pos < hi) {
      const BlockPos bp = locate_block(pos, slab, s_scan, B, p.n_hsub);
      const int phys = __ldg(p.block_tables + static_cast<int64_t>(bp.seq) * p.max_blocks + bp.j);
      if (phys >= 0 && phys < p.num_blocks)
        src = (static_cast<int64_t>(phys) * p.n_kv_heads + bp.kvh) * page_elems;
      if (pos == lo || bp.j == 0) qoff = (bp.seq * p.n_q_heads + bp.kvh * p.group + bp.hsub * GH) * D;
    }
  };
  // Copies of position x into stage `slot` (lane 0 only).
  auto issue = [&](int slot, int64_t src, int qoff) {
    const uint32_t bytes = (src >= 0 ? 2 * page_bytes : 0u) + (qoff >= 0 ? q_bytes : 0u);
    if (src < 0) set_flag(p.err, 0x1u);
    if (bytes == 0) {
      mbar_arrive(fbar + slot);
      return;
    }
    T* dst = wst + slot * stage_elems;
    mbar_arrive_expect_tx(fbar + slot, bytes);
    if (src >= 0) {
      bulk_g2s(dst, kc + src, page_bytes, fbar + slot, pol);
      bulk_g2s(dst + page_elems, vc + src, page_bytes, fbar + slot, pol);
    }
    if (qoff >= 0) bulk_g2s(dst + 2 * page_elems, qg + qoff, q_bytes, fbar + slot, pol);
  };

  int64_t w_src0, w_src1 = -1;
  int w_q0, w_q1 = -1;
  window(0, w_src0, w_q0);
  if (total > 32) window(1, w_src1, w_q1);

  // The ring runs ahead across segment boundaries: position x always sits in
  // stage x % S, and the copy of x + S is issued as soon as x is consumed.
  const int n_first = total < S ? total : S;
  if (issuer) {
    for (int i = 0; i < n_first; ++i) {
      const int64_t src = __shfl_sync(full, w_src0, i);
      const int qo = __shfl_sync(full, w_q0, i);
      if (lane == 0) issue(i, src, qo);
    }
  }
  int issued = n_first;
  __syncwarp();

  // Partial segments (at most two: the one starting at lo, the one ending
  // at hi) whose records wait to be counted.
  bool pend0 = false, pend1 = false;
  int64_t p0_u0 = 0, p1_u0 = 0, p0_unit = 0, p1_unit = 0;
  int p0_nb = 0, p1_nb = 0, p0_seq = 0, p1_seq = 0, p0_h0 = 0, p1_h0 = 0;

  int slot = 0;
  uint32_t par = 0;
  int c = 0;              // positions consumed
  int drain_from = -1;    // first position not consumed when a wait gave up
  int64_t gb = lo;
  while (gb < hi) {
    // ---- segment: the part of one unit inside [lo, hi)
    const BlockPos sg = locate_block(gb, slab, s_scan, B, p.n_hsub);
    const int seg_len = static_cast<int>(((sg.nb - sg.j) < (hi - gb)) ? (sg.nb - sg.j) : (hi - gb));
    const int n_rows = seq_rows(p.context_lens, sg.seq, bs, p.max_blocks);
    const int h0 = sg.kvh * p.group + sg.hsub * GH;  // first query head of the unit
    const int hq0 = h0 + hw * GW;                    // first query head of this warp

    WarpState<T, D, GW> st;
    for (int t = 0; t < seg_len; ++t, ++c) {
      if (c > 0 && (c & 31) == 0) {
        w_src0 = w_src1;
        w_q0 = w_q1;
        w_src1 = -1;
        w_q1 = -1;
        if (c + 32 < total) window((c >> 5) + 1, w_src1, w_q1);
      }
      const int64_t src = __shfl_sync(full, w_src0, c & 31);
      const int cn = c + S;
      const bool in_cur = (cn >> 5) == (c >> 5);
      const int64_t src_n = __shfl_sync(full, in_cur ? w_src0 : w_src1, cn & 31);
      const int q_n = __shfl_sync(full, in_cur ? w_q0 : w_q1, cn & 31);
      const bool ok = mbar_wait_bounded(fbar + slot, par);
      if (__any_sync(full, !ok)) {
        drain_from = c;
        if (lane == 0) set_flag(p.err, 0x8u);
        break;
      }
      const T* kp = wst + slot * stage_elems;
      if (t == 0) {
        // the unit's query rows came with its first page
        const T* qs = kp + 2 * page_elems + hw * GW * D;
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          float f[C::DPL];
#pragma unroll
          for (int j = 0; j < C::NCH; ++j)
            Elem<T>::unpack(lds128(qs + h * D + (dq + C::DL * j) * C::VEC), f + j * C::VEC);
#pragma unroll
          for (int i = 0; i < C::DP2; ++i) {
            st.q[h][i] = make_float2(f[2 * i] * p.qscale, f[2 * i + 1] * p.qscale);
            st.o[h][i] = make_float2(0.f, 0.f);
          }
          st.m[h] = kNegInf;
        }
        st.l = 0.f;
      }
      if (src >= 0) {
        const T* vp = kp + page_elems;
        const int vr = min(bs, n_rows - (sg.j + t) * bs);
        if (vr >= bs) {
          for (int tt = 0; tt < tiles_per_page; ++tt)
            gqa_tile<T, D, GW, false>(kp + tt * 16 * D, vp + tt * 16 * D, 16, st, tq, dq, lane, h_lane);
        } else {
          for (int tt = 0; tt < tiles_per_page; ++tt) {
            const int valid = vr - tt * 16;
            if (valid <= 0) break;
            if (valid >= 16)
              gqa_tile<T, D, GW, false>(kp + tt * 16 * D, vp + tt * 16 * D, 16, st, tq, dq, lane, h_lane);
            else
              gqa_tile<T, D, GW, true>(kp + tt * 16 * D, vp + tt * 16 * D, valid, st, tq, dq, lane, h_lane);
          }
        }
      }
      // Every shared-memory read of this stage fed an instruction issued
      // before this point, so no read of it is outstanding once released.
      __syncwarp();
      if (HW > 1 && lane == 0) mbar_arrive(ebar + slot);
      if (issuer && cn < total) {
        if (HW > 1) {
          // refill once every warp of the stream has released the stage
          bool ok2 = true;
          if (lane == 0) ok2 = mbar_wait_bounded(ebar + slot, par);
          if (!__shfl_sync(full, ok2 ? 1 : 0, 0)) {
            drain_from = c + 1;
            if (lane == 0) set_flag(p.err, 0x8u);
            break;
          }
        }
        if (lane == 0) issue(slot, src_n, q_n);
        ++issued;
      }
      __syncwarp();
      if (++slot == S) {
        slot = 0;
        par ^= 1u;
      }
    }
    if (drain_from >= 0) break;

    // ---- finish the segment: this warp holds every row of it for its heads
#pragma unroll
    for (int msk = C::DL; msk < 32; msk <<= 1) {
#pragma unroll
      for (int h = 0; h < GW; ++h) {
#pragma unroll
        for (int i = 0; i < C::DP2; ++i) {
          st.o[h][i].x += __shfl_xor_sync(full, st.o[h][i].x, msk);
          st.o[h][i].y += __shfl_xor_sync(full, st.o[h][i].y, msk);
        }
      }
    }
    float lw[GW];
#pragma unroll
    for (int hh = 0; hh < GW; ++hh) lw[hh] = warp_sum(h_lane == hh ? st.l : 0.f) * (1.0f / C::DUP);
    const bool whole = (sg.j == 0 && seg_len == sg.nb);
    if (whole) {
      if (tq == 0) {
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          const float inv = 1.0f / lw[h];
          const int64_t ob = (static_cast<int64_t>(sg.seq) * p.n_q_heads + hq0 + h) * D;
#pragma unroll
          for (int j = 0; j < C::NCH; ++j) {
#pragma unroll
            for (int e = 0; e < C::VEC; e += 2) {
              const float2 v = st.o[h][(j * C::VEC + e) / 2];
              const int d = (dq + C::DL * j) * C::VEC + e;
              store_out(p.out, ob + d, v.x * inv, p.out_dtype);
              store_out(p.out, ob + d + 1, v.y * inv, p.out_dtype);
            }
          }
        }
      }
    } else {
      // Record (max, sum, unnormalised output) for this warp's heads; the
      // last worker of the unit to finish merges all of them.
      const int64_t rec = wk * 2 + (gb == lo ? 0 : 1);
      if (tq == 0) {
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          float* ro = p.rec_o + (rec * GH + hw * GW + h) * D;
#pragma unroll
          for (int j = 0; j < C::NCH; ++j) {
#pragma unroll
            for (int e = 0; e < C::VEC; e += 4) {
              const float2 a = st.o[h][(j * C::VEC + e) / 2], b = st.o[h][(j * C::VEC + e) / 2 + 1];
              *reinterpret_cast<float4*>(ro + (dq + C::DL * j) * C::VEC + e) = make_float4(a.x, a.y, b.x, b.y);
            }
          }
        }
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          p.rec_ml[(rec * GH + hw * GW + h) * 2] = st.m[h];
          p.rec_ml[(rec * GH + hw * GW + h) * 2 + 1] = lw[h];
        }
      }
      // counted (and merged, if this worker is the unit's last) once the
      // whole range is done, so that no wait on the count stalls the stream
      if (gb == lo) {
        pend0 = true;
        p0_u0 = gb - sg.j;
        p0_nb = sg.nb;
        p0_seq = sg.seq;
        p0_h0 = h0;
        p0_unit = (static_cast<int64_t>(sg.kvh) * B + sg.seq) * p.n_hsub + sg.hsub;
      } else {
        pend1 = true;
        p1_u0 = gb - sg.j;
        p1_nb = sg.nb;
        p1_seq = sg.seq;
        p1_h0 = h0;
        p1_unit = (static_cast<int64_t>(sg.kvh) * B + sg.seq) * p.n_hsub + sg.hsub;
      }
    }
    gb += seg_len;
  }
  if (drain_from < 0 && (pend0 || pend1)) {
    // Count this worker's records (lane 0: the segment at lo, lane 1: the
    // one ending at hi); the add that completes a unit's count makes its
    // caller the unit's merger and resets the counter for the next call.
    __syncwarp();
    int last = 0;
    if (lane < 2 && (lane == 0 ? pend0 : pend1)) {
      const int64_t u0 = lane == 0 ? p0_u0 : p1_u0;
      const int nbu = lane == 0 ? p0_nb : p1_nb;
      const int64_t unit = lane == 0 ? p0_unit : p1_unit;
      const int64_t c0 = worker_of_block(u0, W, N), c1 = worker_of_block(u0 + nbu - 1, W, N);
      int64_t contributors = c1 - c0 + 1;
      if (N < W) {
        contributors = 0;
        for (int64_t x = c0; x <= c1; ++x)
          contributors += (worker_range_start(x, W, N) != worker_range_start(x + 1, W, N)) ? 1 : 0;
      }
      unsigned int* ctr = p.counters + unit * HW + hw;
      const unsigned int old = atomic_add_acq_rel_gpu(ctr, 1u);
      if (old + 1 == static_cast<unsigned int>(contributors)) {
        last = 1;
        *ctr = 0u;
      } else if (old + 1 > static_cast<unsigned int>(contributors)) {
        set_flag(p.err, 0x10u);  // the workspace counters were not zero
        atomicExch(ctr, 0u);
      }
    }
    // the warp barrier orders the other lanes' record reads after the acquire
    const int last0 = __shfl_sync(full, last, 0), last1 = __shfl_sync(full, last, 1);
    if (last0) merge_unit_warp<D, GH, GW>(p, p0_u0, p0_nb, W, N, p0_seq, p0_h0 + hw * GW, hw * GW, lane);
    if (last1) merge_unit_warp<D, GH, GW>(p, p1_u0, p1_nb, W, N, p1_seq, p1_h0 + hw * GW, hw * GW, lane);
  }
  if (drain_from >= 0 && issuer) {
    // Copies issued but not consumed (at most S) must land before the CTA
    // can exit and its shared memory be reused.
    for (int x = drain_from; x < issued; ++x) (void)mbar_wait_bounded(fbar + x % S, (x / S) & 1u);
  }
}

}  // namespace kvc
