// Paged decode attention for MHA / GQA / MQA on CUDA cores.
//
// What is computed (knowledge point 2 of "KV缓存原理与显存估算"): for each
// sequence i and query head h, with kv head h / g,
//     z_t = scale * q . k_t,   a = softmax(z) (max subtracted),   o = sum_t a_t v_t
// over the context_lens[i] rows gathered in logical order through the block
// table (PagedAttention, "KV Cache（键值缓存）" section 2.3).
//
// How (sm_103a):
// * Work unit = (kv head, sequence, head subgroup of GH <= 4 query heads).
//   All GH query heads of a unit share every K/V page that is loaded. A
//   stream of pages is consumed by one warp (or, as a build option, by a warp
//   pair that splits the heads).
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

// Merges the records that CTAs c0..c1 left for one unit (blocks starting at
// global index u0) and writes the normalised output. Record ids are staged in
// s_rec in chunks of `cap` CTAs; pass 0 finds the maxima, pass 1 sums.
template <int GH>
__device__ void merge_records(const GqaParams& p, int D, int64_t u0, int64_t c0, int64_t c1, int64_t G, int64_t N,
                              int seq, int h0, int* s_rec, int cap) {
  constexpr int kMaxOwned = 8;  // GH * D <= 8 * blockDim for GH <= 4, D <= 256, 128 threads
  const int tid = threadIdx.x, nt = blockDim.x;
  const int span = static_cast<int>(c1 - c0 + 1);
  float M[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) M[h] = kNegInf;
  float O[kMaxOwned], Ls[kMaxOwned];
#pragma unroll
  for (int k = 0; k < kMaxOwned; ++k) O[k] = Ls[k] = 0.f;
  for (int pass = 0; pass < 2; ++pass) {
    for (int base = 0; base < span; base += cap) {
      const int n = min(cap, span - base);
      __syncthreads();
      for (int t = tid; t < n; t += nt) {
        const int64_t c = c0 + base + t;
        const int64_t f0 = cta_range_start(c, G, N);
        const int64_t f1 = cta_range_start(c + 1, G, N);
        s_rec[t] = (f0 == f1) ? -1 : static_cast<int>(c * 2 + ((u0 > f0) ? 1 : 0));
      }
      __syncthreads();
      for (int t = 0; t < n; ++t) {
        const int64_t rec = s_rec[t];
        if (rec < 0) continue;
        if (pass == 0) {
#pragma unroll
          for (int h = 0; h < GH; ++h) M[h] = fmaxf(M[h], __ldcg(p.rec_ml + (rec * GH + h) * 2));
        } else {
#pragma unroll
          for (int k = 0; k < kMaxOwned; ++k) {
            const int idx = tid + k * nt;
            if (idx >= GH * D) break;
            const int h = idx / D, d = idx - (idx / D) * D;
            const float mc = __ldcg(p.rec_ml + (rec * GH + h) * 2);
            if (mc == kNegInf) continue;
            const float f = fast_exp2(mc - select_head<GH>(M, h));
            Ls[k] += f * __ldcg(p.rec_ml + (rec * GH + h) * 2 + 1);
            O[k] += f * __ldcg(p.rec_o + (rec * GH + h) * D + d);
          }
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxOwned; ++k) {
    const int idx = tid + k * nt;
    if (idx >= GH * D) break;
    const int h = idx / D, d = idx - (idx / D) * D;
    store_out(p.out, (static_cast<int64_t>(seq) * p.n_q_heads + h0 + h) * D + d, O[k] / Ls[k], p.out_dtype);
  }
}

template <typename T, int D, int GH>
__global__ void __launch_bounds__(kGqaWarps * 32, 2) gqa_decode_kernel(const GqaParams p) {
  constexpr int HW = gqa_warps_per_stream(GH);  // warps sharing one page stream
  constexpr int GW = GH / HW;                    // query heads per warp
  constexpr int NP = kGqaWarps / HW;             // page streams per CTA
  using C = GqaCfg<T, D, GW>;
  extern __shared__ __align__(128) unsigned char smem[];
  const GqaSmem L = gqa_smem_layout(sizeof(T), D, GH, p.block_size, p.stages, p.batch);
  T* s_stage = reinterpret_cast<T*>(smem + L.stage_off);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + L.bar_off);  // [NP * S] full, then [NP * S] empty
  float* s_o = reinterpret_cast<float*>(smem + L.o_off);              // [kGqaWarps][GW][D]
  float* s_ml = reinterpret_cast<float*>(smem + L.ml_off);            // [kGqaWarps][GW][2]
  int* s_scan = reinterpret_cast<int*>(smem + L.scan_off);
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int sp = w / HW, hw = w % HW;  // page stream of this warp, and its half of the heads
  const bool issuer = (hw == 0);       // lane 0 of the stream's first warp issues the copies
  const int tq = lane / C::DL, dq = lane % C::DL;
  const int base_i = C::NV >= C::DL ? C::NVF * dq : dq / C::DUP;
  const int h_lane = base_i / C::RT;
  const int bs = p.block_size, S = p.stages;
  const int B = p.batch;
  const int tiles_per_page = bs / 16;
  const size_t page_elems = static_cast<size_t>(bs) * D;
  const uint32_t page_bytes = static_cast<uint32_t>(page_elems * sizeof(T));
  const T* kc = static_cast<const T*>(p.k_cache);
  const T* vc = static_cast<const T*>(p.v_cache);

  if (tid < NP * S) {
    mbar_init(s_bar + tid, 1);               // full: one arrive (with the copy bytes)
    mbar_init(s_bar + NP * S + tid, HW);     // empty: every warp of the stream releases
  }
  fence_barrier_init();

  // Block range of this CTA.
  int64_t lo, hi, slab = 0, N = 0;
  const int64_t G = gridDim.x;
  if (p.unit_mode) {
    lo = 0;
    hi = 1;
    __syncthreads();
  } else {
    scan_blocks(p.context_lens, B, bs, p.max_blocks, s_scan);
    slab = static_cast<int64_t>(p.n_hsub) * s_scan[B];
    N = slab * p.n_kv_heads;
    lo = cta_range_start(blockIdx.x, G, N);
    hi = cta_range_start(blockIdx.x + 1, G, N);
  }
  if (blockIdx.x == 0) {
    // Validate every length once; in the split mode CTA 0 also writes the
    // zero outputs of sequences whose length is invalid (no CTA visits them).
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

  const uint64_t pol = policy_evict_first();
  uint32_t ticket = 0;  // tiles of this stream consumed so far (stage/parity bookkeeping)
  bool aborted = false;

  for (int64_t gb = lo; gb < hi;) {
    // ---- locate the unit containing global block gb
    int kvh, seq, hsub, j0, nb, seg_len;
    if (p.unit_mode) {
      const int u = blockIdx.x;
      hsub = u % p.n_hsub;
      seq = (u / p.n_hsub) % B;
      kvh = u / (p.n_hsub * B);
      nb = seq_blocks(p.context_lens, seq, bs, p.max_blocks);
      j0 = 0;
      seg_len = nb;
    } else {
      kvh = static_cast<int>(gb / slab);
      const int64_t r = gb - kvh * slab;
      int a = 0, b = B - 1;  // largest seq with n_hsub*S[seq] <= r
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (static_cast<int64_t>(p.n_hsub) * s_scan[mid] <= r) a = mid; else b = mid - 1;
      }
      seq = a;
      nb = s_scan[seq + 1] - s_scan[seq];
      const int64_t r2 = r - static_cast<int64_t>(p.n_hsub) * s_scan[seq];
      hsub = static_cast<int>(r2 / nb);
      j0 = static_cast<int>(r2 - static_cast<int64_t>(hsub) * nb);
      const int64_t left = nb - j0;
      seg_len = static_cast<int>((hi - gb) < left ? (hi - gb) : left);
    }
    const bool whole = (j0 == 0 && seg_len == nb);
    const int which = (gb == lo) ? 0 : 1;
    const int64_t u0 = gb - j0;  // global index of the unit's first block (split mode)
    gb = p.unit_mode ? hi : gb + seg_len;
    const int h0 = kvh * p.group + hsub * GH;  // first query head of the unit
    const int hq0 = h0 + hw * GW;              // first query head of this warp
    const int n_rows = seq_rows(p.context_lens, seq, bs, p.max_blocks);

    if (nb == 0) {
      // invalid length: zero output (only reachable in unit mode)
      for (int idx = tid; idx < GH * D; idx += blockDim.x)
        store_out(p.out, (static_cast<int64_t>(seq) * p.n_q_heads + h0 + idx / D) * D + idx % D, 0.f,
                  p.out_dtype);
      continue;
    }

    // ---- per-warp state
    WarpState<T, D, GW> st;
    {
      const T* qp = static_cast<const T*>(p.q) + (static_cast<int64_t>(seq) * p.n_q_heads + hq0) * D;
#pragma unroll
      for (int h = 0; h < GW; ++h) {
        float f[C::DPL];
#pragma unroll
        for (int j = 0; j < C::NCH; ++j)
          Elem<T>::unpack(__ldg(reinterpret_cast<const uint4*>(qp + h * D + (dq + C::DL * j) * C::VEC)),
                          f + j * C::VEC);
#pragma unroll
        for (int i = 0; i < C::DP2; ++i) {
          st.q[h][i] = make_float2(f[2 * i] * p.qscale, f[2 * i + 1] * p.qscale);
          st.o[h][i] = make_float2(0.f, 0.f);
        }
        st.m[h] = kNegInf;
      }
      st.l = 0.f;
    }

    const int nbw = seg_len > sp ? (seg_len - sp + NP - 1) / NP : 0;  // this stream's blocks
    const int32_t* bt = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks;
    T* wst = s_stage + static_cast<size_t>(sp) * S * 2 * page_elems;
    uint64_t* fbar = s_bar + sp * S;
    uint64_t* ebar = s_bar + NP * S + sp * S;

    // Block-table entries of this stream's tiles, 32 at a time: lane L holds
    // the entry of tile 32*window + L (one coalesced load per window, issued a
    // window ahead), handed to the issuing lane by shuffles.
    auto load_window = [&](int win) -> int {
      const int t = win * 32 + lane;
      return t < nbw ? __ldg(bt + j0 + sp + NP * t) : -1;
    };
    int bt_cur = load_window(0);
    int bt_nxt = nbw > 32 ? load_window(1) : -1;

    // Stage bookkeeping without divisions: tile t of this segment sits in
    // stage `slot`, whose barriers are in phase parity `par`; both advance by
    // one tile per iteration.
    const int stage_elems = 2 * bs * D;
    const int slot0 = static_cast<int>(ticket % static_cast<uint32_t>(S));
    const uint32_t par0 = (ticket / static_cast<uint32_t>(S)) & 1u;

    auto issue = [&](int slot, int phys) {
      if (phys < 0 || phys >= p.num_blocks) {
        set_flag(p.err, 0x1u);
        mbar_arrive(fbar + slot);
      } else {
        const size_t src = (static_cast<size_t>(phys) * p.n_kv_heads + kvh) * page_elems;
        T* dst = wst + slot * stage_elems;
        mbar_arrive_expect_tx(fbar + slot, 2 * page_bytes);
        bulk_g2s(dst, kc + src, page_bytes, fbar + slot, pol);
        bulk_g2s(dst + page_elems, vc + src, page_bytes, fbar + slot, pol);
      }
    };

    // All stages are free here: every warp finished the previous segment
    // before the CTA-wide barrier that ended it.
    if (!aborted && issuer) {
      int sl = slot0;
      for (int t = 0; t < S && t < nbw; ++t) {
        const int ph = __shfl_sync(0xffffffffu, bt_cur, t);
        if (lane == 0) issue(sl, ph);
        sl = (sl + 1 == S) ? 0 : sl + 1;
      }
    }
    __syncwarp();

    int drain_from = -1;  // first tile not consumed when a wait gave up
    int slot = slot0;
    uint32_t par = par0;
    for (int t = 0; t < nbw; ++t) {
      if (aborted) break;
      if (t > 0 && (t & 31) == 0) {
        bt_cur = bt_nxt;
        bt_nxt = (t + 32 < nbw) ? load_window((t >> 5) + 1) : -1;
      }
      const int phys = __shfl_sync(0xffffffffu, bt_cur, t & 31);
      const int tn = t + S;
      const int phys_next = __shfl_sync(0xffffffffu, (tn >> 5) == (t >> 5) ? bt_cur : bt_nxt, tn & 31);
      const bool ok = mbar_wait_bounded(fbar + slot, par);
      if (__any_sync(0xffffffffu, !ok)) {
        aborted = true;
        drain_from = t;
        if (lane == 0) set_flag(p.err, 0x8u);
        break;
      }
      const int j = j0 + sp + NP * t;
      if (phys >= 0 && phys < p.num_blocks) {
        const T* kp = wst + slot * stage_elems;
        const T* vp = kp + page_elems;
        const int vr = min(bs, n_rows - j * bs);
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
      // Every shared-memory read of this stage fed an FMA issued before this
      // point, so no read of it is outstanding once the warp releases it.
      __syncwarp();
      if (HW > 1 && lane == 0) mbar_arrive(ebar + slot);
      if (issuer && tn < nbw) {
        if (HW > 1) {
          // Refill once every warp of the stream has released the stage.
          bool ok2 = true;
          if (lane == 0) ok2 = mbar_wait_bounded(ebar + slot, par);
          if (!__shfl_sync(0xffffffffu, ok2 ? 1 : 0, 0)) {
            aborted = true;
            drain_from = t + 1;
            if (lane == 0) set_flag(p.err, 0x8u);
            break;
          }
        }
        if (lane == 0) issue(slot, phys_next);
      }
      __syncwarp();
      if (++slot == S) {
        slot = 0;
        par ^= 1u;
      }
    }
    if (drain_from >= 0 && issuer) {
      // Copies issued but not consumed (at most S) must land before this
      // shared memory is reused or the CTA exits.
      for (int t = drain_from; t < nbw && t < drain_from + S; ++t)
        (void)mbar_wait_bounded(fbar + (ticket + t) % S, ((ticket + t) / S) & 1u);
    }
    ticket += nbw;

    // ---- combine the warps of this CTA
#pragma unroll
    for (int msk = C::DL; msk < 32; msk <<= 1) {
#pragma unroll
      for (int h = 0; h < GW; ++h) {
#pragma unroll
        for (int i = 0; i < C::DP2; ++i) {
          st.o[h][i].x += __shfl_xor_sync(0xffffffffu, st.o[h][i].x, msk);
          st.o[h][i].y += __shfl_xor_sync(0xffffffffu, st.o[h][i].y, msk);
        }
      }
    }
    float lw[GW];
#pragma unroll
    for (int hh = 0; hh < GW; ++hh) lw[hh] = warp_sum(h_lane == hh ? st.l : 0.f) * (1.0f / C::DUP);
    if (tq == 0) {
#pragma unroll
      for (int h = 0; h < GW; ++h) {
#pragma unroll
        for (int j = 0; j < C::NCH; ++j) {
#pragma unroll
          for (int e = 0; e < C::VEC; e += 2) {
            const float2 v = st.o[h][(j * C::VEC + e) / 2];
            s_o[(w * GW + h) * D + (dq + C::DL * j) * C::VEC + e] = v.x;
            s_o[(w * GW + h) * D + (dq + C::DL * j) * C::VEC + e + 1] = v.y;
          }
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < GW; ++h) {
        s_ml[(w * GW + h) * 2] = st.m[h];
        s_ml[(w * GW + h) * 2 + 1] = lw[h];
      }
    }
    __syncthreads();
    const int64_t rec = static_cast<int64_t>(blockIdx.x) * 2 + which;
    for (int idx = tid; idx < GH * D; idx += blockDim.x) {
      const int h = idx / D, d = idx - (idx / D) * D;
      // head h of the unit lives in warp (stream, h / GW), slot h % GW
      const int hw_h = h / GW, jh = h - hw_h * GW;
      float M = kNegInf;
#pragma unroll
      for (int ss = 0; ss < NP; ++ss) M = fmaxf(M, s_ml[((ss * HW + hw_h) * GW + jh) * 2]);
      float Lsum = 0.f, O = 0.f;
#pragma unroll
      for (int ss = 0; ss < NP; ++ss) {
        const int r = (ss * HW + hw_h) * GW + jh;
        const float mw = s_ml[r * 2];
        if (mw == kNegInf) continue;
        const float f = fast_exp2(mw - M);
        Lsum += f * s_ml[r * 2 + 1];
        O += f * s_o[r * D + d];
      }
      if (whole) {
        store_out(p.out, (static_cast<int64_t>(seq) * p.n_q_heads + h0 + h) * D + d, O / Lsum, p.out_dtype);
      } else {
        p.rec_o[(rec * GH + h) * D + d] = O;
        if (d == 0) {
          p.rec_ml[(rec * GH + h) * 2] = M;
          p.rec_ml[(rec * GH + h) * 2 + 1] = Lsum;
        }
      }
    }
    if (!whole) {
      // Publish this record, count it, and let the last contributor merge.
      __threadfence();
      __syncthreads();
      const int64_t c0 = cta_of_block(u0, G, N), c1 = cta_of_block(u0 + nb - 1, G, N);
      const int64_t unit = (static_cast<int64_t>(kvh) * B + seq) * p.n_hsub + hsub;
      if (tid == 0) {
        int contributors = 0;
        for (int64_t c = c0; c <= c1; ++c)
          contributors += (cta_range_start(c, G, N) != cta_range_start(c + 1, G, N)) ? 1 : 0;
        const unsigned int old = atomicAdd(p.counters + unit, 1u);
        s_last = 0;
        if (old + 1 == static_cast<unsigned int>(contributors)) {
          s_last = 1;
        } else if (old + 1 > static_cast<unsigned int>(contributors)) {
          set_flag(p.err, 0x10u);  // the workspace counters were not zero
          atomicExch(p.counters + unit, 0u);
        }
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        merge_records<GH>(p, D, u0, c0, c1, G, N, seq, h0, reinterpret_cast<int*>(s_o), NP * GH * D);
        if (tid == 0) p.counters[unit] = 0u;
      }
    }
    __syncthreads();
  }
}

}  // namespace kvc
