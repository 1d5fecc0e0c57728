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
//   All GH query heads of a unit share every K/V page that is loaded.
// * Balanced split: the cache blocks of all units are laid end to end
//   (kv head major, then sequence, then subgroup, so units that read the
//   same pages sit next to each other) and CTA c takes blocks
//   [c*N/G, (c+1)*N/G). A CTA finishes whole units itself and leaves at most
//   two partial results (its first and last segment) as fp32 records; the
//   merge kernel combines records with the log-sum-exp rule.
// * Each warp streams its own pages: lane 0 issues 1-D bulk copies (TMA) of
//   the K page and V page of a block into a per-warp ring of shared-memory
//   stages, completion counted on an mbarrier; every wait is bounded.
// * Per 16-row tile a lane owns 16 (or 8) head dimensions of TL-strided rows.
//   Partial dot products are reduced across the lanes of a row with a
//   reduce-scatter (each lane ends holding whole scores of one head), softmax
//   runs online in the log2 domain with a lazy rescale (the reference maximum
//   moves only when a score exceeds it by more than 8, i.e. a factor 256), and
//   the weights are gathered back for the V accumulation in fp32.
#pragma once

#include "decode_gqa.h"
#include "kvc_device.cuh"

namespace kvc {

template <typename T, int D, int GH>
struct GqaCfg {
  static constexpr int NW = kGqaWarps;
  static constexpr int DPL = (D >= 64) ? 16 : 8;  // dims per lane
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
  // inclusive warp scan of per-thread sums
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
  float q[GH][C::DPL];
  float o[GH][C::DPL];
  float m[GH];
  float l;  // partial sum of this lane's weights (head h_lane)
};

template <typename T, int D, int GH>
__device__ __forceinline__ float select_head(const float (&v)[GH], int h) {
  float r = v[0];
#pragma unroll
  for (int i = 1; i < GH; ++i) r = (h == i) ? v[i] : r;
  return r;
}

// One 16-row tile of a page: scores, online softmax, V accumulation.
template <typename T, int D, int GH, bool PARTIAL>
__device__ __forceinline__ void gqa_tile(const T* __restrict__ kp, const T* __restrict__ vp, int valid,
                                         WarpState<T, D, GH>& st, int tq, int dq, int lane, int h_lane) {
  using C = GqaCfg<T, D, GH>;
  float s[C::NV];
#pragma unroll
  for (int r = 0; r < C::RT; ++r) {
    const T* rp = kp + (r * C::TL + tq) * D;
    float kf[C::DPL];
#pragma unroll
    for (int j = 0; j < C::NCH; ++j) Elem<T>::unpack(lds128(rp + (dq + C::DL * j) * C::VEC), kf + j * C::VEC);
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < C::DPL; ++e) acc = fmaf(st.q[h][e], kf[e], acc);
      s[h * C::RT + r] = acc;
    }
  }
  ReduceScatter<C::NV, C::DL / 2>::run(s, dq);

  // Score k of this lane has value index i = h*RT + r.
  const int base_i = C::NV >= C::DL ? C::NVF * dq : dq / C::DUP;
  float m_l = select_head<T, D, GH>(st.m, h_lane);
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
#pragma unroll
      for (int e = 0; e < C::DPL; ++e) st.o[hh][e] *= alpha;
      if (h_lane == hh) st.l *= alpha;
      st.m[hh] = mn;
    }
    m_l = select_head<T, D, GH>(st.m, h_lane);
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
    const T* rp = vp + (r * C::TL + tq) * D;
    float vf[C::DPL];
#pragma unroll
    for (int j = 0; j < C::NCH; ++j) Elem<T>::unpack(lds128(rp + (dq + C::DL * j) * C::VEC), vf + j * C::VEC);
    if (PARTIAL && r * C::TL + tq >= valid) {
#pragma unroll
      for (int e = 0; e < C::DPL; ++e) vf[e] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < GH; ++h) {
#pragma unroll
      for (int e = 0; e < C::DPL; ++e) st.o[h][e] = fmaf(pa[h * C::RT + r], vf[e], st.o[h][e]);
    }
  }
}

template <typename T, int D, int GH>
__global__ void __launch_bounds__(kGqaWarps * 32) gqa_decode_kernel(const GqaParams p) {
  using C = GqaCfg<T, D, GH>;
  extern __shared__ __align__(128) unsigned char smem[];
  const GqaSmem L = gqa_smem_layout(sizeof(T), D, GH, p.block_size, p.stages, p.batch);
  T* s_stage = reinterpret_cast<T*>(smem + L.stage_off);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  float* s_o = reinterpret_cast<float*>(smem + L.o_off);
  float* s_ml = reinterpret_cast<float*>(smem + L.ml_off);
  int* s_scan = reinterpret_cast<int*>(smem + L.scan_off);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
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

  if (tid < kGqaWarps * S) mbar_init(s_bar + tid, 1);
  fence_barrier_init();

  // Block range of this CTA.
  int64_t lo, hi, slab = 0, N = 0;
  if (p.unit_mode) {
    lo = 0;
    hi = 1;
    __syncthreads();
  } else {
    scan_blocks(p.context_lens, B, bs, p.max_blocks, s_scan);
    slab = static_cast<int64_t>(p.n_hsub) * s_scan[B];
    N = slab * p.n_kv_heads;
    lo = cta_range_start(blockIdx.x, gridDim.x, N);
    hi = cta_range_start(blockIdx.x + 1, gridDim.x, N);
  }
  if (blockIdx.x == 0 && tid < B) {
    const int n = __ldg(p.context_lens + tid);
    if (n < 1 || n > bs * p.max_blocks) set_flag(p.err, 0x2u);
  }
  if (blockIdx.x == 0 && tid == 0) {
    for (int b = kGqaWarps * 32; b < B; ++b) {
      const int n = __ldg(p.context_lens + b);
      if (n < 1 || n > bs * p.max_blocks) set_flag(p.err, 0x2u);
    }
  }

  const uint64_t pol = policy_evict_first();
  uint32_t ticket = 0;  // tiles consumed by this warp so far (stage/parity bookkeeping)
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
      gb = hi;
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
    if (!p.unit_mode) gb += seg_len;
    const int h0 = kvh * p.group + hsub * GH;
    const int n_rows = seq_rows(p.context_lens, seq, bs, p.max_blocks);

    if (nb == 0) {
      // invalid length: zero output (only reachable in unit mode)
      for (int idx = tid; idx < GH * D; idx += blockDim.x)
        store_out(p.out, (static_cast<int64_t>(seq) * p.n_q_heads + h0 + idx / D) * D + idx % D, 0.f,
                  p.out_dtype);
      continue;
    }

    // ---- per-warp state
    WarpState<T, D, GH> st;
    {
      const T* qp = static_cast<const T*>(p.q) + (static_cast<int64_t>(seq) * p.n_q_heads + h0) * D;
#pragma unroll
      for (int h = 0; h < GH; ++h) {
#pragma unroll
        for (int j = 0; j < C::NCH; ++j) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(qp + h * D + (dq + C::DL * j) * C::VEC));
          float f[C::VEC];
          Elem<T>::unpack(u, f);
#pragma unroll
          for (int e = 0; e < C::VEC; ++e) st.q[h][j * C::VEC + e] = f[e] * p.qscale;
        }
#pragma unroll
        for (int e = 0; e < C::DPL; ++e) st.o[h][e] = 0.f;
        st.m[h] = kNegInf;
      }
      st.l = 0.f;
    }

    const int nbw = seg_len > w ? (seg_len - w + kGqaWarps - 1) / kGqaWarps : 0;  // this warp's blocks
    const int32_t* bt = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks;
    T* wst = s_stage + static_cast<size_t>(w) * S * 2 * page_elems;
    uint64_t* wbar = s_bar + w * S;

    auto issue = [&](int t) {
      const int j = j0 + w + kGqaWarps * t;
      const int slot = (ticket + t) % S;
      const int phys = __ldg(bt + j);
      if (phys < 0 || phys >= p.num_blocks) {
        set_flag(p.err, 0x1u);
        mbar_arrive(wbar + slot);
      } else {
        const size_t src = (static_cast<size_t>(phys) * p.n_kv_heads + kvh) * page_elems;
        mbar_arrive_expect_tx(wbar + slot, 2 * page_bytes);
        bulk_g2s(wst + static_cast<size_t>(slot) * 2 * page_elems, kc + src, page_bytes, wbar + slot, pol);
        bulk_g2s(wst + static_cast<size_t>(slot) * 2 * page_elems + page_elems, vc + src, page_bytes, wbar + slot,
                 pol);
      }
    };

    if (lane == 0 && !aborted) {
      for (int t = 0; t < S && t < nbw; ++t) issue(t);
    }
    __syncwarp();

    int drain_from = -1;  // first tile not consumed when a wait gave up
    for (int t = 0; t < nbw; ++t) {
      const int slot = (ticket + t) % S;
      const uint32_t parity = ((ticket + t) / S) & 1u;
      if (aborted) break;
      const bool ok = mbar_wait_bounded(wbar + slot, parity);
      if (__any_sync(0xffffffffu, !ok)) {
        aborted = true;
        drain_from = t;
        if (lane == 0) set_flag(p.err, 0x8u);
        break;
      }
      const int j = j0 + w + kGqaWarps * t;
      const int phys = __ldg(bt + j);
      if (phys >= 0 && phys < p.num_blocks) {
        const T* kp = wst + static_cast<size_t>(slot) * 2 * page_elems;
        const T* vp = kp + page_elems;
        const int vr = min(bs, n_rows - j * bs);
        for (int tt = 0; tt < tiles_per_page; ++tt) {
          const int valid = vr - tt * 16;
          if (valid <= 0) break;
          if (valid >= 16)
            gqa_tile<T, D, GH, false>(kp + tt * 16 * D, vp + tt * 16 * D, 16, st, tq, dq, lane, h_lane);
          else
            gqa_tile<T, D, GH, true>(kp + tt * 16 * D, vp + tt * 16 * D, valid, st, tq, dq, lane, h_lane);
        }
      }
      __syncwarp();
      if (lane == 0 && t + S < nbw) {
        fence_proxy_async_smem();
        issue(t + S);
      }
      __syncwarp();
    }
    if (drain_from >= 0) {
      // Copies issued but not consumed (at most S) must land before this
      // shared memory is reused or the CTA exits.
      for (int t = drain_from; t < nbw && t < drain_from + S; ++t)
        (void)mbar_wait_bounded(wbar + (ticket + t) % S, ((ticket + t) / S) & 1u);
    }
    ticket += nbw;

    // ---- combine the warps of this CTA
#pragma unroll
    for (int msk = C::DL; msk < 32; msk <<= 1) {
#pragma unroll
      for (int h = 0; h < GH; ++h) {
#pragma unroll
        for (int e = 0; e < C::DPL; ++e) st.o[h][e] += __shfl_xor_sync(0xffffffffu, st.o[h][e], msk);
      }
    }
    float lw[GH];
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) lw[hh] = warp_sum(h_lane == hh ? st.l : 0.f) * (1.0f / C::DUP);
    if (tq == 0) {
#pragma unroll
      for (int h = 0; h < GH; ++h) {
#pragma unroll
        for (int j = 0; j < C::NCH; ++j) {
#pragma unroll
          for (int e = 0; e < C::VEC; ++e)
            s_o[(w * GH + h) * D + (dq + C::DL * j) * C::VEC + e] = st.o[h][j * C::VEC + e];
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        s_ml[(w * GH + h) * 2] = st.m[h];
        s_ml[(w * GH + h) * 2 + 1] = lw[h];
      }
    }
    __syncthreads();
    const int64_t rec = static_cast<int64_t>(blockIdx.x) * 2 + which;
    for (int idx = tid; idx < GH * D; idx += blockDim.x) {
      const int h = idx / D, d = idx - (idx / D) * D;
      float M = kNegInf;
#pragma unroll
      for (int ww = 0; ww < kGqaWarps; ++ww) M = fmaxf(M, s_ml[(ww * GH + h) * 2]);
      float Lsum = 0.f, O = 0.f;
#pragma unroll
      for (int ww = 0; ww < kGqaWarps; ++ww) {
        const float mw = s_ml[(ww * GH + h) * 2];
        if (mw == kNegInf) continue;
        const float f = fast_exp2(mw - M);
        Lsum += f * s_ml[(ww * GH + h) * 2 + 1];
        O += f * s_o[(ww * GH + h) * D + d];
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
    __syncthreads();
  }
}

// Combines the partial records of units split across CTAs; writes zeros for
// units whose length was invalid. One CTA per unit.
template <int GH>
__global__ void __launch_bounds__(128) gqa_merge_kernel(const GqaParams p, int D, int G) {
  extern __shared__ __align__(16) unsigned char smem[];
  int* s_scan = reinterpret_cast<int*>(smem);
  const int B = p.batch, bs = p.block_size;
  scan_blocks(p.context_lens, B, bs, p.max_blocks, s_scan);
  const int u = blockIdx.x;
  const int hsub = u % p.n_hsub;
  const int seq = (u / p.n_hsub) % B;
  const int kvh = u / (p.n_hsub * B);
  const int h0 = kvh * p.group + hsub * GH;
  const int nb = s_scan[seq + 1] - s_scan[seq];
  if (nb == 0) {
    for (int idx = threadIdx.x; idx < GH * D; idx += blockDim.x)
      store_out(p.out, (static_cast<int64_t>(seq) * p.n_q_heads + h0 + idx / D) * D + idx % D, 0.f, p.out_dtype);
    return;
  }
  const int64_t slab = static_cast<int64_t>(p.n_hsub) * s_scan[B];
  const int64_t N = slab * p.n_kv_heads;
  const int64_t u0 = kvh * slab + static_cast<int64_t>(p.n_hsub) * s_scan[seq] + static_cast<int64_t>(hsub) * nb;
  const int64_t u1 = u0 + nb;
  const int64_t c0 = cta_of_block(u0, G, N), c1 = cta_of_block(u1 - 1, G, N);
  if (c0 == c1) return;
  for (int idx = threadIdx.x; idx < GH * D; idx += blockDim.x) {
    const int h = idx / D, d = idx - (idx / D) * D;
    float M = kNegInf;
    for (int64_t c = c0; c <= c1; ++c) {
      const int64_t f0 = cta_range_start(c, G, N);
      if (f0 == cta_range_start(c + 1, G, N)) continue;
      const int64_t rec = c * 2 + ((u0 > f0) ? 1 : 0);
      M = fmaxf(M, p.rec_ml[(rec * GH + h) * 2]);
    }
    float Lsum = 0.f, O = 0.f;
    for (int64_t c = c0; c <= c1; ++c) {
      const int64_t f0 = cta_range_start(c, G, N);
      if (f0 == cta_range_start(c + 1, G, N)) continue;
      const int64_t rec = c * 2 + ((u0 > f0) ? 1 : 0);
      const float mc = p.rec_ml[(rec * GH + h) * 2];
      if (mc == kNegInf) continue;
      const float f = fast_exp2(mc - M);
      Lsum += f * p.rec_ml[(rec * GH + h) * 2 + 1];
      O += f * p.rec_o[(rec * GH + h) * D + d];
    }
    store_out(p.out, (static_cast<int64_t>(seq) * p.n_q_heads + h0 + h) * D + d, O / Lsum, p.out_dtype);
  }
}

}  // namespace kvc
