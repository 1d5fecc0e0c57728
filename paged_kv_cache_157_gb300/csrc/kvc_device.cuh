// Device-side helpers: element conversion, mbarrier and bulk-copy (TMA) PTX
// wrappers with bounded waits, warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace kvc {

// Bounds of an mbarrier wait: about one second of %globaltimer time (a copy
// normally lands within microseconds), with a poll cap as a second guard.
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ void set_flag(unsigned int* word, unsigned int bit) {
  if (word != nullptr) atomicOr(word, bit);
}

// ------------------------------------------------------------------ convert

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16-byte chunk
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static float to_float(float x) { return x; }
  // Elements 2c and 2c+1 of a 16-byte chunk as an fp32 pair.
  __device__ __forceinline__ static float2 pair(const uint4& u, int c) {
    return c == 0 ? make_float2(__uint_as_float(u.x), __uint_as_float(u.y))
                  : make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
  }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static void unpack2(uint32_t w, float* f) {
    // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits.
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xffff0000u);
  }
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    unpack2(u.x, f + 0);
    unpack2(u.y, f + 2);
    unpack2(u.z, f + 4);
    unpack2(u.w, f + 6);
  }
  __device__ __forceinline__ static float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
  // Element `hi` (0: low half, 1: high half) of a 32-bit word of two bf16.
  __device__ __forceinline__ static float half_to_float(uint32_t w, int hi) {
    return hi ? __uint_as_float(w & 0xffff0000u) : __uint_as_float(w << 16);
  }
  __device__ __forceinline__ static float2 pair(const uint4& u, int c) {
    const uint32_t w = c == 0 ? u.x : (c == 1 ? u.y : (c == 2 ? u.z : u.w));
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
};
template <> struct Elem<__half> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static void unpack2(uint32_t w, float* f) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    float2 t = __half22float2(h);
    f[0] = t.x;
    f[1] = t.y;
  }
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    unpack2(u.x, f + 0);
    unpack2(u.y, f + 2);
    unpack2(u.z, f + 4);
    unpack2(u.w, f + 6);
  }
  __device__ __forceinline__ static float to_float(__half x) { return __half2float(x); }
  __device__ __forceinline__ static float half_to_float(uint32_t w, int hi) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(hi ? (w >> 16) : (w & 0xffffu))));
  }
  __device__ __forceinline__ static float2 pair(const uint4& u, int c) {
    uint32_t w = c == 0 ? u.x : (c == 1 ? u.y : (c == 2 ? u.z : u.w));
    return __half22float2(*reinterpret_cast<__half2*>(&w));
  }
};

// FP8 e4m3 cache element (1 byte; no infinities, largest finite 448).
struct fp8e4m3 {
  unsigned char bits;
};

// Two e4m3 values (low byte first) as an fp32 pair, through the hardware
// e4m3x2 -> f16x2 conversion (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ float2 fp8x2_to_float2(uint32_t two) {
  uint32_t h2;
  const unsigned short in = static_cast<unsigned short>(two & 0xffffu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// Rounds two fp32 values to e4m3 (nearest, ties to even, saturating at +-448;
// NaN stays NaN); returns them packed, a in the low byte.
__device__ __forceinline__ unsigned short float2_to_fp8x2(float a, float b) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// INT8 cache element (symmetric codes in [-127, 127]).
struct s8q {
  signed char bits;
};

// int8 codes to fp32 without the integer-to-float unit (a quarter-rate
// pipe). Flipping the sign bits (s8_flip) turns code c into the byte c + 128;
// placed in the low mantissa byte of the float 2^23 (s8_biased) that byte
// gives 2^23 + c + 128, and one packed subtraction of 2^23 + 128 leaves c
// exactly (s8_unbias).
__device__ __forceinline__ uint32_t s8_flip(uint32_t w) { return w ^ 0x80808080u; }

// Byte `b` (0..3) of a flipped word as the float 2^23 + c + 128.
__device__ __forceinline__ float s8_biased(uint32_t flipped, int b) {
  return __uint_as_float(__byte_perm(flipped, 0x4B000000u, 0x7440u | static_cast<unsigned>(b)));
}

__device__ __forceinline__ float2 s8_unbias(float2 x) {
  union {
    float2 f;
    unsigned long long u;
  } a, c, r;
  a.f = x;
  c.f = make_float2(-8388736.0f, -8388736.0f);
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.u) : "l"(a.u), "l"(c.u));
  return r.f;
}

// Two int8 codes (low byte first) as an fp32 pair (exact).
__device__ __forceinline__ float2 s8x2_to_float2(uint32_t two) {
  const uint32_t u = s8_flip(two);
  return s8_unbias(make_float2(s8_biased(u, 0), s8_biased(u, 1)));
}

// Rounds an fp32 value to an int8 code: nearest, ties to even, saturating at
// +-127 (-128 is never produced).
__device__ __forceinline__ int float_to_s8(float x) {
  const int r = __float2int_rn(x);
  return r < -127 ? -127 : (r > 127 ? 127 : r);
}

template <> struct Elem<s8q> {
  static constexpr int kVec = 16;
  __device__ __forceinline__ static float2 pair(const uint4& u, int c) {
    const int wi = c >> 1;
    const uint32_t w = s8_flip(wi == 0 ? u.x : (wi == 1 ? u.y : (wi == 2 ? u.z : u.w)));
    const int b = 2 * (c & 1);  // bytes b and b + 1 of the word
    return s8_unbias(make_float2(s8_biased(w, b), s8_biased(w, b + 1)));
  }
};

template <> struct Elem<fp8e4m3> {
  static constexpr int kVec = 16;
  // Elements 2c and 2c+1 of a 16-byte chunk (c in [0, 8)) as an fp32 pair.
  __device__ __forceinline__ static float2 pair(const uint4& u, int c) {
    const int wi = c >> 1;
    const uint32_t w = wi == 0 ? u.x : (wi == 1 ? u.y : (wi == 2 ? u.z : u.w));
    return fp8x2_to_float2((c & 1) ? (w >> 16) : w);
  }
};

// Stores one fp32 value as the output dtype (0 f32, 1 f16, 2 bf16).
__device__ __forceinline__ void store_out(void* out, int64_t idx, float v, int out_dtype) {
  if (out_dtype == 0) {
    static_cast<float*>(out)[idx] = v;
  } else if (out_dtype == 1) {
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  } else {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  }
}

// Stores N consecutive fp32 values as the output dtype, with one vector
// store when the destination is aligned for it.
template <int N>
__device__ __forceinline__ void store_out_vec(void* out, int64_t idx, const float* v, int out_dtype) {
  if (out_dtype == 0) {
    float* dst = static_cast<float*>(out) + idx;
    if constexpr (N % 4 == 0) {
      if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        return;
      }
    } else if constexpr (N % 2 == 0) {
      if ((reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 2) *reinterpret_cast<float2*>(dst + i) = make_float2(v[i], v[i + 1]);
        return;
      }
    }
#pragma unroll
    for (int i = 0; i < N; ++i) dst[i] = v[i];
    return;
  }
  uint32_t w[(N + 1) / 2];
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float b = (i + 1 < N) ? v[i + 1] : 0.f;
    if (out_dtype == 1) {
      __half2 h = __floats2half2_rn(v[i], b);
      w[i / 2] = *reinterpret_cast<uint32_t*>(&h);
    } else {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[i], b);
      w[i / 2] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  unsigned short* dst = static_cast<unsigned short*>(out) + idx;
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
  if constexpr (N == 8) {
    if ((a & 15u) == 0) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      return;
    }
  } else if constexpr (N == 4) {
    if ((a & 7u) == 0) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      return;
    }
  } else if constexpr (N == 2) {
    if ((a & 3u) == 0) {
      *reinterpret_cast<uint32_t*>(dst) = w[0];
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i) dst[i] = static_cast<unsigned short>(i & 1 ? (w[i / 2] >> 16) : (w[i / 2] & 0xffffu));
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar` to complete; returns false when the wait
// bounds run out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && globaltimer_ns() - t0 > kWaitNs) return false;
  }
  return false;
}

// Non-blocking probe of a phase (test_wait never suspends the thread, where
// try_wait may wait a while inside the instruction).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same wait for data a copy brings, with an optional poll limit: polls
// == 0 keeps the bound above; polls > 0 gives up after that many
// non-blocking probes (a test hook that makes a kernel take its abort path on
// a healthy GPU).
__device__ __forceinline__ bool mbar_wait_data(uint64_t* bar, uint32_t parity, uint32_t polls) {
  if (polls == 0) return mbar_wait_bounded(bar, parity);
  for (uint32_t i = 0; i < polls; ++i)
    if (mbar_test_wait(bar, parity)) return true;
  return false;
}

// --------------------------------------------------------------- bulk copy

// 1-D bulk copy global -> shared through the TMA unit; completion is
// signalled on `bar` as transaction bytes. Both addresses 16-byte aligned,
// `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// ------------------------------------------------------------ reductions

// Atomic add with acquire-release semantics at GPU scope: it publishes the
// writes that precede it in this thread (or that a warp barrier ordered
// before it) and makes the writes published by earlier such adds on the same
// word visible to this thread's later reads.
__device__ __forceinline__ unsigned int atomic_add_acq_rel_gpu(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Packed fp32x2 arithmetic of sm_100+: one instruction, two independent
// IEEE fp32 operations (round to nearest even).
union F2U64 {
  float2 f;
  unsigned long long u;
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  F2U64 A, Bv, Cv, R;
  A.f = a;
  Bv.f = b;
  Cv.f = c;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(R.u) : "l"(A.u), "l"(Bv.u), "l"(Cv.u));
  return R.f;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  F2U64 A, Bv, R;
  A.f = a;
  Bv.f = b;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(R.u) : "l"(A.u), "l"(Bv.u));
  return R.f;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace kvc
