"""FP8 (e4m3) and INT8 KV-cache quantisation (oracle; test infrastructure only).

"KV-Cache——为什么AI回复越来越快" section 08 (KV-Cache quantisation): the FP16
K and V matrices are stored as FP8 (1 byte), halving the cache; V is
quantised per token (each token's K/V scaled on its own, suited to V whose
distribution varies), K per channel (each head dimension scaled on its own,
suited to K whose distribution is stable).

Readings where the page fixes nothing:

* FP8 format: e4m3 without infinities (1 sign bit, 4 exponent bits with bias
  7, 3 mantissa bits; exponent 15 with mantissa 7 is NaN; largest finite
  value 448; subnormals are m * 2^-9);
* rounding: to the nearest representable value, ties to the even code
  (mantissa bit 0 clear), values beyond 448 saturate to +-448;
* K: code = e4m3(k / k_scale[h, d]) with k_scale [n_kv_heads, head_dim]
  given by the caller (a calibration constant); the division is in float32;
* V: one scale per (token, kv head), s = max_d |v[d]| / 448 in float32 (1.0
  when the row is all zero), code = e4m3(v / s) in float32; the scales live
  in a pool [num_blocks, n_kv_heads, block_size] paged like the values;
* decode attends over k = e4m3value(code) * k_scale and
  v = e4m3value(code) * s, exactly as the full-precision decode does.
"""

from __future__ import annotations

import numpy as np

MAX_E4M3 = 448.0


def e4m3_value(code: int) -> float:
    """Value of one e4m3 code (float('nan') for the two NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
# non-negative finite codes 0x00..0x7E in increasing value order
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = _TABLE[:0x7F]


def decode_e4m3(codes) -> np.ndarray:
    return _TABLE[np.asarray(codes, dtype=np.int64) & 0xFF]


def encode_e4m3(x) -> np.ndarray:
    """Round float32 values to e4m3 codes: nearest, ties to even, saturate at +-448; NaN stays NaN."""
    x = np.asarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    for i, v in enumerate(flat):
        v = float(v)
        if v != v:
            out[i] = 0x7F
            continue
        neg = v < 0 or (v == 0 and np.signbit(v))
        a = min(abs(v), MAX_E4M3)
        j = int(np.searchsorted(_POS_VALUES, a))  # first value >= a
        if j < len(_POS_VALUES) and _POS_VALUES[j] == a:
            c = j
        else:
            lo, hi = j - 1, j
            dlo, dhi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
            if dlo < dhi:
                c = lo
            elif dhi < dlo:
                c = hi
            else:
                c = lo if (lo & 1) == 0 else hi  # tie: the even code
        out[i] = (0x80 if neg else 0) | int(_POS_CODES[c])
    return out.reshape(x.shape)


def quantize_k(k, k_scale) -> np.ndarray:
    """k [T, Hkv, D] (float32-representable), k_scale [Hkv, D] -> codes [T, Hkv, D]."""
    q = np.asarray(k, dtype=np.float32) / np.asarray(k_scale, dtype=np.float32)[None]
    return encode_e4m3(q.astype(np.float32))


def v_token_scale(v) -> np.ndarray:
    """v [T, Hkv, D] -> per (token, kv head) scale [T, Hkv] = max |v| / 448 (float32; 1 for zero rows)."""
    m = np.max(np.abs(np.asarray(v, dtype=np.float32)), axis=-1)
    s = (m / np.float32(MAX_E4M3)).astype(np.float32)
    return np.where(m > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_v(v, s) -> np.ndarray:
    q = np.asarray(v, dtype=np.float32) / np.asarray(s, dtype=np.float32)[..., None]
    return encode_e4m3(q.astype(np.float32))


def append_fp8(k, v, slot_mapping, k_cache, v_cache, v_scale_pool, k_scale):
    """Quantise and write token t's K/V at slot_mapping[t] (negative: skip).

    k_cache, v_cache: uint8 [num_blocks, Hkv, bs, D]; v_scale_pool: float32
    [num_blocks, Hkv, bs]. Returns new arrays.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    vs = np.array(v_scale_pool, copy=True)
    bs = kc.shape[2]
    kq = quantize_k(k, k_scale)
    s = v_token_scale(v)
    vq = quantize_v(v, s)
    for t, slot in enumerate(np.asarray(slot_mapping).reshape(-1)):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // bs, slot % bs
        kc[blk, :, off, :] = kq[t]
        vc[blk, :, off, :] = vq[t]
        vs[blk, :, off] = s[t]
    return kc, vc, vs


def dequantized_pools(k_cache, v_cache, v_scale_pool, k_scale):
    """float64 K and V pools the quantised cache stands for."""
    K = decode_e4m3(k_cache) * np.asarray(k_scale, dtype=np.float64)[None, :, None, :]
    V = decode_e4m3(v_cache) * np.asarray(v_scale_pool, dtype=np.float64)[..., None]
    return K, V


# ---------------------------------------------------------------- INT8
#
# The same section names INT8 next to FP8 (one byte per element, V scaled per
# token, K per channel). Readings where the page fixes nothing:
#
# * symmetric codes in [-127, 127] (-128 is never produced, so the range is
#   symmetric like the scales), code = round(x) with ties to even, values
#   beyond +-127 saturate;
# * K: code = int8(k / k_scale[h, d]) with caller-given per-channel scales;
#   V: s = max_d |v[d]| / 127 per (token, kv head) (1.0 for an all-zero row),
#   code = int8(v / s); divisions in float32;
# * decode attends over k = code * k_scale and v = code * s.

MAX_INT8 = 127.0


def encode_int8(x) -> np.ndarray:
    """Round float32 values to int8 codes: nearest, ties to even, saturating at +-127."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    return np.clip(np.rint(x), -MAX_INT8, MAX_INT8).astype(np.int8)


def quantize_k_int8(k, k_scale) -> np.ndarray:
    """k [T, Hkv, D], k_scale [Hkv, D] -> int8 codes [T, Hkv, D]."""
    q = np.asarray(k, dtype=np.float32) / np.asarray(k_scale, dtype=np.float32)[None]
    return encode_int8(q.astype(np.float32))


def v_token_scale_int8(v) -> np.ndarray:
    """v [T, Hkv, D] -> per (token, kv head) scale [T, Hkv] = max |v| / 127 (float32; 1 for zero rows)."""
    m = np.max(np.abs(np.asarray(v, dtype=np.float32)), axis=-1)
    s = (m / np.float32(MAX_INT8)).astype(np.float32)
    return np.where(m > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_v_int8(v, s) -> np.ndarray:
    q = np.asarray(v, dtype=np.float32) / np.asarray(s, dtype=np.float32)[..., None]
    return encode_int8(q.astype(np.float32))


def append_int8(k, v, slot_mapping, k_cache, v_cache, v_scale_pool, k_scale):
    """Quantise and write token t's K/V at slot_mapping[t] (negative: skip); int8 pools, float32 V scales."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    vs = np.array(v_scale_pool, copy=True)
    bs = kc.shape[2]
    kq = quantize_k_int8(k, k_scale)
    s = v_token_scale_int8(v)
    vq = quantize_v_int8(v, s)
    for t, slot in enumerate(np.asarray(slot_mapping).reshape(-1)):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // bs, slot % bs
        kc[blk, :, off, :] = kq[t]
        vc[blk, :, off, :] = vq[t]
        vs[blk, :, off] = s[t]
    return kc, vc, vs


def dequantized_pools_int8(k_cache, v_cache, v_scale_pool, k_scale):
    """float64 K and V pools the int8 cache stands for."""
    K = np.asarray(k_cache, dtype=np.int8).astype(np.float64) * np.asarray(k_scale, dtype=np.float64)[None, :, None, :]
    V = np.asarray(v_cache, dtype=np.int8).astype(np.float64) * np.asarray(v_scale_pool, dtype=np.float64)[..., None]
    return K, V
