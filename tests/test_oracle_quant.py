"""Pins of the e4m3 codec and the FP8 KV quantisation oracle (CPU only)."""

import numpy as np
import pytest

from oracle import paged as P
from oracle import quant as Q


def test_known_codes():
    # values fixed by the e4m3 format (bias 7, 3 mantissa bits, no infinities)
    assert Q.e4m3_value(0x38) == 1.0
    assert Q.e4m3_value(0x7E) == 448.0
    assert Q.e4m3_value(0x01) == 2.0 ** -9
    assert Q.e4m3_value(0x08) == 2.0 ** -6
    assert Q.e4m3_value(0x07) == 7 * 2.0 ** -9
    assert Q.e4m3_value(0xC0) == -2.0
    assert np.isnan(Q.e4m3_value(0x7F)) and np.isnan(Q.e4m3_value(0xFF))
    assert Q.e4m3_value(0x80) == 0.0


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], dtype=np.uint8)
    vals = Q.decode_e4m3(codes).astype(np.float32)
    assert np.array_equal(Q.encode_e4m3(vals), codes)


def test_rounding_nearest_ties_even_and_saturation():
    # 1.0625 lies halfway between 1.0 (0x38, even) and 1.125 (0x39): the even code wins
    assert Q.encode_e4m3(np.float32(1.0625)) == 0x38
    # 1.1875 halfway between 1.125 (0x39) and 1.25 (0x3A, even)
    assert Q.encode_e4m3(np.float32(1.1875)) == 0x3A
    assert Q.encode_e4m3(np.float32(1.05)) == 0x38 and Q.encode_e4m3(np.float32(1.07)) == 0x39
    assert Q.encode_e4m3(np.float32(1e6)) == 0x7E and Q.encode_e4m3(np.float32(-1e6)) == 0xFE
    assert Q.encode_e4m3(np.float32(2.0 ** -11)) == 0x00  # below half the smallest subnormal
    assert Q.encode_e4m3(np.float32(3 * 2.0 ** -11)) == 0x01


def test_encode_is_nearest_by_brute_force():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(2000) * 30).astype(np.float32)
    codes = Q.encode_e4m3(x)
    table = np.array([Q.e4m3_value(c) for c in range(0x7F)])
    for v, c in zip(x, codes):
        a = min(abs(float(v)), 448.0)
        best = np.min(np.abs(table - a))
        assert abs(abs(Q.e4m3_value(c)) - a) == best


def test_v_scale_maps_the_row_maximum_to_448():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((5, 2, 16)).astype(np.float32)
    s = Q.v_token_scale(v)
    codes = Q.quantize_v(v, s)
    deq = Q.decode_e4m3(codes)
    assert np.all(np.max(np.abs(deq), axis=-1) == 448.0)
    assert np.all(Q.v_token_scale(np.zeros((1, 1, 4), np.float32)) == 1.0)


def test_quantisation_error_within_half_an_e4m3_step():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((40, 2, 32)).astype(np.float32)
    s = Q.v_token_scale(v)
    deq = Q.decode_e4m3(Q.quantize_v(v, s)) * s[..., None]
    # 3 mantissa bits: relative error <= 2^-4 for normal values, absolute <= 2^-10 * s near zero
    err = np.abs(deq - v)
    assert np.all(err <= np.maximum(np.abs(v) * 2.0 ** -4, s[..., None] * 2.0 ** -10) * (1 + 1e-6))


def test_append_fp8_and_dequantised_decode():
    rng = np.random.default_rng(3)
    nb, hkv, bs, D = 4, 2, 16, 8
    kc = np.zeros((nb, hkv, bs, D), np.uint8)
    vc = np.zeros((nb, hkv, bs, D), np.uint8)
    vs = np.ones((nb, hkv, bs), np.float32)
    ks = (0.5 + rng.random((hkv, D))).astype(np.float32)
    k = rng.standard_normal((3, hkv, D)).astype(np.float32)
    v = rng.standard_normal((3, hkv, D)).astype(np.float32)
    kc2, vc2, vs2 = Q.append_fp8(k, v, np.array([5, -1, 33]), kc, vc, vs, ks)
    assert np.array_equal(kc2[0, :, 5], Q.quantize_k(k[:1], ks)[0]) and np.all(kc2[0, :, 6] == 0)
    assert np.array_equal(vs2[2, :, 1], Q.v_token_scale(v[2:3])[0])
    K, V = Q.dequantized_pools(kc2, vc2, vs2, ks)
    assert np.allclose(K[2, :, 1], Q.decode_e4m3(Q.quantize_k(k[2:3], ks))[0] * ks)
    # a decode over the dequantised pools is the ordinary paged decode of those values
    out = P.paged_decode(rng.standard_normal((1, 4, D)), K, V, np.array([[0, 1, 2]]), np.array([34]), 0.3)
    assert np.all(np.isfinite(out))


# ------------------------------------------------------------------ INT8


def test_int8_rounds_to_nearest_with_ties_to_even():
    x = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 2.49, 2.51, 0.0, -0.0], np.float32)
    assert Q.encode_int8(x).tolist() == [0, 2, 2, 4, 0, -2, -2, 2, 3, 0, 0]


def test_int8_saturates_symmetrically():
    x = np.array([126.4, 126.5, 127.0, 127.6, 200.0, -127.4, -127.6, -300.0, 1e30, -1e30], np.float32)
    assert Q.encode_int8(x).tolist() == [126, 126, 127, 127, 127, -127, -127, -127, 127, -127]
    assert Q.encode_int8(np.float32(-128.0)).item() == -127  # -128 is never produced


def test_int8_nearest_by_brute_force():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(3000) * 60).astype(np.float32)
    codes = Q.encode_int8(x).astype(np.int64)
    grid = np.arange(-127, 128)
    for xi, c in zip(x.tolist(), codes.tolist()):
        d = np.abs(grid - min(max(xi, -127.0), 127.0))
        best = grid[d == d.min()]
        assert c in best.tolist()
        if len(best) == 2:
            assert c % 2 == 0  # a tie goes to the even code


def test_int8_v_rows_map_their_maximum_to_127():
    rng = np.random.default_rng(12)
    v = rng.standard_normal((50, 2, 64)).astype(np.float32)
    s = Q.v_token_scale_int8(v)
    codes = Q.quantize_v_int8(v, s).astype(np.int64)
    assert np.all(np.max(np.abs(codes), axis=-1) == 127)
    assert np.all(Q.v_token_scale_int8(np.zeros((1, 1, 4), np.float32)) == 1.0)
    assert np.all(Q.quantize_v_int8(np.zeros((1, 1, 4), np.float32), np.ones((1, 1), np.float32)) == 0)


def test_int8_error_within_half_a_step():
    rng = np.random.default_rng(13)
    v = rng.standard_normal((40, 2, 32)).astype(np.float32)
    s = Q.v_token_scale_int8(v)
    deq = Q.quantize_v_int8(v, s).astype(np.float64) * s[..., None]
    assert np.all(np.abs(deq - v) <= s[..., None] * (0.5 + 1e-6))
    ks = (0.01 + rng.random((2, 32))).astype(np.float32)
    k = (rng.standard_normal((40, 2, 32)) * 0.5).astype(np.float32)
    inside = np.abs(k / ks[None]) <= 127
    kdeq = Q.quantize_k_int8(k, ks).astype(np.float64) * ks[None]
    assert np.all(np.abs(kdeq - k)[inside] <= (ks[None] * (0.5 + 1e-6)).repeat(40, 0)[inside])


def test_append_int8_and_dequantised_pools():
    rng = np.random.default_rng(14)
    nb, hkv, bs, D = 4, 2, 16, 8
    kc = np.zeros((nb, hkv, bs, D), np.int8)
    vc = np.zeros((nb, hkv, bs, D), np.int8)
    vs = np.ones((nb, hkv, bs), np.float32)
    ks = (0.01 + rng.random((hkv, D))).astype(np.float32)
    k = rng.standard_normal((3, hkv, D)).astype(np.float32)
    v = rng.standard_normal((3, hkv, D)).astype(np.float32)
    kc2, vc2, vs2 = Q.append_int8(k, v, np.array([5, -1, 33]), kc, vc, vs, ks)
    assert np.array_equal(kc2[0, :, 5], Q.quantize_k_int8(k[:1], ks)[0]) and np.all(kc2[0, :, 6] == 0)
    assert np.array_equal(vs2[2, :, 1], Q.v_token_scale_int8(v[2:3])[0])
    K, V = Q.dequantized_pools_int8(kc2, vc2, vs2, ks)
    assert np.array_equal(V[2, :, 1], Q.quantize_v_int8(v[2:3], Q.v_token_scale_int8(v[2:3]))[0] *
                          Q.v_token_scale_int8(v[2:3])[0][:, None].astype(np.float64))
    assert np.allclose(K[0, :, 5], k[0], atol=float(ks.max()) * 0.5 + 1e-6)
