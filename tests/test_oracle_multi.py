"""Pins of the multi-token (chunked prefill / speculative) paged decode oracle (CPU only).

The T new query tokens of a sequence see the cache causally: token t sees rows
up to n - T + t, the mask rule of "单请求 KV Cache" (row i of a chunk sees
columns up to past_len + i). The pins compare with the full causal recompute
on contiguous K/V (a separate oracle form) and with single-token decode.
"""

import numpy as np
import pytest

from oracle import attention as A
from oracle import paged as P


def _paged(rng, n, hkv, D, bs):
    nb = -(-n // bs)
    perm = rng.permutation(nb + 2)[:nb]
    table = perm[None, :].astype(np.int64)
    K = rng.standard_normal((n, hkv, D))
    V = rng.standard_normal((n, hkv, D))
    kc = np.full((nb + 2, hkv, bs, D), np.nan)
    vc = np.full((nb + 2, hkv, bs, D), np.nan)
    for pos in range(n):
        kc[perm[pos // bs], :, pos % bs] = K[pos]
        vc[perm[pos // bs], :, pos % bs] = V[pos]
    return kc, vc, table, K, V


@pytest.mark.parametrize("n,T", [(1, 1), (5, 5), (20, 4), (33, 3), (40, 16)])
def test_multi_equals_the_last_rows_of_causal_recompute(n, T):
    rng = np.random.default_rng(n * 7 + T)
    hkv, g, D, bs = 2, 2, 8, 16
    kc, vc, table, K, V = _paged(rng, n, hkv, D, bs)
    q = rng.standard_normal((1, T, hkv * g, D))
    out = P.paged_decode_multi(q, kc, vc, table, np.array([n]), 0.4)
    for h in range(hkv * g):
        kvh = h // g
        ref = A.causal_attention_full(q[0, :, h], K[:, kvh], V[:, kvh], 0.4, past_len=n - T)
        assert np.max(np.abs(out[0, :, h] - ref)) < 1e-12


def test_single_token_is_ordinary_decode():
    rng = np.random.default_rng(9)
    kc, vc, table, _, _ = _paged(rng, 29, 2, 8, 16)
    q = rng.standard_normal((1, 1, 4, 8))
    assert np.array_equal(P.paged_decode_multi(q, kc, vc, table, np.array([29]), 0.3)[:, 0],
                          P.paged_decode(q[:, 0], kc, vc, table, np.array([29]), 0.3))


def test_earlier_tokens_never_see_later_rows():
    # poisoning the rows after token t's position must not change token t's output
    rng = np.random.default_rng(10)
    n, T, bs = 30, 5, 16
    kc, vc, table, _, _ = _paged(rng, n, 1, 8, bs)
    q = rng.standard_normal((1, T, 1, 8))
    ref = P.paged_decode_multi(q, kc, vc, table, np.array([n]), 0.3)
    kc2, vc2 = kc.copy(), vc.copy()
    for pos in range(n - T + 1, n):  # rows only tokens >= 1 may see
        kc2[table[0, pos // bs], :, pos % bs] = 1e6
        vc2[table[0, pos // bs], :, pos % bs] = 1e6
    got = P.paged_decode_multi(q, kc2, vc2, table, np.array([n]), 0.3)
    assert np.array_equal(got[:, 0], ref[:, 0])
    assert not np.allclose(got[:, 1], ref[:, 1])


def test_context_must_hold_the_new_rows():
    rng = np.random.default_rng(11)
    kc, vc, table, _, _ = _paged(rng, 3, 1, 4, 16)
    with pytest.raises(ValueError):
        P.paged_decode_multi(rng.standard_normal((1, 4, 1, 4)), kc, vc, table, np.array([3]), 0.3)
