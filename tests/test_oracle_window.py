"""Pins of the sliding-window decode oracle (CPU only).

The window keeps the newest W rows ("KV-Cache——为什么AI回复越来越快" section 08,
Window Attention / Sliding Window); the reading is that row n - 1 is the
current token, so rows [max(0, n - W), n) are visible. Each pin fixes the
visible range independently of the oracle's own slicing.
"""

import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import paged as P


def _pool(n, D, bs, rng, hkv=1, values=None):
    nb = -(-n // bs)
    perm = rng.permutation(nb + 3)[:nb]
    table = np.zeros((1, nb), dtype=np.int64)
    table[0, :] = perm
    kc = rng.standard_normal((nb + 3, hkv, bs, D))
    vc = rng.standard_normal((nb + 3, hkv, bs, D))
    if values is not None:
        for pos in range(n):
            vc[perm[pos // bs], :, pos % bs, :] = values[pos]
    return kc, vc, table


@pytest.mark.parametrize("n,W", [(1, 1), (5, 1), (40, 1), (40, 17), (40, 39), (40, 40), (40, 100), (33, 16)])
def test_zero_query_gives_exact_mean_of_the_last_w_rows(n, W):
    # q = 0 makes every visible weight equal, so the output is the mean of exactly the
    # visible value rows; one row more or less changes it (row values are distinct integers)
    rng = np.random.default_rng(1)
    D, bs = 4, 16
    vals = np.arange(n, dtype=np.float64)[:, None] * np.ones((1, D)) * 3.0
    kc, vc, table = _pool(n, D, bs, rng, values=vals)
    out = P.paged_decode_window(np.zeros((1, 1, D)), kc, vc, table, np.array([n]), 0.5, W)
    lo = max(0, n - W)
    expect = np.mean(vals[lo:n], axis=0)
    assert np.array_equal(out[0, 0], expect) or np.max(np.abs(out[0, 0] - expect)) < 1e-12


def test_window_one_returns_the_newest_value_exactly():
    rng = np.random.default_rng(2)
    kc, vc, table = _pool(37, 8, 16, rng)
    q = rng.standard_normal((1, 1, 8))
    out = P.paged_decode_window(q, kc, vc, table, np.array([37]), 0.35, 1)
    newest = vc[table[0, 36 // 16], 0, 36 % 16, :]
    assert np.array_equal(out[0, 0], newest)


def test_rows_outside_the_window_never_reach_the_output():
    rng = np.random.default_rng(3)
    n, W, bs, D = 50, 20, 16, 8
    kc, vc, table = _pool(n, D, bs, rng, hkv=2)
    q = rng.standard_normal((1, 4, D))
    ref = P.paged_decode_window(q, kc, vc, table, np.array([n]), 0.3, W)
    kc2, vc2 = kc.copy(), vc.copy()
    for pos in range(n - W):  # poison every dropped row
        kc2[table[0, pos // bs], :, pos % bs, :] = np.nan
        vc2[table[0, pos // bs], :, pos % bs, :] = np.nan
    got = P.paged_decode_window(q, kc2, vc2, table, np.array([n]), 0.3, W)
    assert np.array_equal(ref, got)


def test_large_window_is_full_attention():
    rng = np.random.default_rng(4)
    n, bs, D = 29, 16, 8
    kc, vc, table = _pool(n, D, bs, rng, hkv=2)
    q = rng.standard_normal((1, 4, D))
    full = P.paged_decode(q, kc, vc, table, np.array([n]), 0.3)
    for W in (n, n + 1, 10 * n):
        assert np.array_equal(P.paged_decode_window(q, kc, vc, table, np.array([n]), 0.3, W), full)


@pytest.mark.parametrize("n,W", [(9, 4), (12, 12), (7, 3)])
def test_matches_scalar_loops_on_the_last_w_rows(n, W):
    # brute force: gather rows by hand and run the scalar-loop form of attention
    rng = np.random.default_rng(5)
    bs, D = 4, 3
    kc, vc, table = _pool(n, D, bs, rng)
    q = rng.standard_normal(D)
    rows = range(n - W, n)
    K = [kc[table[0, r // bs], 0, r % bs, :] for r in rows]
    V = [vc[table[0, r // bs], 0, r % bs, :] for r in rows]
    loops = A.attention_loops(list(q), [list(k) for k in K], [list(v) for v in V], 0.7)
    got = P.paged_decode_window(q[None, None, :], kc, vc, table, np.array([n]), 0.7, W)[0, 0]
    assert np.max(np.abs(np.asarray(loops) - got)) < 1e-13


def test_window_must_be_positive():
    with pytest.raises(ValueError):
        P.window_start(10, 0)
