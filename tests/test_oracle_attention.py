"""Pins for the attention oracle: worked example, closed forms, invariants, brute force."""

import json
import math
import os

import numpy as np
import pytest

from oracle import attention as A
from oracle import paged as P


def test_worked_example_keep_and_drop_history(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_attention.json")))
    q = np.array(g["query"])
    k_hist = np.array([[0.7]])  # any key: q = 0 makes every score 0
    out, w, keys, values = A.cached_attention(q, k_hist, np.array(g["past_values"]), np.array([-1.3]),
                                              np.array(g["new_value"]))
    assert np.array_equal(out, np.array(g["with_history_output"]))
    assert np.array_equal(w, np.array(g["with_history_weights"]))
    assert keys.shape == (2, 1) and values.shape == (2, 1)
    out2, w2, _, _ = A.cached_attention(q, np.zeros((0, 1)), np.zeros((0, 1)), np.array([-1.3]),
                                        np.array(g["new_value"]))
    assert np.array_equal(out2, np.array(g["without_history_output"]))
    assert np.array_equal(w2, np.array([1.0]))


def test_swap_pairs_invariant_swap_keys_only_changes():
    # Same page, same paragraph: swapping whole K/V pairs leaves the result unchanged,
    # swapping only the keys changes it (needs a non-zero query to show).
    rng = np.random.default_rng(0)
    q = rng.normal(size=4)
    K = rng.normal(size=(5, 4))
    V = rng.normal(size=(5, 3))
    base, _ = A.attend_rows(q, K, V, 0.5)
    perm = np.array([3, 0, 4, 1, 2])
    pairs, _ = A.attend_rows(q, K[perm], V[perm], 0.5)
    keys_only, _ = A.attend_rows(q, K[perm], V, 0.5)
    assert np.allclose(base, pairs, rtol=0, atol=1e-14)
    assert np.max(np.abs(base - keys_only)) > 1e-3


def test_default_scale_is_inverse_sqrt_d():
    # d = 4, default scale 1/2; z1 - z0 = (1/2)(2 ln 3) = ln 3 -> weights 1/4, 3/4 -> output 3.
    q = np.array([1.0, 0.0, 0.0, 0.0])
    out, w, _, _ = A.cached_attention(q, np.zeros((1, 4)), np.array([[0.0]]),
                                      np.array([2.0 * math.log(3.0), 0.0, 0.0, 0.0]), np.array([4.0]))
    assert np.allclose(w, [0.25, 0.75], rtol=0, atol=1e-15)
    assert abs(out[0] - 3.0) < 1e-14


def test_causal_mask_is_lower_triangular_and_decode_row_sees_all():
    # "单请求 KV Cache" change 3: prefill rows see 0..i; a decode row with past_len = 4 sees 0..4.
    V = np.eye(4)
    out = A.causal_attention_full(np.zeros((4, 3)), np.zeros((4, 3)), V, 1.0, past_len=0)
    for i in range(4):
        expect = np.array([1.0 / (i + 1) if j <= i else 0.0 for j in range(4)])
        assert np.allclose(out[i], expect, rtol=0, atol=1e-15)
    V5 = np.eye(5)
    row = A.causal_attention_full(np.zeros((1, 3)), np.zeros((5, 3)), V5, 1.0, past_len=4)
    assert np.allclose(row[0], np.full(5, 0.2), rtol=0, atol=1e-15)
    # two new tokens on top of three cached ones: row 0 sees 0..3, row 1 sees 0..4
    two = A.causal_attention_full(np.zeros((2, 3)), np.zeros((5, 3)), V5, 1.0, past_len=3)
    assert np.allclose(two[0], [0.25, 0.25, 0.25, 0.25, 0.0], atol=1e-15)
    assert np.allclose(two[1], np.full(5, 0.2), atol=1e-15)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_special_cases(seed):
    rng = np.random.default_rng(seed)
    D = 8
    V = rng.normal(size=(11, D))
    K = rng.normal(size=(11, D))
    # n = 1: output is that value row exactly
    out, _ = A.attend_rows(rng.normal(size=D), K[:1], V[:1], 0.3)
    assert np.array_equal(out, V[0])
    # q = 0: mean of V
    out, lse = A.attend_rows(np.zeros(D), K, V, 0.3)
    assert np.allclose(out, V.mean(axis=0), rtol=0, atol=1e-14)
    assert abs(lse - math.log(11)) < 1e-14
    # identical keys: mean of V
    out, _ = A.attend_rows(rng.normal(size=D), np.repeat(K[:1], 11, axis=0), V, 0.3)
    assert np.allclose(out, V.mean(axis=0), rtol=0, atol=1e-14)
    # one dominant key (score gap > 100): its value
    Kd = np.zeros((11, D))
    Kd[6, 0] = 1000.0
    q = np.zeros(D)
    q[0] = 1.0
    out, _ = A.attend_rows(q, Kd, V, 1.0)
    assert np.allclose(out, V[6], rtol=0, atol=1e-14)
    # weights sum to one
    _, w, _, _ = A.cached_attention(rng.normal(size=D), K[:-1], V[:-1], K[-1], V[-1])
    assert abs(w.sum() - 1.0) < 1e-14 and np.all(w > 0)


@pytest.mark.parametrize("n,d,dv", [(1, 1, 1), (2, 3, 2), (7, 5, 4), (40, 8, 8), (17, 8, 3)])
def test_numpy_forms_match_python_loops(n, d, dv):
    rng = np.random.default_rng(n * 100 + d)
    q = rng.normal(size=d)
    K = rng.normal(size=(n, d)) * 2.0
    V = rng.normal(size=(n, dv))
    scale = 1.0 / math.sqrt(d)
    ref = np.array(A.attention_loops(q, K, V, scale))
    a, _ = A.attend_rows(q, K, V, scale)
    out_a, _, _, _ = A.cached_attention(q, K[:-1], V[:-1], K[-1], V[-1], scale)
    Q = rng.normal(size=(n, d))
    Q[-1] = q
    out_b = A.decode_by_recompute(Q, K, V, scale)
    for x in (a, out_a, out_b):
        assert np.max(np.abs(x - ref)) < 1e-13


def test_cached_equals_recompute_every_step_tiny_model():
    # "KV-Cache——为什么AI回复越来越快" section 05: cached generation equals recomputation
    # (printed max difference 1.39e-16 in float64). 1 sequence, 4 heads, d 32, 69 tokens.
    rng = np.random.default_rng(42)
    T, H, D = 69, 4, 32
    Q = rng.normal(size=(T, H, D))
    K = rng.normal(size=(T, H, D))
    V = rng.normal(size=(T, H, D))
    scale = 1.0 / math.sqrt(D)
    worst = 0.0
    for t in range(T):
        for h in range(H):
            a, _, _, _ = A.cached_attention(Q[t, h], K[:t, h], V[:t, h], K[t, h], V[t, h], scale)
            b = A.decode_by_recompute(Q[: t + 1, h], K[: t + 1, h], V[: t + 1, h], scale)
            worst = max(worst, float(np.max(np.abs(a - b))))
    assert worst < 1e-12


def test_input_validation_matches_page_rules():
    with pytest.raises(ValueError):
        A.cached_attention([], np.zeros((0, 0)), np.zeros((0, 1)), [], [1.0])
    with pytest.raises(ValueError):
        A.cached_attention([1.0, 2.0], np.zeros((1, 2)), np.zeros((2, 1)), [1.0, 0.0], [1.0])
    with pytest.raises(ValueError):
        A.cached_attention([1.0], np.zeros((0, 1)), np.zeros((0, 1)), [np.inf], [1.0])
    with pytest.raises(ValueError):
        A.attend_rows(np.zeros(2), np.zeros((0, 2)), np.zeros((0, 2)), 1.0)
