"""Pins of the MLA oracle's read of the paged latent cache, by routes that do not use that read.

"KV Cache（键值缓存）" (llm-compass) section 2.2 caches one row per token: the
latent c_t (d_c wide) followed by the decoupled RoPE part (d_R wide); section
2.3 addresses a sequence's rows through its block table (logical block j of a
sequence lives in physical block table[j], row position % block_size). The
absorbed decode attends with the whole row as the key and its first d_c
elements as the value.

Each test below fixes the rows the oracle must read by something outside
``oracle/mla.py``: hand-placed integer rows whose mean is known in closed
form, a NaN in rows the table must never reach, the single-row case, and the
GQA oracle's own gather (``paged.gather_logical``, pinned separately) over the
latent pool viewed as a pool with one kv head.
"""

from __future__ import annotations

import math

import numpy as np

from oracle import mla as M
from oracle import paged as P
from oracle.attention import attend_rows

D_C, D_R = 12, 4
W = D_C + D_R


def _pool_with_marked_rows(n, bs, table, nblk, fill=1000.0):
    """Latent pool whose logical row p (read through `table`) holds p + 1 in every column.

    Every other row of the pool holds `fill`, so any row read from the wrong
    block or offset moves the mean."""
    pool = np.full((nblk, bs, W), fill, dtype=np.float64)
    for p in range(n):
        pool[table[p // bs], p % bs, :] = p + 1
    return pool


def test_zero_query_gives_exact_mean_of_logical_rows():
    # q = 0: every score is 0, so every weight is 1/n and the output is the
    # mean of the first d_c columns of the n logical rows: (n + 1) / 2 (up to
    # the rounding of the weights 1/n).
    bs, nblk = 4, 9
    table = np.array([7, 2, 5, 0, 8, 1])  # permuted: logical block j lives in block table[j]
    for n in (1, 3, 4, 5, 9, 13, 21, 24):
        pool = _pool_with_marked_rows(n, bs, table, nblk)
        out, _ = M.mla_absorbed_decode(np.zeros((1, 2, W)), pool, table[None, :], [n], 0.25, D_C)
        assert out.shape == (1, 2, D_C)
        assert np.max(np.abs(out - (n + 1) / 2.0)) < 1e-12, n


def test_gather_reads_each_block_through_its_own_table_entry():
    # Sequences of different lengths share a pool; each must see only its
    # own rows. Row values identify (sequence, position).
    bs, nblk = 4, 12
    tables = np.array([[3, 9, 0, 4], [11, 6, 2, 8]])
    lens = [14, 9]
    pool = np.full((nblk, bs, W), -50.0)
    for i, n in enumerate(lens):
        for p in range(n):
            pool[tables[i, p // bs], p % bs, :] = 100 * (i + 1) + p
    out, _ = M.mla_absorbed_decode(np.zeros((2, 1, W)), pool, tables, lens, 1.0, D_C)
    for i, n in enumerate(lens):
        expect = 100 * (i + 1) + (n - 1) / 2.0
        assert np.max(np.abs(out[i, 0] - expect)) < 1e-10


def test_nan_in_unused_tail_and_other_blocks_never_reaches_output():
    # Rows at or beyond n in the last block, and every block the table does
    # not name, hold NaN; a read of any of them would poison the output.
    rng = np.random.default_rng(5)
    bs, nblk, n = 8, 10, 19
    table = np.array([6, 1, 9])
    pool = np.full((nblk, bs, W), np.nan)
    rows = rng.normal(size=(n, W))
    for p in range(n):
        pool[table[p // bs], p % bs, :] = rows[p]
    q = rng.normal(size=(1, 3, W))
    out, lse = M.mla_absorbed_decode(q, pool, table[None, :], [n], 0.2, D_C)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    for h in range(3):
        ref, ref_lse = attend_rows(q[0, h], rows, rows[:, :D_C], 0.2)
        assert np.max(np.abs(out[0, h] - ref)) < 1e-13
        assert abs(lse[0, h] - ref_lse) < 1e-12


def test_single_row_returns_its_latent_part_exactly():
    # n = 1: the only weight is exactly 1, so the output is the first d_c
    # elements of the row in table[0], offset 0, bit for bit.
    rng = np.random.default_rng(6)
    bs, nblk = 4, 5
    pool = rng.normal(size=(nblk, bs, W))
    table = np.array([3, 0])
    q = rng.normal(size=(1, 4, W))
    out, _ = M.mla_absorbed_decode(q, pool, table[None, :], [1], 0.3, D_C)
    for h in range(4):
        assert np.array_equal(out[0, h], pool[3, 0, :D_C])


def test_equals_gqa_gather_over_latent_pool_as_one_kv_head():
    # The latent pool [blocks, bs, W] is a K pool [blocks, 1, bs, W] with one
    # kv head; its V pool is the first d_c columns. The GQA oracle's gather
    # (pinned by its own tests) must then give the same attention.
    rng = np.random.default_rng(7)
    bs, nblk = 4, 16
    lens = [1, 6, 13, 16]
    tables = np.stack([rng.permutation(nblk)[:4] for _ in lens])
    pool = rng.normal(size=(nblk, bs, W))
    q = rng.normal(size=(len(lens), 3, W))
    scale = 1.0 / math.sqrt(W)
    out, lse = M.mla_absorbed_decode(q, pool, tables, lens, scale, D_C)
    k_pool = pool[:, None, :, :]
    v_pool = pool[:, None, :, :D_C]
    ref, ref_lse = P.paged_decode_lse(q, k_pool, v_pool, tables, lens, scale)
    assert np.max(np.abs(out - ref)) < 1e-13
    assert np.max(np.abs(lse - ref_lse)) < 1e-12


def test_mla_one_matches_batch_form():
    rng = np.random.default_rng(8)
    bs, nblk = 4, 8
    pool = rng.normal(size=(nblk, bs, W))
    table = np.array([5, 2, 7])
    q = rng.normal(size=(1, 2, W))
    out, lse = M.mla_absorbed_decode(q, pool, table[None, :], [10], 0.5, D_C)
    for h in range(2):
        o1, l1 = M.mla_absorbed_one(q[0, h], pool, table, 10, 0.5, D_C)
        assert np.array_equal(o1, out[0, h]) and l1 == lse[0, h]
