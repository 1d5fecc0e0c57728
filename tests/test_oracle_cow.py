"""Pins of the copy-on-write pool model and block copy (CPU only).

PagedAttention shares blocks between sequences by reference count and copies
a shared block before one holder writes into it ("KV Cache（键值缓存）" section
2.3, parallel sampling / beam search). The expected tables, slots and counts
below are worked out by hand for block size 16.
"""

import numpy as np
import pytest

from oracle import paged as P
from oracle.pool_model import NoBlocks, PoolModel


def test_fork_then_write_copies_only_the_partial_block():
    pool = PoolModel(num_blocks=8, block_size=16)
    a = pool.add()
    assert pool.reserve(a, 20) == list(range(20))        # blocks 0 (full) and 1 (4 rows)
    b = pool.fork(a)                                      # both hold blocks 0, 1
    slots, copy = pool.reserve_cow(b, 1)                  # b writes row 20 into block 1 -> copy first
    assert copy == (1, 2) and slots == [2 * 16 + 4]
    assert pool.table(b, 2) == [0, 2] and pool.table(a, 2) == [0, 1]
    assert pool.ref[:3] == [2, 1, 1]
    slots, copy = pool.reserve_cow(a, 1)                  # a is now the only holder of block 1: no copy
    assert copy is None and slots == [1 * 16 + 4]
    st = pool.stats()
    assert (st["unique_blocks"], st["table_entries"], st["useful_tokens"]) == (3, 4, 42)


def test_no_copy_when_the_last_block_is_full_or_private():
    pool = PoolModel(num_blocks=8, block_size=16)
    a = pool.add()
    pool.reserve(a, 32)                                   # two full blocks
    b = pool.fork(a)
    slots, copy = pool.reserve_cow(b, 3)                  # a fresh block, nothing to copy
    assert copy is None and slots == [2 * 16, 2 * 16 + 1, 2 * 16 + 2]
    c = pool.add()
    pool.reserve(c, 5)
    slots, copy = pool.reserve_cow(c, 2)                  # private partial block
    assert copy is None and slots == [3 * 16 + 5, 3 * 16 + 6]


def test_exhaustion_allocates_nothing():
    pool = PoolModel(num_blocks=2, block_size=16)
    a = pool.add()
    pool.reserve(a, 20)                                   # uses both blocks
    b = pool.fork(a)
    before = list(pool.ref)
    with pytest.raises(NoBlocks):
        pool.reserve_cow(b, 1)
    assert pool.ref == before and pool.table(b, 2) == [0, 1] and pool.length(b) == 20


def test_copied_block_keeps_history_and_isolates_writers():
    # rows 0..19 written through a's table, b forks and writes row 20 after the copy:
    # b sees a's 20 rows plus its own, a still sees its own 20 rows only
    rng = np.random.default_rng(0)
    pool = PoolModel(num_blocks=6, block_size=16)
    a = pool.add()
    slots_a = pool.reserve(a, 20)
    kc = np.full((6, 1, 16, 4), np.nan)
    hist = rng.standard_normal((20, 1, 4))
    kc, _ = P.append_to_paged(hist, hist, slots_a, kc, kc)
    b = pool.fork(a)
    slots_b, copy = pool.reserve_cow(b, 1)
    kc = P.copy_blocks(kc, [copy])
    new_b = rng.standard_normal((1, 1, 4))
    kc, _ = P.append_to_paged(new_b, new_b, slots_b, kc, kc)
    got_b = P.gather_logical(kc, pool.table(b, 2), 21, 0)
    got_a = P.gather_logical(kc, pool.table(a, 2), 20, 0)
    assert np.array_equal(got_b[:20], hist[:, 0]) and np.array_equal(got_b[20], new_b[0, 0])
    assert np.array_equal(got_a, hist[:, 0])
    slots_a2, copy_a = pool.reserve_cow(a, 1)             # a writes row 20 into its own block 1
    assert copy_a is None
    new_a = rng.standard_normal((1, 1, 4))
    kc, _ = P.append_to_paged(new_a, new_a, slots_a2, kc, kc)
    assert np.array_equal(P.gather_logical(kc, pool.table(b, 2), 21, 0)[20], new_b[0, 0])


def test_copy_blocks_copies_whole_blocks_and_nothing_else():
    cache = np.arange(5 * 2 * 3, dtype=np.float64).reshape(5, 2, 3)
    out = P.copy_blocks(cache, [(1, 3), (4, 0)])
    assert np.array_equal(out[3], cache[1]) and np.array_equal(out[0], cache[4])
    assert np.array_equal(out[[1, 2, 4]], cache[[1, 2, 4]])
