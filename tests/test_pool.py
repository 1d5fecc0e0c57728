"""The C++ block pool against the oracle's pool model and the pages' sharing counts (host only)."""

import json
import os
import random

import pytest
import torch

from oracle import layout as L
from oracle import paged as P
from oracle.pool_model import NoBlocks, PoolModel, Unsupported


def _same_state(pool, model, live, max_blocks):
    st = pool.stats()
    ms = model.stats()
    for k in ("num_blocks", "free_blocks", "unique_blocks", "table_entries", "useful_tokens", "live_seqs"):
        assert st[k] == ms[k], k
    if live:
        rows, lens = pool.tables(live, max_blocks)
        for sid, row, n in zip(live, rows, lens):
            assert row == model.table(sid, max_blocks)
            assert n == model.length(sid)
    for b in range(model.num_blocks):
        assert pool.refcount(b) == model.ref[b]


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_model(kvc, seed):
    rng = random.Random(seed)
    nblk, bs = 40, rng.choice([4, 16])
    pool = kvc.BlockPool(nblk, bs)
    model = PoolModel(nblk, bs)
    live = []
    max_blocks = nblk
    for _ in range(300):
        op = rng.random()
        if op < 0.15 or not live:
            a, b = pool.add(), model.add()
            assert a == b
            live.append(a)
        elif op < 0.25:
            parent = rng.choice(live)
            a, b = pool.fork(parent), model.fork(parent)
            assert a == b
            live.append(a)
        elif op < 0.35:
            sid = rng.choice(live)
            pool.free(sid)
            model.free(sid)
            live.remove(sid)
        elif op < 0.55:
            # copy-on-write reservation: same slots and the same (shared, fresh) pair as the model
            sid = rng.choice(live)
            n = rng.choice([1, 2, bs, 2 * bs + 3])
            try:
                expect = model.reserve_cow(sid, n)
                err = None
            except NoBlocks as e:
                expect, err = None, e
            if err is None:
                assert pool.reserve_cow(sid, n) == expect
            else:
                with pytest.raises(kvc.KvcError) as ei:
                    pool.reserve_cow(sid, n)
                assert ei.value.status == kvc.ERR_NO_BLOCKS
        else:
            sid = rng.choice(live)
            n = rng.choice([1, 1, 2, 5, bs, 3 * bs + 1])
            try:
                expect = model.reserve(sid, n)
                err = None
            except (NoBlocks, Unsupported) as e:
                expect, err = None, e
            if err is None:
                assert pool.reserve(sid, n) == expect
            else:
                with pytest.raises(kvc.KvcError) as ei:
                    pool.reserve(sid, n)
                code = kvc.ERR_NO_BLOCKS if isinstance(err, NoBlocks) else kvc.ERR_UNSUPPORTED
                assert ei.value.status == code
        _same_state(pool, model, live, max_blocks)
    # slots are consistent with the tables (oracle slot encoding)
    if live:
        rows, lens = pool.tables(live, max_blocks)
        for row, n in zip(rows, lens):
            if n:
                got = kvc.slots_from_tables(torch.tensor([row], dtype=torch.int32), bs, [0] * n, list(range(n)))
                assert got.tolist() == list(P.slots_for_positions(row, range(n), bs))
    pool.close()


def test_sharing_counts_from_the_page(kvc, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_layout_examples.json")))
    s = g["sharing"]
    pool = kvc.BlockPool(16, s["block_size"])
    a = pool.add()
    pool.reserve(a, s["shared_prompt_tokens"])
    b = pool.fork(a)
    pool.reserve(a, s["private_tokens_each"])
    pool.reserve(b, s["private_tokens_each"])
    st = pool.stats()
    assert st["table_entries"] == s["table_entries"]
    assert st["unique_blocks"] == s["unique_blocks"]
    rows, lens = pool.tables([a, b], 3)
    entries, unique, unique_bytes, summed = L.unique_block_bytes(rows, lens, 16, g["bytes_per_token"])
    assert unique_bytes == s["unique_mib"] << 20 and summed == s["summed_mib"] << 20
    assert pool.refcount(rows[0][0]) == 2 and pool.refcount(rows[0][2]) == 1


def test_tail_waste_example(kvc, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_layout_examples.json")))["case_17_31_32"]
    pool = kvc.BlockPool(16, 16)
    ids = []
    for n in g["lengths"]:
        sid = pool.add()
        pool.reserve(sid, n)
        ids.append(sid)
    st = pool.stats()
    assert st["unique_blocks"] * 16 == g["slots"]
    assert st["useful_tokens"] == g["useful_tokens"]
    assert st["unique_blocks"] * 16 - st["useful_tokens"] == g["tail_waste_tokens"]


def test_pool_errors(kvc):
    with pytest.raises(kvc.KvcError):
        kvc.BlockPool(0, 16)
    pool = kvc.BlockPool(2, 16)
    a = pool.add()
    with pytest.raises(kvc.KvcError) as e:
        pool.reserve(a, 33)
    assert e.value.status == kvc.ERR_NO_BLOCKS
    assert pool.length(a) == 0 and pool.stats()["free_blocks"] == 2
    with pytest.raises(kvc.KvcError) as e:
        pool.free(12345)
    assert e.value.status == kvc.ERR_INVALID_ARG
    with pytest.raises(kvc.KvcError):
        kvc.slots_from_tables(torch.zeros((1, 2), dtype=torch.int32), 16, [0], [32])


def test_config3_sharing_layout(kvc):
    # 8 prompts x 2048 tokens (128 full blocks, shared 8 ways) + 256 private tokens each
    pool = kvc.BlockPool(2048 + 10, 16)
    seqs = []
    for p in range(8):
        root = pool.add()
        pool.reserve(root, 2048)
        kids = [pool.fork(root) for _ in range(8)]
        pool.free(root)
        for k in kids:
            pool.reserve(k, 256)
        seqs.extend(kids)
    st = pool.stats()
    assert st["unique_blocks"] == 8 * 128 + 64 * 16 == 2048
    assert st["table_entries"] == 64 * 144
    rows, lens = pool.tables(seqs, 144)
    assert all(n == 2304 for n in lens)
    assert pool.refcount(rows[0][0]) == 8 and pool.refcount(rows[0][130]) == 1


@pytest.mark.parametrize("seed", range(4))
def test_reserve_batch_equals_sequential_reserves(kvc, seed):
    # the batch call on one pool, single reserves (the model's) on the other: same slots, same state
    rng = random.Random(100 + seed)
    nblk, bs = 64, rng.choice([4, 16])
    pool = kvc.BlockPool(nblk, bs)
    model = PoolModel(nblk, bs)
    live = []
    for _ in range(6):
        a, b = pool.add(), model.add()
        assert a == b
        live.append(a)
    for _ in range(40):
        batch = rng.sample(live, rng.randint(1, len(live)))
        n_new = rng.choice([1, 2, bs - 1, bs + 1])
        try:
            expect = [model.reserve(s, n_new) for s in batch]
            ok = True
        except NoBlocks:
            ok = False
        if ok:
            assert pool.reserve_batch(batch, n_new) == expect
        else:
            # the model may have served part of the batch before it ran out: rebuild it from the pool's state
            before = pool.stats()
            with pytest.raises(kvc.KvcError) as e:
                pool.reserve_batch(batch, n_new)
            assert e.value.status == kvc.ERR_NO_BLOCKS
            assert pool.stats() == before  # all or nothing
            break
        _same_state(pool, model, live, nblk)


def test_reserve_batch_refusals_change_nothing(kvc):
    pool = kvc.BlockPool(8, 16)
    a = pool.add()
    pool.reserve(a, 20)
    b = pool.fork(a)  # shares a's partly filled second block
    c = pool.add()
    before = pool.stats()
    for seqs, n_new, status in (([c, c], 1, kvc.ERR_INVALID_ARG), ([c, 999], 1, kvc.ERR_INVALID_ARG),
                                ([c, b], 1, kvc.ERR_UNSUPPORTED), ([c], 16 * 7 + 1, kvc.ERR_NO_BLOCKS)):
        with pytest.raises(kvc.KvcError) as e:
            pool.reserve_batch(seqs, n_new)
        assert e.value.status == status
        assert pool.stats() == before
        assert pool.length(c) == 0
    assert pool.reserve_batch([], 3) == [] and pool.reserve_batch([c], 0) == [[]]
    assert pool.reserve_batch([c], 2) == [[2 * 16, 2 * 16 + 1]]  # lowest free block is 2
