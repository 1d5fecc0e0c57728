"""GPU parity: copy-on-write of shared blocks (kvc_seq_reserve_cow + kvc_copy_blocks) before a forked
sequence writes, then decode of parents and forks, against the oracle running the same pool operations."""

import math

import numpy as np
import pytest
import torch

from oracle import paged as OP
from oracle.pool_model import PoolModel
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import TOL, f64, max_err

pytestmark = pytest.mark.gpu


def _tables(rows, lens):
    return torch.tensor(rows, dtype=torch.int32), torch.tensor(lens, dtype=torch.int32)


@pytest.mark.parametrize("prompt_len,fanout,steps,dtype", [(20, 2, 3, "bf16"), (2050, 4, 5, "bf16"),
                                                          (33, 3, 1, "f32")])
def test_fork_write_decode(kvc, prompt_len, fanout, steps, dtype):
    Hq, Hkv, D, bs = 16, 4, 128, 16
    n_prompts = 2
    rng_seed = 70 + prompt_len
    max_len = prompt_len + steps
    nblk = n_prompts * fanout * (-(-max_len // bs) + 1) + 8
    pool = kvc.BlockPool(nblk, bs)
    model = PoolModel(nblk, bs)
    g = torch.Generator().manual_seed(rng_seed)
    k_cache = W.normal((nblk, Hkv, bs, D), dtype, g)
    v_cache = W.normal((nblk, Hkv, bs, D), dtype, g)
    kc_ref, vc_ref = f64(k_cache), f64(v_cache)
    kc_dev, vc_dev = k_cache.cuda(), v_cache.cuda()

    def write(seqs, slot_lists):
        # one new K/V row per listed slot, written on both sides
        nonlocal kc_ref, vc_ref
        slots = [s for sl in slot_lists for s in sl]
        kn = W.normal((len(slots), Hkv, D), dtype, g)
        vn = W.normal((len(slots), Hkv, D), dtype, g)
        kvc.append(kn.cuda(), vn.cuda(), torch.tensor(slots, dtype=torch.int64, device="cuda"), kc_dev, vc_dev)
        kc_ref, vc_ref = OP.append_to_paged(f64(kn), f64(vn), np.array(slots), kc_ref, vc_ref)

    def cow(pairs):
        nonlocal kc_ref, vc_ref
        if not pairs:
            return
        p = torch.tensor(pairs, dtype=torch.int64, device="cuda")
        kvc.copy_blocks(kc_dev, p)
        kvc.copy_blocks(vc_dev, p)
        kc_ref, vc_ref = OP.copy_blocks(kc_ref, pairs), OP.copy_blocks(vc_ref, pairs)

    parents = []
    for _ in range(n_prompts):
        a, b = pool.add(), model.add()
        assert a == b
        assert pool.reserve(a, prompt_len) == model.reserve(b, prompt_len)
        parents.append(a)
    # prompt rows, written once through the parents' tables
    for a in parents:
        row = model.table(a, nblk)
        write([a], [list(OP.slots_for_positions(row, range(prompt_len), bs))])
    forks = []
    for a in parents:
        for _ in range(fanout - 1):
            c, d = pool.fork(a), model.fork(a)
            assert c == d
            forks.append(c)
    seqs = parents + forks
    n_copies = 0
    for _ in range(steps):
        slot_lists, pairs = [], []
        for sid in seqs:
            got = pool.reserve_cow(sid, 1)
            assert got == model.reserve_cow(sid, 1)
            slot_lists.append(got[0])
            if got[1] is not None:
                pairs.append(got[1])
        n_copies += len(pairs)
        cow(pairs)
        write(seqs, slot_lists)
    # every sequence but one per prompt had to copy its shared tail block once
    if prompt_len % bs:
        assert n_copies == n_prompts * (fanout - 1)
    rows, lens = pool.tables(seqs, nblk)
    bt, cl = _tables(rows, lens)
    q = W.normal((len(seqs), Hq, D), dtype, g)
    out = torch.empty((len(seqs), Hq, D), dtype=torch.float32, device="cuda")
    ws = kvc.new_decode_workspace(len(seqs), Hq, Hkv, D, bs, nblk)
    scale = 1.0 / math.sqrt(D)
    kvc.decode_attention(q.cuda(), kc_dev, vc_dev, bt.cuda(), cl.cuda(), scale, out, ws)
    torch.cuda.synchronize()
    ref = OP.paged_decode(f64(q), kc_ref, vc_ref, bt.numpy(), cl.numpy(), scale)
    assert max_err(out, ref) <= TOL[dtype]
    # the pools match the oracle's bit for bit (copies and appends are exact)
    assert np.array_equal(f64(kc_dev), kc_ref) and np.array_equal(f64(vc_dev), vc_ref)
    assert kvc.get_error_flags() == 0
    pool.close()


def test_copy_blocks_bad_ids_are_skipped_and_flagged(kvc):
    cache = torch.arange(6 * 4 * 16 * 8, dtype=torch.float32, device="cuda").reshape(6, 4, 16, 8)
    before = cache.clone()
    pairs = torch.tensor([[1, 3], [7, 2], [4, -1], [5, 5]], dtype=torch.int64, device="cuda")
    kvc.copy_blocks(cache, pairs)
    torch.cuda.synchronize()
    assert torch.equal(cache[3], before[1])
    for b in (0, 1, 2, 4, 5):
        assert torch.equal(cache[b], before[b])
    assert kvc.get_error_flags() == kvc.FLAG_BAD_BLOCK
