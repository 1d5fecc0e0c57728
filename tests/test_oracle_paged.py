"""Pins for the paged-cache, MLA, byte-accounting and pool parts of the oracle."""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as A
from oracle import layout as L
from oracle import mla as M
from oracle import paged as P
from oracle.pool_model import NoBlocks, PoolModel, Unsupported


def _contiguous_and_paged(rng, lens, Hkv, D, bs):
    """Logical K/V per sequence, plus the same data scattered into a permuted paged pool."""
    need = [-(-n // bs) for n in lens]
    nblk = sum(need) + 3
    perm = rng.permutation(nblk)
    kc = np.full((nblk, Hkv, bs, D), np.nan)
    vc = np.full((nblk, Hkv, bs, D), np.nan)
    tables = np.zeros((len(lens), max(need)), dtype=np.int64)
    logical_k, logical_v = [], []
    pos = 0
    for i, n in enumerate(lens):
        tables[i, : need[i]] = perm[pos: pos + need[i]]
        pos += need[i]
        Kl = rng.normal(size=(n, Hkv, D))
        Vl = rng.normal(size=(n, Hkv, D))
        logical_k.append(Kl)
        logical_v.append(Vl)
        for p in range(n):
            kc[tables[i, p // bs], :, p % bs] = Kl[p]
            vc[tables[i, p // bs], :, p % bs] = Vl[p]
    return kc, vc, tables, logical_k, logical_v


def test_paged_gather_reads_logical_order_and_ignores_tail():
    rng = np.random.default_rng(7)
    lens = [17, 31, 32, 1, 16]
    kc, vc, tables, lk, lv = _contiguous_and_paged(rng, lens, 2, 4, 16)
    for i, n in enumerate(lens):
        for h in range(2):
            assert np.array_equal(P.gather_logical(kc, tables[i], n, h), lk[i][:, h])
    # NaN padding in the unused tail slots must not reach the output
    q = rng.normal(size=(len(lens), 2, 4))
    out = P.paged_decode(q, kc, vc, tables, lens, 0.5)
    assert np.all(np.isfinite(out))


def test_group_mapping_contiguous_groups():
    # kv head j holds constant value rows equal to j: query head h must read kv head h // g.
    Hq, Hkv, D, bs = 8, 2, 4, 16
    kc = np.zeros((2, Hkv, bs, D))
    vc = np.zeros((2, Hkv, bs, D))
    for j in range(Hkv):
        vc[:, j] = float(j + 1)
    rng = np.random.default_rng(3)
    kc[:] = rng.normal(size=kc.shape)
    q = rng.normal(size=(1, Hq, D))
    out = P.paged_decode(q, kc, vc, np.array([[1, 0]]), [20], 0.5)
    for h in range(Hq):
        assert np.allclose(out[0, h], h // (Hq // Hkv) + 1.0, rtol=0, atol=1e-14)
    with pytest.raises(ValueError):
        P.paged_decode(np.zeros((1, 3, D)), kc, vc, np.array([[0, 1]]), [5], 0.5)


def test_paged_decode_equals_cached_attention_per_head():
    rng = np.random.default_rng(11)
    lens = [5, 16, 33]
    Hq, Hkv, D = 6, 3, 8
    kc, vc, tables, lk, lv = _contiguous_and_paged(rng, lens, Hkv, D, 16)
    q = rng.normal(size=(3, Hq, D))
    out, lse = P.paged_decode_lse(q, kc, vc, tables, lens, 0.25)
    for i, n in enumerate(lens):
        for h in range(Hq):
            kvh = h // 2
            ref, _, _, _ = A.cached_attention(q[i, h], lk[i][:-1, kvh], lv[i][:-1, kvh], lk[i][-1, kvh],
                                              lv[i][-1, kvh], 0.25)
            assert np.max(np.abs(out[i, h] - ref)) < 1e-13
            z = lk[i][:, kvh] @ q[i, h] * 0.25
            assert abs(lse[i, h] - math.log(np.sum(np.exp(z)))) < 1e-12


def test_append_writes_exact_slots_and_skips_negative():
    rng = np.random.default_rng(5)
    nblk, Hkv, bs, D = 4, 2, 16, 8
    kc = np.full((nblk, Hkv, bs, D), -7.0, dtype=np.float32)
    vc = np.full((nblk, Hkv, bs, D), -9.0, dtype=np.float32)
    k = rng.normal(size=(3, Hkv, D)).astype(np.float32)
    v = rng.normal(size=(3, Hkv, D)).astype(np.float32)
    slots = np.array([2 * bs + 5, -1, 0 * bs + 15], dtype=np.int64)
    kc2, vc2 = P.append_to_paged(k, v, slots, kc, vc)
    assert np.array_equal(kc2[2, :, 5], k[0]) and np.array_equal(vc2[2, :, 5], v[0])
    assert np.array_equal(kc2[0, :, 15], k[2]) and np.array_equal(vc2[0, :, 15], v[2])
    changed = (kc2 != kc).any(axis=(1, 3))
    assert changed.sum() == 2
    assert np.array_equal(kc, np.full_like(kc, -7.0))  # input untouched


def test_slot_encoding():
    row = [9, 4, 7]
    assert P.slot_of(row, 0, 16) == 9 * 16
    assert P.slot_of(row, 17, 16) == 4 * 16 + 1
    assert list(P.slots_for_positions(row, [31, 32, 47], 16)) == [4 * 16 + 15, 7 * 16, 7 * 16 + 15]


def test_decode_via_paged_append_equals_recompute_tiny_model():
    # prompt of 5 tokens appended at once, then 64 steps of append 1 + decode, 2 layers, 4 heads, d 32
    rng = np.random.default_rng(42)
    T, H, D, bs, layers = 69, 4, 32, 16, 2
    pool = PoolModel(num_blocks=8, block_size=bs)
    sid = pool.add()
    data = [(rng.normal(size=(T, H, D)), rng.normal(size=(T, H, D)), rng.normal(size=(T, H, D)))
            for _ in range(layers)]
    caches = [(np.zeros((8, H, bs, D)), np.zeros((8, H, bs, D))) for _ in range(layers)]
    scale = 1.0 / math.sqrt(D)
    slots = pool.reserve(sid, 5)
    for l in range(layers):
        Q, K, V = data[l]
        caches[l] = P.append_to_paged(K[:5], V[:5], slots, *caches[l])
    worst = 0.0
    for t in range(5, T):
        slot = pool.reserve(sid, 1)
        table = np.array([pool.table(sid, 5)])
        for l in range(layers):
            Q, K, V = data[l]
            caches[l] = P.append_to_paged(K[t:t + 1], V[t:t + 1], slot, *caches[l])
            out = P.paged_decode(Q[t][None], caches[l][0], caches[l][1], table, [t + 1], scale)
            for h in range(H):
                ref = A.decode_by_recompute(Q[: t + 1, h], K[: t + 1, h], V[: t + 1, h], scale)
                worst = max(worst, float(np.max(np.abs(out[0, h] - ref))))
    assert worst < 1e-12


def test_mla_absorbed_equals_explicit():
    # llm-compass section 2.2: W^UK / W^UV absorbed into the query / output side.
    rng = np.random.default_rng(46)
    B, H, d_h, d_c, d_r, bs = 2, 3, 6, 10, 4, 4
    lens = [7, 9]
    nblk = 8
    latent = rng.normal(size=(nblk, bs, d_c + d_r))
    tables = np.array([[5, 1, 0], [2, 7, 3]])
    W_UK = rng.normal(size=(H, d_h, d_c))
    W_UV = rng.normal(size=(H, 5, d_c))
    q_nope = rng.normal(size=(B, H, d_h))
    q_rope = rng.normal(size=(B, H, d_r))
    scale = 1.0 / math.sqrt(d_h + d_r)
    explicit = M.mla_explicit_decode(q_nope, q_rope, latent, tables, lens, W_UK, W_UV, scale, d_c)
    q_abs = M.absorb_query(q_nope, q_rope, W_UK)
    lat_out, _ = M.mla_absorbed_decode(q_abs, latent, tables, lens, scale, d_c)
    absorbed = np.einsum("hvc,bhc->bhv", W_UV, lat_out)
    assert np.max(np.abs(absorbed - explicit)) < 1e-10
    # a wrong absorption (W^UK not transposed into latent space) would not even type-check
    # at these shapes; a dropped RoPE part must change the result:
    q_bad = q_abs.copy()
    q_bad[..., d_c:] = 0.0
    bad, _ = M.mla_absorbed_decode(q_bad, latent, tables, lens, scale, d_c)
    assert np.max(np.abs(np.einsum("hvc,bhc->bhv", W_UV, bad) - explicit)) > 1e-3


def test_mla_latent_is_576_elements(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "per_token_bytes.json")))["mla"]
    assert g["d_c"] + g["d_r"] == g["elements"]
    assert 2 * 128 * 128 == g["mha_elements"]


def test_cache_size_scenarios(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_cache_scenarios.json")))
    for s in g["scenarios"]:
        got = L.kv_cache_bytes(s["L"], s["layers"], s["kv_heads"], s["d_head"], s["bytes"], s["batch"])
        if "contradiction" in s:
            # the page's own formula disagrees with this one printed line: follow the formula
            assert got == s["formula_bytes"] == 2 * s["printed_bytes"], s["name"]
        else:
            assert got == s["printed_bytes"], s["name"]


def test_per_token_bytes(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "per_token_bytes.json")))
    for c in g["cases"]:
        got = L.kv_layout([1], c["layers"], c["kv_heads"], c["head_dim"], c["bytes"], 16)["bytes_per_token"]
        assert got == c["expect_bytes"], c["cite"]


def test_kv_layout_examples(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_layout_examples.json")))
    m = g["model"]
    MiB = 1 << 20
    a = L.kv_layout(g["case_1024_3072"]["lengths"], m["layers"], m["kv_heads"], m["head_dim"],
                    m["element_bytes"], m["block_size"])
    assert a["bytes_per_token"] == g["bytes_per_token"]
    assert a["useful_bytes"] == g["case_1024_3072"]["useful_mib"] * MiB
    assert a["paged_bytes"] == g["case_1024_3072"]["paged_mib"] * MiB
    assert a["padded_bytes"] == g["case_1024_3072"]["padded_mib"] * MiB
    b = L.kv_layout(g["case_17_31_32"]["lengths"], m["layers"], m["kv_heads"], m["head_dim"],
                    m["element_bytes"], m["block_size"])
    c = g["case_17_31_32"]
    assert b["slots"] == c["slots"]
    assert sum(c["lengths"]) == c["useful_tokens"]
    assert b["tail_waste_tokens"] == c["tail_waste_tokens"]
    assert b["tail_waste_tokens"] * b["bytes_per_token"] == c["tail_waste_mib"] * MiB
    with pytest.raises(ValueError):
        L.kv_layout([-1], 1, 1, 1, 1, 16)
    with pytest.raises(ValueError):
        L.kv_layout([3], 1, 0, 1, 1, 16)


def test_pool_model_sharing_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_layout_examples.json")))
    s = g["sharing"]
    pool = PoolModel(num_blocks=16, block_size=s["block_size"])
    a = pool.add()
    pool.reserve(a, s["shared_prompt_tokens"])
    b = pool.fork(a)
    pool.reserve(a, s["private_tokens_each"])
    pool.reserve(b, s["private_tokens_each"])
    st = pool.stats()
    assert st["table_entries"] == s["table_entries"]
    assert st["unique_blocks"] == s["unique_blocks"]
    tables = [pool.table(a, 3), pool.table(b, 3)]
    lens = [pool.length(a), pool.length(b)]
    entries, unique, unique_bytes, summed = L.unique_block_bytes(tables, lens, 16, g["bytes_per_token"])
    assert (entries, unique) == (s["table_entries"], s["unique_blocks"])
    assert unique_bytes == s["unique_mib"] << 20
    assert summed == s["summed_mib"] << 20


def test_pool_model_rules():
    pool = PoolModel(num_blocks=4, block_size=16)
    a = pool.add()
    assert pool.reserve(a, 17) == list(range(17))
    b = pool.fork(a)  # shares a partial block
    with pytest.raises(Unsupported):
        pool.reserve(b, 1)
    pool.free(b)
    assert pool.reserve(a, 15)[-1] == 1 * 16 + 15  # a is sole holder again
    c = pool.add()
    with pytest.raises(NoBlocks):
        pool.reserve(c, 33)  # needs 3, only 2 free: nothing allocated
    assert pool.stats()["free_blocks"] == 2
    assert pool.reserve(c, 32) == list(range(32, 64))
    pool.free(a)
    assert pool.stats()["free_blocks"] == 2
    d = pool.add()
    assert pool.reserve(d, 1) == [0]
