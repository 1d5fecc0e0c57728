"""Paged KV cache: slot encoding, append and block-table gather (oracle; test infrastructure only).

Definitions follow the PagedAttention description of "KV Cache（键值缓存）"
(llm-compass) section 2.3: every sequence's cache is cut into blocks of
``block_size`` tokens and a per-sequence block table maps logical block j
to a physical block anywhere in the pool. The in-place write is the
preallocated cache of "单请求 KV Cache" (production practice: write only the
current position, never copy history); the read is the single-step attention
of "KV缓存原理与显存估算" knowledge point 2, over the rows gathered in
logical order.

Readings where the pages fix nothing:

* physical layout of the pools: ``k_cache[num_blocks, n_kv_heads, block_size, head_dim]``
  (head-major inside a block, like the [batch, heads, seq_len, head_dim]
  DynamicLayer layout the wiki cites); the same for ``v_cache``;
* slot encoding: ``slot = physical_block * block_size + (position % block_size)``,
  int64, a negative slot means "no write";
* query head h reads kv head ``h // (n_q_heads // n_kv_heads)`` (contiguous
  groups, MHA/GQA/MQA);
* ``context_lens[i]`` counts the cached rows including the token appended
  this step; it must be >= 1.
"""

from __future__ import annotations

import math

import numpy as np

from .attention import attend_rows


def slot_of(block_table_row, position: int, block_size: int) -> int:
    """Slot of logical ``position`` for a sequence with the given block table row."""
    return int(block_table_row[position // block_size]) * block_size + position % block_size


def slots_for_positions(block_table_row, positions, block_size: int) -> np.ndarray:
    return np.array([slot_of(block_table_row, int(p), block_size) for p in positions], dtype=np.int64)


def append_to_paged(k, v, slot_mapping, k_cache, v_cache):
    """Write token t's K/V rows for every kv head at slot_mapping[t]; skip negative slots.

    k, v: [T, Hkv, D]; k_cache, v_cache: [num_blocks, Hkv, bs, D]. Returns new
    arrays (inputs are not modified). Values are copied bit for bit (same dtype).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    bs = kc.shape[2]
    for t, slot in enumerate(np.asarray(slot_mapping).reshape(-1)):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // bs, slot % bs
        kc[blk, :, off, :] = k[t]
        vc[blk, :, off, :] = v[t]
    return kc, vc


def copy_blocks(cache, pairs):
    """Copy-on-write step: block dst becomes a copy of block src for every (src, dst) pair.

    PagedAttention sharing ("KV Cache（键值缓存）" section 2.3): a block held by
    several sequences is copied before one of them writes into it. cache is a
    pool [num_blocks, ...]; returns a new array (the input is not modified).
    """
    out = np.array(cache, copy=True)
    for src, dst in pairs:
        out[int(dst)] = cache[int(src)]
    return out


def gather_logical(cache, block_table_row, n: int, kv_head: int) -> np.ndarray:
    """Rows 0..n-1 of one sequence and one kv head, in logical order: [n, D]."""
    bs = cache.shape[2]
    rows = []
    for pos in range(n):
        blk = int(block_table_row[pos // bs])
        rows.append(np.asarray(cache[blk, kv_head, pos % bs, :], dtype=np.float64))
    return np.stack(rows, axis=0) if rows else np.zeros((0, cache.shape[3]))


def paged_decode_lse(q, k_cache, v_cache, block_tables, context_lens, scale):
    """Decode attention over the paged cache; returns (out [B, Hq, D], lse [B, Hq]).

    q: [B, Hq, D]; pools [num_blocks, Hkv, bs, D]; block_tables [B, max_blocks];
    context_lens [B]. lse is the natural log of sum_t exp(scale * q.k_t).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("n_q_heads must be a multiple of n_kv_heads")
    g = Hq // Hkv
    out = np.zeros((B, Hq, v_cache.shape[3]), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    for i in range(B):
        n = int(context_lens[i])
        if n < 1:
            raise ValueError("context_len must be >= 1 (the new token is always attended)")
        for kvh in range(Hkv):
            K = gather_logical(k_cache, block_tables[i], n, kvh)
            V = gather_logical(v_cache, block_tables[i], n, kvh)
            for h in range(kvh * g, (kvh + 1) * g):
                out[i, h], lse[i, h] = attend_rows(q[i, h], K, V, scale)
    return out, lse


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale):
    """Decode attention output [B, Hq, D] over the paged cache (see paged_decode_lse)."""
    return paged_decode_lse(q, k_cache, v_cache, block_tables, context_lens, scale)[0]


def paged_decode_one(q_row, k_cache, v_cache, table_row, n, kv_head, scale):
    """One (sequence, query head) output, for sampled checks at large sizes."""
    K = gather_logical(k_cache, table_row, n, kv_head)
    V = gather_logical(v_cache, table_row, n, kv_head)
    return attend_rows(q_row, K, V, scale)


def window_start(n: int, window: int) -> int:
    """First visible row of a sequence of n cached rows under a sliding window of W rows.

    "KV-Cache——为什么AI回复越来越快" section 08 (Window Attention / Sliding
    Window): only the most recent W tokens' K/V are kept and attended; the
    closing section of "KV缓存原理与显存估算" notes that this drops the
    out-of-window state because the visible range itself is redefined.
    Reading: the newest row is the current token, so the visible rows are
    [max(0, n - W), n); W >= n is full attention.
    """
    if window < 1:
        raise ValueError("window must be >= 1")
    return max(0, n - window)


def paged_decode_window_lse(q, k_cache, v_cache, block_tables, context_lens, scale, window):
    """Sliding-window decode: as paged_decode_lse, over the last ``window`` rows only."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, Hq, v_cache.shape[3]), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    for i in range(B):
        n = int(context_lens[i])
        if n < 1:
            raise ValueError("context_len must be >= 1 (the new token is always attended)")
        s0 = window_start(n, window)
        for kvh in range(Hkv):
            K = gather_logical(k_cache, block_tables[i], n, kvh)[s0:]
            V = gather_logical(v_cache, block_tables[i], n, kvh)[s0:]
            for h in range(kvh * g, (kvh + 1) * g):
                out[i, h], lse[i, h] = attend_rows(q[i, h], K, V, scale)
    return out, lse


def paged_decode_window(q, k_cache, v_cache, block_tables, context_lens, scale, window):
    return paged_decode_window_lse(q, k_cache, v_cache, block_tables, context_lens, scale, window)[0]


def paged_decode_multi(q, k_cache, v_cache, block_tables, context_lens, scale):
    """Several new query tokens per sequence attending the paged cache causally.

    q: [B, T, Hq, D]; context_lens count every cached row including the T new
    ones (already appended). Query token t of sequence i sits at position
    n_i - T + t and sees rows 0 .. n_i - T + t: the prefill/decode mask rule of
    "单请求 KV Cache" (a query row i of a chunk sees columns up to past_len + i),
    applied through the block table. Returns [B, T, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    B, T = q.shape[0], q.shape[1]
    out = np.zeros(q.shape[:3] + (v_cache.shape[3],), dtype=np.float64)
    lens = np.asarray(context_lens).reshape(-1)
    if np.any(lens < T):
        raise ValueError("every context must hold the T new rows")
    for t in range(T):
        out[:, t] = paged_decode(q[:, t], k_cache, v_cache, block_tables, lens - T + t + 1, scale)
    return out


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
