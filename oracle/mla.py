"""MLA (multi-head latent attention) decode over a paged latent cache (oracle; test infrastructure only).

"KV Cache（键值缓存）" (llm-compass) section 2.2: the cache holds one shared
latent c_t = W^DKV h_t in R^{d_c} per token plus a decoupled RoPE part of width
d_R, concatenated (DeepSeek-V2: d_c = 512, d_R = 64, 576 elements per token
per layer). Per head, k_t^C = W^UK c_t and v_t^C = W^UV c_t; the page notes
that W^UK and W^UV can be absorbed into the query and output projections so
K/V never need to be rebuilt. Section 4 adds that the kernel must be
rewritten for this (absorbed) form.

Plainest absorbed reading (the pages give no worked MLA example):

* the absorbed query of head h is q~_h = [ (W^UK_h)^T q^C_h , q^R_h ]  (576 wide);
* the score of cached token t is scale * q~_h . [c_t, k^R_t];
* the latent output is o~_h = sum_t a_{h,t} c_t (d_c wide), and the head
  output is W^UV_h o~_h, applied by the caller with the output projection.

``mla_explicit_decode`` computes the same attention the long way (per-head
keys and values rebuilt from the latent), so the absorption algebra can be
checked against it.
"""

from __future__ import annotations

import numpy as np

from .attention import attend_rows


def _latent_rows(latent_cache, table_row, n):
    bs = latent_cache.shape[1]
    rows = [np.asarray(latent_cache[int(table_row[p // bs]), p % bs, :], dtype=np.float64) for p in range(n)]
    return np.stack(rows, axis=0)


def mla_absorbed_decode(q_abs, latent_cache, block_tables, context_lens, scale, d_c):
    """Latent-space decode: returns (out [B, H, d_c], lse [B, H]).

    q_abs: [B, H, d_c + d_r]; latent_cache: [num_blocks, bs, d_c + d_r];
    keys are whole cached rows, values are their first d_c elements.
    """
    q_abs = np.asarray(q_abs, dtype=np.float64)
    B, H, W = q_abs.shape
    if latent_cache.shape[2] != W:
        raise ValueError("query width must equal the cached row width d_c + d_r")
    out = np.zeros((B, H, d_c), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    for i in range(B):
        n = int(context_lens[i])
        if n < 1:
            raise ValueError("context_len must be >= 1")
        C = _latent_rows(latent_cache, block_tables[i], n)
        for h in range(H):
            out[i, h], lse[i, h] = attend_rows(q_abs[i, h], C, C[:, :d_c], scale)
    return out, lse


def mla_absorbed_one(q_row, latent_cache, table_row, n, scale, d_c):
    C = _latent_rows(latent_cache, table_row, n)
    return attend_rows(q_row, C, C[:, :d_c], scale)


def absorb_query(q_nope, q_rope, W_UK):
    """q~_h = [ W_UK[h]^T q_nope[h], q_rope[h] ].

    q_nope: [B, H, d_h]; q_rope: [B, H, d_r]; W_UK: [H, d_h, d_c] (k^C = W_UK[h] c).
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    W_UK = np.asarray(W_UK, dtype=np.float64)
    lat = np.einsum("bhk,hkc->bhc", q_nope, W_UK)
    return np.concatenate([lat, q_rope], axis=-1)


def mla_explicit_decode(q_nope, q_rope, latent_cache, block_tables, context_lens, W_UK, W_UV, scale, d_c):
    """Non-absorbed MLA decode: rebuild per-head K and V from the latent, then attend.

    Head h's key for token t is [W_UK[h] c_t, k^R_t] and its value W_UV[h] c_t.
    Returns [B, H, d_v].
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    W_UK = np.asarray(W_UK, dtype=np.float64)
    W_UV = np.asarray(W_UV, dtype=np.float64)
    B, H, _ = q_nope.shape
    out = np.zeros((B, H, W_UV.shape[1]), dtype=np.float64)
    for i in range(B):
        n = int(context_lens[i])
        rows = _latent_rows(latent_cache, block_tables[i], n)
        c, kr = rows[:, :d_c], rows[:, d_c:]
        for h in range(H):
            K = np.concatenate([c @ W_UK[h].T, kr], axis=1)
            V = c @ W_UV[h].T
            q = np.concatenate([q_nope[i, h], q_rope[i, h]])
            out[i, h], _ = attend_rows(q, K, V, scale)
    return out
