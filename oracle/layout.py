"""KV-cache byte accounting (oracle; test infrastructure only).

* ``kv_cache_bytes``: "KV-Cache——为什么AI回复越来越快" section 07, the cache
  size 2 x L x N_layers x H_kv x D_h x dtype_bytes x batch (the factor 2 is K
  and V).
* ``kv_layout``: "KV缓存原理与显存估算" knowledge point 1: cost per token
  c = 2 L H_kv d s bytes, useful bytes c * sum T_i, padded bytes
  c * B * max T_i, independently paged bytes c * b * sum ceil(T_i / b), and
  the tail waste in token slots.
* ``unique_block_bytes``: the same page's closing section on block sharing:
  physical bytes count each shared physical block once.
"""

from __future__ import annotations


def kv_cache_bytes(seq_len, n_layers, n_kv_heads, d_head, dtype_bytes=2, batch=1):
    return 2 * seq_len * n_layers * n_kv_heads * d_head * dtype_bytes * batch


def _check_count(x, name, minimum):
    if type(x) is not int or x < minimum:
        raise ValueError(f"{name} must be an integer >= {minimum}")


def kv_layout(lengths, layers, kv_heads, head_dim, element_bytes, block_size):
    lengths = list(lengths)
    for n in lengths:
        _check_count(n, "length", 0)
    for x, name in ((layers, "layers"), (kv_heads, "kv_heads"), (head_dim, "head_dim"),
                    (element_bytes, "element_bytes"), (block_size, "block_size")):
        _check_count(x, name, 1)
    per_token = 2 * layers * kv_heads * head_dim * element_bytes
    useful_tokens = sum(lengths)
    longest = max(lengths) if lengths else 0
    blocks = sum(-(-n // block_size) for n in lengths)
    slots = blocks * block_size
    return {
        "bytes_per_token": per_token,
        "useful_bytes": useful_tokens * per_token,
        "padded_bytes": len(lengths) * longest * per_token,
        "paged_bytes": slots * per_token,
        "blocks": blocks,
        "slots": slots,
        "tail_waste_tokens": slots - useful_tokens,
    }


def unique_block_bytes(block_tables, lengths, block_size, bytes_per_token):
    """Physical bytes of a set of sequences whose tables may share blocks.

    block_tables: list of per-sequence lists of physical block ids; lengths:
    tokens held by each sequence. Only the first ceil(len / block_size)
    entries of each table are in use. Returns (table_entries, unique_blocks,
    unique_bytes, summed_bytes) where summed_bytes is the (wrong) count that
    adds every table entry.
    """
    used = []
    for row, n in zip(block_tables, lengths):
        used.extend(int(b) for b in list(row)[: -(-n // block_size)])
    unique = set(used)
    per_block = block_size * bytes_per_token
    return len(used), len(unique), len(unique) * per_block, len(used) * per_block
