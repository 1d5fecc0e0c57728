"""Seeded synthetic inputs shared by the tests and the benchmark.

Only random draws live here: normal values rounded to the storage dtype,
uniform context lengths, and random physical block assignments. Nothing here
computes attention, slots or byte counts; the library and the oracle each do
that themselves from these inputs.

Every tensor is produced from a ``torch.Generator`` seeded with the given
seed, as float32 N(0, 1) and then rounded to the storage dtype, so the library
(after a copy to the device) and the oracle (after a widening to float64) see
the same values. Parity tests draw on the CPU; the benchmark may draw the large
value tensors on the GPU (``device="cuda"``) where they are needed anyway.
"""

from __future__ import annotations

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, dtype: str, gen: torch.Generator) -> torch.Tensor:
    """N(0, 1) drawn as float32 on the generator's device, rounded to ``dtype``.

    Large tensors are drawn in slices so the float32 staging copy stays small.
    """
    dev = gen.device
    out = torch.empty(*shape, dtype=DTYPES[dtype], device=dev)
    flat = out.view(-1)
    step = 1 << 26
    for a in range(0, flat.numel(), step):
        b = min(flat.numel(), a + step)
        flat[a:b] = torch.randn(b - a, generator=gen, dtype=torch.float32, device=dev).to(DTYPES[dtype])
    return out


def uniform_lengths(batch: int, lo: int, hi: int, gen: torch.Generator) -> torch.Tensor:
    # lengths are always drawn on the CPU so a case has the same structure on every device
    return torch.randint(lo, hi + 1, (batch,), generator=gen, dtype=torch.int64).to(torch.int32)


def random_block_tables(lens, block_size: int, spare_frac: float, gen: torch.Generator, permute: bool = True):
    """Give each sequence ceil(len / block_size) distinct physical blocks.

    The pool has the exact need plus ``spare_frac`` spare blocks; physical ids
    are a random permutation of the pool when ``permute`` (else ascending).
    Returns (block_tables int32 [B, max_blocks], num_blocks). Unused entries
    are 0.
    """
    lens = [int(x) for x in lens]
    need = [-(-n // block_size) for n in lens]
    total = sum(need)
    num_blocks = max(1, total + int(round(total * spare_frac)))
    ids = torch.randperm(num_blocks, generator=gen) if permute else torch.arange(num_blocks)
    max_blocks = max(need) if need else 1
    table = torch.zeros((len(lens), max(1, max_blocks)), dtype=torch.int32)
    pos = 0
    for i, k in enumerate(need):
        table[i, :k] = ids[pos:pos + k].to(torch.int32)
        pos += k
    return table, num_blocks


def shared_prefix_block_tables(n_prompts: int, fanout: int, prompt_len: int, private_len: int,
                               block_size: int, gen: torch.Generator, spare_frac: float = 0.0):
    """Tables for ``n_prompts`` prompts each continued by ``fanout`` sequences.

    All sequences of one prompt share that prompt's blocks; each then owns
    ceil(private_len / block_size) private blocks. ``prompt_len`` must be a
    whole number of blocks (no shared partial block). Physical ids are a
    random permutation. Returns (tables int32 [n_prompts * fanout, max_blocks],
    lens int32, num_blocks).
    """
    if prompt_len % block_size != 0:
        raise ValueError("prompt_len must be a multiple of block_size")
    pb = prompt_len // block_size
    qb = -(-private_len // block_size)
    total = n_prompts * pb + n_prompts * fanout * qb
    num_blocks = total + int(round(total * spare_frac))
    ids = torch.randperm(num_blocks, generator=gen).to(torch.int32)
    B = n_prompts * fanout
    table = torch.zeros((B, pb + qb), dtype=torch.int32)
    pos = 0
    prompt_ids = []
    for p in range(n_prompts):
        prompt_ids.append(ids[pos:pos + pb])
        pos += pb
    for p in range(n_prompts):
        for f in range(fanout):
            i = p * fanout + f
            table[i, :pb] = prompt_ids[p]
            table[i, pb:] = ids[pos:pos + qb]
            pos += qb
    lens = torch.full((B,), prompt_len + private_len, dtype=torch.int32)
    return table, lens, num_blocks


def gqa_case(batch, n_q_heads, n_kv_heads, head_dim, block_size, lens, dtype, seed,
             spare_frac=0.10, permute=True, device="cpu"):
    """A paged GQA/MHA/MQA decode step.

    ``lens`` is a list of context lengths (each including the new token) or a
    (lo, hi) tuple for uniform random lengths. Draw order (fixed): lengths,
    table permutation, K pool, V pool, q, new k, new v. Lengths and tables
    always come from a CPU generator; values from a generator on ``device``
    (the same seed gives different values on "cpu" and "cuda").
    """
    g = _gen(seed)
    gv = g if device == "cpu" else _gen(seed, device)
    if isinstance(lens, tuple):
        lens_t = uniform_lengths(batch, lens[0], lens[1], g)
    else:
        lens_t = torch.tensor([int(x) for x in lens], dtype=torch.int32)
    table, num_blocks = random_block_tables(lens_t.tolist(), block_size, spare_frac, g, permute)
    shape = (num_blocks, n_kv_heads, block_size, head_dim)
    return {
        "context_lens": lens_t,
        "block_tables": table,
        "num_blocks": num_blocks,
        "k_cache": normal(shape, dtype, gv),
        "v_cache": normal(shape, dtype, gv),
        "q": normal((batch, n_q_heads, head_dim), dtype, gv),
        "k_new": normal((batch, n_kv_heads, head_dim), dtype, gv),
        "v_new": normal((batch, n_kv_heads, head_dim), dtype, gv),
        "dtype": dtype,
        "block_size": block_size,
    }


def shared_case(n_prompts, fanout, prompt_len, private_len, n_heads, head_dim, block_size, dtype, seed,
                device="cpu"):
    """MHA decode step where groups of sequences share their prompt blocks."""
    g = _gen(seed)
    gv = g if device == "cpu" else _gen(seed, device)
    table, lens, num_blocks = shared_prefix_block_tables(n_prompts, fanout, prompt_len, private_len,
                                                         block_size, g)
    B = n_prompts * fanout
    shape = (num_blocks, n_heads, block_size, head_dim)
    return {
        "context_lens": lens,
        "block_tables": table,
        "num_blocks": num_blocks,
        "k_cache": normal(shape, dtype, gv),
        "v_cache": normal(shape, dtype, gv),
        "q": normal((B, n_heads, head_dim), dtype, gv),
        "k_new": normal((B, n_heads, head_dim), dtype, gv),
        "v_new": normal((B, n_heads, head_dim), dtype, gv),
        "dtype": dtype,
        "block_size": block_size,
    }


def mla_case(batch, n_heads, d_c, d_r, block_size, lens, dtype, seed, spare_frac=0.10, device="cpu"):
    """An MLA absorbed decode step over a paged latent cache [num_blocks, bs, d_c + d_r]."""
    g = _gen(seed)
    gv = g if device == "cpu" else _gen(seed, device)
    if isinstance(lens, tuple):
        lens_t = uniform_lengths(batch, lens[0], lens[1], g)
    else:
        lens_t = torch.tensor([int(x) for x in lens], dtype=torch.int32)
    table, num_blocks = random_block_tables(lens_t.tolist(), block_size, spare_frac, g, True)
    W = d_c + d_r
    return {
        "context_lens": lens_t,
        "block_tables": table,
        "num_blocks": num_blocks,
        "latent_cache": normal((num_blocks, block_size, W), dtype, gv),
        "q": normal((batch, n_heads, W), dtype, gv),
        "c_new": normal((batch, W), dtype, gv),
        "dtype": dtype,
        "block_size": block_size,
    }


def tiny_sequence(n_tokens, n_layers, n_heads, head_dim, dtype, seed):
    """Per-layer q/k/v for every position of one sequence: lists of [n_tokens, H, D]."""
    g = _gen(seed)
    layers = []
    for _ in range(n_layers):
        layers.append({
            "q": normal((n_tokens, n_heads, head_dim), dtype, g),
            "k": normal((n_tokens, n_heads, head_dim), dtype, g),
            "v": normal((n_tokens, n_heads, head_dim), dtype, g),
        })
    return layers


def fp8_case(batch, n_q_heads, n_kv_heads, head_dim, block_size, lens, seed, spare_frac=0.10, device="cpu"):
    """A paged decode step over an FP8 (e4m3) cache: random codes (never the two NaN codes), per-channel K
    scales [Hkv, D] and a per-token V-scale pool [num_blocks, Hkv, bs] (positive, around 4/448 as for N(0,1)
    data), bf16 queries and bf16 new K/V rows. Draw order: lengths, table permutation, K codes, V codes,
    K scales, V scales, q, new k, new v."""
    g = _gen(seed)
    gv = g if device == "cpu" else _gen(seed, device)
    if isinstance(lens, tuple):
        lens_t = uniform_lengths(batch, lens[0], lens[1], g)
    else:
        lens_t = torch.tensor([int(x) for x in lens], dtype=torch.int32)
    table, num_blocks = random_block_tables(lens_t.tolist(), block_size, spare_frac, g, True)
    shape = (num_blocks, n_kv_heads, block_size, head_dim)

    def codes():
        # uniform over the 254 finite codes: draw 0..253 and skip 0x7F
        c = torch.randint(0, 254, shape, generator=gv, dtype=torch.int32, device=gv.device)
        return (c + (c >= 0x7F).to(torch.int32)).to(torch.uint8)

    kc, vc = codes(), codes()
    k_scale = ((0.5 + torch.rand((n_kv_heads, head_dim), generator=gv, device=gv.device)) * (4.0 / 448.0)).float()
    v_scale = ((0.5 + torch.rand(shape[:3], generator=gv, device=gv.device)) * (4.0 / 448.0)).float()
    return {
        "context_lens": lens_t,
        "block_tables": table,
        "num_blocks": num_blocks,
        "k_cache": kc,
        "v_cache": vc,
        "k_scale": k_scale,
        "v_scale": v_scale,
        "q": normal((batch, n_q_heads, head_dim), "bf16", gv),
        "k_new": normal((batch, n_kv_heads, head_dim), "bf16", gv),
        "v_new": normal((batch, n_kv_heads, head_dim), "bf16", gv),
        "block_size": block_size,
    }


def int8_case(batch, n_q_heads, n_kv_heads, head_dim, block_size, lens, seed, spare_frac=0.10, device="cpu"):
    """A paged decode step over an INT8 cache: codes uniform in [-127, 127], per-channel K scales [Hkv, D] and a
    per-token V-scale pool [num_blocks, Hkv, bs] (positive, around 4/127 as for N(0,1) data), bf16 queries and
    bf16 new K/V rows. Draw order: lengths, table permutation, K codes, V codes, K scales, V scales, q, new k,
    new v."""
    g = _gen(seed)
    gv = g if device == "cpu" else _gen(seed, device)
    if isinstance(lens, tuple):
        lens_t = uniform_lengths(batch, lens[0], lens[1], g)
    else:
        lens_t = torch.tensor([int(x) for x in lens], dtype=torch.int32)
    table, num_blocks = random_block_tables(lens_t.tolist(), block_size, spare_frac, g, True)
    shape = (num_blocks, n_kv_heads, block_size, head_dim)

    def codes():
        return torch.randint(-127, 128, shape, generator=gv, dtype=torch.int32, device=gv.device).to(torch.int8)

    kc, vc = codes(), codes()
    k_scale = ((0.5 + torch.rand((n_kv_heads, head_dim), generator=gv, device=gv.device)) * (4.0 / 127.0)).float()
    v_scale = ((0.5 + torch.rand(shape[:3], generator=gv, device=gv.device)) * (4.0 / 127.0)).float()
    return {
        "context_lens": lens_t,
        "block_tables": table,
        "num_blocks": num_blocks,
        "k_cache": kc,
        "v_cache": vc,
        "k_scale": k_scale,
        "v_scale": v_scale,
        "q": normal((batch, n_q_heads, head_dim), "bf16", gv),
        "k_new": normal((batch, n_kv_heads, head_dim), "bf16", gv),
        "v_new": normal((batch, n_kv_heads, head_dim), "bf16", gv),
        "block_size": block_size,
    }


def multi_case(batch, n_tok, n_q_heads, n_kv_heads, head_dim, block_size, lens, dtype, seed, spare_frac=0.10,
               device="cpu"):
    """A paged step with ``n_tok`` new query tokens per sequence (chunked prefill or speculative verification).

    ``lens`` count every row including the n_tok new ones (each at least n_tok). The cache part is
    ``gqa_case`` with the same seed; then, from a second generator seeded ``seed + 1``, in this order:
    q [B, n_tok, Hq, D], new k and new v [B, n_tok, Hkv, D] (the rows of positions n - n_tok .. n - 1).
    """
    c = gqa_case(batch, n_q_heads, n_kv_heads, head_dim, block_size, lens, dtype, seed, spare_frac, True, device)
    g2 = _gen(seed + 1, device if device != "cpu" else "cpu")
    c["q"] = normal((batch, n_tok, n_q_heads, head_dim), dtype, g2)
    c["k_new"] = normal((batch, n_tok, n_kv_heads, head_dim), dtype, g2)
    c["v_new"] = normal((batch, n_tok, n_kv_heads, head_dim), dtype, g2)
    c["n_tok"] = n_tok
    return c
