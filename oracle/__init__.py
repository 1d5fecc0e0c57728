"""CPU oracle for paged KV-cache decode attention: TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct statement of what the GPU
path computes. It is written in NumPy float64 (and, for the smallest cases,
pure-Python loops) directly from the definitions on the source pages:

* "KV缓存原理与显存估算" (LLM Systems Wiki, kv-cache), knowledge point 2:
  single-step attention that appends the current K/V and then applies a
  max-subtracted softmax over every cached position; knowledge point 1:
  the useful / padded / paged byte accounting; the closing "boundary"
  section: unique-physical-block accounting under block sharing.
* "KV-Cache——为什么AI回复越来越快" (dataqian.wang), section 02: the cache
  recurrence K_cache(t) = Concat(K_cache(t-1), K_{p+t}) and
  output = Attention(Q_{p+t}, K_cache, V_cache); section 05: cached and
  recomputed generation agree; section 07: the cache-size formula.
* "单请求 KV Cache" (mini-vllm tutorial step 07): the prefill/decode causal
  mask rule (row i sees columns <= past_len + i) and the in-place
  preallocated write at the current position.
* "KV Cache（键值缓存）" (llm-compass), section 2.2: MLA latent
  c_t = W^DKV h_t, up-projections W^UK / W^UV that can be absorbed into the
  query / output projections, decoupled RoPE part of width d_R, 576 cached
  elements per token for DeepSeek-V2; section 2.3: PagedAttention block
  tables mapping logical blocks to physical blocks.

Who may use it: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``. The product
library under ``paged_kv_cache_157_gb300`` never imports, links or calls
anything here, and nothing here imports the product. The two share no
kernels, headers, helpers, tables or constants.
"""

from .attention import (  # noqa: F401
    stable_softmax,
    cached_attention,
    causal_attention_full,
    decode_by_recompute,
    attention_loops,
)
from .paged import (  # noqa: F401
    slot_of,
    slots_for_positions,
    append_to_paged,
    gather_logical,
    paged_decode,
    paged_decode_lse,
)
from .mla import (  # noqa: F401
    mla_absorbed_decode,
    mla_explicit_decode,
    absorb_query,
)
from .layout import (  # noqa: F401
    kv_cache_bytes,
    kv_layout,
    unique_block_bytes,
)
from .pool_model import PoolModel  # noqa: F401
