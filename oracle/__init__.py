"""Float64 CPU oracle for the attention forward -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The library never does.
"""

from .attention import (  # noqa: F401
    attention_dense,
    attention_masked,
    attention_paged,
    attention_paged_prefill,
    attention_single,
    attention_block_sparse,
    attention_varlen,
    check_cu_seqlens,
    kv_cache_write,
    paged_gather,
    softmax_weights,
    visible_mask,
    vsa_block_map,
    vsa_pool,
    vsa_blocks,
)
