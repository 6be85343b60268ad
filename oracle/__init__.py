"""fp64 CPU oracle for one continuous-batching attention step over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute anything in
this package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs use it.  It shares no code with the CUDA library (no headers, no helpers, no
constants); the only module both sides use is ``synthetic``, which draws the seeded inputs.

What it computes is the plain definition the pages give: paged attention is ordinary attention,
softmax of the query times the keys over the whole history, applied to values that are fetched
block by block through a per-sequence block table ("Serving LLMs with vLLM: Continuous Batching
and PagedAttention Explained", sections "Blocks and Block Tables", "Attention Over Scattered
Blocks", "Growing During Decode").  Every function names the passage it follows.
"""

from .arithmetic import (  # noqa: F401
    blocks_for_tokens,
    kv_bytes_per_token,
    prefix_sharing_blocks,
    static_batch_utilization,
)
from .e4m3 import decode as e4m3_decode, encode_f32 as e4m3_encode_f32  # noqa: F401
from .paged_kv import (  # noqa: F401
    attention_partial,
    bf16_bits_to_f64,
    cache_append,
    gather_context,
    lse_merge,
    paged_attention,
    run_step,
)
from .parallel import cache_append_parallel, paged_attention_parallel  # noqa: F401,E402
