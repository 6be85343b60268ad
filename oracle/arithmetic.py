"""Memory arithmetic the pages state for a paged KV cache.

Test infrastructure only (see the package docstring).  These helpers fix the sizes the harness
and the benchmark use (bytes per token, block counts, savings from a shared prefix) and are
pinned by the worked numbers the pages print.
"""

from __future__ import annotations

from typing import Sequence


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_value: int) -> int:
    """Key plus value bytes one token costs across all layers.

    "Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained", section "The KV
    Cache Is Big": a key and a value per token in every layer, i.e. 2 x layers x hidden x bytes,
    where for multi-head attention hidden = kv_heads x head_dim.
    """
    return 2 * layers * kv_heads * head_dim * bytes_per_value


def blocks_for_tokens(num_tokens: int, block_size: int):
    """(blocks, slots, wasted slots) for one sequence of ``num_tokens`` tokens.

    Same page, sections "Blocks and Block Tables" and "Worked Example: Fragmentation Saved": a
    sequence takes a new block only when its current one is full, so it holds the token count
    divided by the block size, rounded up; only the last block can be partly empty.
    """
    blocks = -(-num_tokens // block_size)
    slots = blocks * block_size
    return blocks, slots, slots - num_tokens


def prefix_sharing_blocks(prefix_blocks: int, requests: int):
    """(blocks without sharing, blocks with sharing, blocks saved) for a common prefix.

    Same page, sections "Shared Prefixes" and "The Savings in Numbers": without sharing every
    request stores its own copy; with sharing one copy is stored and referenced by all.
    """
    unshared = prefix_blocks * requests
    shared = prefix_blocks
    return unshared, shared, unshared - shared


def static_batch_utilization(lengths: Sequence[int]) -> float:
    """Useful slot-steps over paid slot-steps when a static batch runs to its longest member.

    Same page, sections "Static Batching" and "Worked Example: Wasted Slots".
    """
    lengths = list(lengths)
    return sum(lengths) / (max(lengths) * len(lengths))
