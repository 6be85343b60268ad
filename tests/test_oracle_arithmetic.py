"""Pins of the oracle's memory arithmetic and of the harness's block layout against the worked
numbers the pages print (tests/golden/page_arithmetic.txt carries each number's citation)."""

import numpy as np
import pytest

from conftest import load_golden
from oracle import (blocks_for_tokens, cache_append, kv_bytes_per_token, prefix_sharing_blocks,
                    static_batch_utilization)
from synthetic import make_config, make_workload

G = load_golden("page_arithmetic.txt")


def gi(k):
    return int(G[k])


def test_kv_bytes_per_token_7b():
    # hidden 4096 = 32 heads x 128 per head for a multi-head model
    per = kv_bytes_per_token(gi("kv_bytes_7b_layers"), 32, gi("kv_bytes_7b_hidden") // 32,
                             gi("kv_bytes_7b_bytes_per_value"))
    assert per == gi("kv_bytes_7b_per_token")
    total = per * gi("kv_tokens_for_2gb")
    assert total == 2 * 1024 ** 3          # "roughly 2 gigabytes"
    # eight-bit values halve it (P1, "The memory that concurrency actually costs")
    assert kv_bytes_per_token(32, 32, 128, 1) * 2 == per


def test_fragmentation_example():
    blocks, slots, waste = blocks_for_tokens(gi("frag_tokens"), gi("frag_block_size"))
    assert (blocks, slots, waste) == (gi("frag_blocks"), gi("frag_slots"), gi("frag_waste"))
    assert gi("frag_reserved_slots") - gi("frag_tokens") == gi("frag_reserved_waste")
    worst = max(blocks_for_tokens(n, 16)[2] for n in range(1, 2000))
    assert worst == gi("frag_max_waste_per_seq")
    # "nearly 900 megabytes" saved at half a megabyte per token
    saved_mb = (gi("frag_reserved_slots") - slots) * 0.5
    assert 850 < saved_mb < 900


def test_prefix_sharing_example():
    assert gi("prefix_tokens") // gi("frag_block_size") == gi("prefix_blocks")
    un, sh, saved = prefix_sharing_blocks(gi("prefix_blocks"), gi("prefix_requests"))
    assert (un, sh, saved) == (gi("prefix_unshared_blocks"), gi("prefix_shared_blocks"),
                               gi("prefix_saved_blocks"))
    assert saved * 16 == gi("prefix_saved_tokens")
    assert saved * 16 * 0.5 == gi("prefix_saved_mb")


def test_static_batch_example():
    lengths = [int(x) for x in G["static_lengths"].split(",")]
    assert sum(lengths) == gi("static_useful")
    assert max(lengths) * len(lengths) == gi("static_paid")
    assert round(100 * static_batch_utilization(lengths)) == gi("static_utilization_pct")


def test_qwen3_capacity_example():
    # Assumed architecture (the page states only the per-token total): 36 layers, 8 kv heads,
    # head_dim 128, FP16.
    per = kv_bytes_per_token(36, 8, 128, 2)
    assert per == gi("qwen3_kib_per_token") * 1024
    assert round(gi("qwen3_tokens") * per / 1e9, 1) == float(G["qwen3_kv_gb"])
    approx = 10 * 1024 ** 3 / per
    assert abs(approx - gi("qwen3_tokens_per_10gb")) / gi("qwen3_tokens_per_10gb") < 0.02


def test_append_fills_blocks_like_the_300_token_example():
    """300 tokens appended one slot at a time land in 19 blocks: 18 full, the last with 12
    written slots and 4 empty (P2, "Worked Example: Fragmentation Saved"); block = pos // 16,
    offset = pos % 16 through the table ("Growing During Decode")."""
    w = make_workload([300], [300], num_q_heads=1, num_kv_heads=1, head_dim=8, pool_factor=2.0,
                      pool_fill="nan", seed=7)
    kp, vp = cache_append(w.empty_pool(), w.empty_pool(), w.k_new_bits, w.v_new_bits,
                          w.slot_mapping, w.block_size)
    written = (kp != 0x7FC0).all(axis=-1)[:, 0, :]          # [NB][bs]
    table = w.block_tables[0, :19]
    per_block = written[table].sum(axis=1)
    assert per_block.tolist() == [16] * 18 + [12]
    assert written.sum() == 300
    assert not written[np.setdiff1d(np.arange(w.num_blocks), table)].any()
    # the last block's written slots are its first 12 offsets
    assert written[table[-1]].tolist() == [True] * 12 + [False] * 4
    # position p of the sequence is in table[p // 16] at offset p % 16
    for p in (0, 15, 16, 17, 250, 299):
        assert np.array_equal(kp[table[p // 16], 0, p % 16], w.k_new_bits[p, 0])


@pytest.mark.parametrize("cid", [1, 4])
def test_named_workload_shapes(cid):
    w = make_config(cid)
    if cid == 1:
        assert w.context_lens.tolist() == [10, 40, 20, 80]
        assert w.num_blocks == 32 and w.unique_blocks() == 11
        assert w.attended_tokens() == 150
    else:
        assert w.num_tokens == 1072
        assert w.query_lens.tolist()[-2:] == [512, 512]
        assert w.context_lens.tolist()[-2:] == [512, 2560]


def test_shared_prefix_accounting_small():
    """Every table points its first m logical blocks at the same m physical blocks; the pool
    holds one copy (P2, "Shared Prefixes")."""
    w = make_workload([100, 70, 64], [1, 1, 1], num_q_heads=2, num_kv_heads=1, head_dim=8,
                      shared_prefix_blocks=3, seed=3)
    assert (w.block_tables[:, :3] == w.block_tables[0, :3]).all()
    un, sh, saved = prefix_sharing_blocks(3, 3)
    logical = sum(-(-int(L) // 16) for L in w.context_lens)
    assert w.unique_blocks() == logical - saved
