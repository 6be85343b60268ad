"""The benchmark's accounting, pinned by hand counts and brute force on tiny steps.

Every throughput that bench.py reports divides one of these counts by a time: the attention's
algorithmic bytes (each K/V block it touches once, q read, out written, metadata), the append's
bytes, the attended (query, key) pairs, and the flops of the tensor-core prefill tiles.
"""

import bench
from synthetic import make_workload


def test_algorithmic_bytes_by_hand():
    # two sequences of 20 and 16 keys with one new token each; 2 kv heads of 64 dims, bf16
    w = make_workload([20, 16], [1, 1], num_q_heads=2, num_kv_heads=2, head_dim=64, seed=1)
    kv = 2 * 3 * 2 * 16 * 64 * 2        # K and V: 3 blocks (2 + 1) x 2 heads x 16 x 64 bf16
    q = 2 * 2 * 64 * 2                  # 2 tokens x 2 heads x 64, bf16
    meta = 4 * (2 * 2 + 1) + 4 * 3      # context_lens, query_start_loc, 3 table entries
    assert w.algorithmic_bytes() == kv + q + 2 * 2 * 64 * 4 + meta          # fp32 out
    assert w.algorithmic_bytes(out_bytes_per_elem=2) == kv + q + 2 * 2 * 64 * 2 + meta
    # only the second sequence: its one block, its token, its metadata
    assert w.algorithmic_bytes(seqs=[1]) == \
        2 * 1 * 2 * 16 * 64 * 2 + 1 * 2 * 64 * (2 + 4) + 4 * (2 + 1) + 4 * 1


def test_shared_prefix_blocks_count_once():
    # three sequences of 64 keys (4 blocks) whose first 2 blocks are one shared prefix
    args = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, seed=2)
    w = make_workload([64, 64, 64], [1, 1, 1], shared_prefix_blocks=2, **args)
    assert w.unique_blocks() == 2 + 3 * 2
    d = make_workload([64, 64, 64], [1, 1, 1], **args)
    assert d.unique_blocks() == 3 * 4
    e4m3 = make_workload([64, 64, 64], [1, 1, 1], shared_prefix_blocks=2,
                         cache_dtype="fp8_e4m3", **args)
    kv_bf16 = 2 * 8 * 2 * 16 * 64 * 2
    assert w.algorithmic_bytes() - e4m3.algorithmic_bytes() == kv_bf16 // 2


def test_append_bytes_by_hand():
    args = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, seed=3)
    w = make_workload([20, 16], [3, 2], **args)
    per = 2 * 64                                  # kv heads x head dims of one token
    assert w.append_bytes() == 5 * per * 2 * 2 + 5 * per * 2 * 2 + 5 * 8
    f = make_workload([20, 16], [3, 2], cache_dtype="fp8_e4m3", **args)
    assert f.append_bytes() == 5 * per * 2 * 2 + 5 * per * 1 * 2 + 5 * 8


def test_attended_pairs_and_prefill_flops_by_brute_force():
    ctx, ql = [40, 300, 17, 9, 70], [1, 40, 17, 5, 4]
    hq, hkv, d = 8, 2, 128                        # groups of 4
    w = make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=4)
    pairs = {s: sum(L - n + i + 1 for i in range(n)) for s, (L, n) in enumerate(zip(ctx, ql))}
    assert w.attended_tokens() == sum(pairs.values())
    # the tensor-core tiles serve runs of more than 16 tokens or more than 16 token x head
    # rows: here the 40-, 17- and 5-token runs (5 x 4 = 20 rows), not 1 x 4 or 4 x 4
    tiled = [s for s, n in enumerate(ql) if n > 16 or n * (hq // hkv) > 16]
    assert tiled == [1, 2, 3]
    # QK^T and PV: 2 x 2 flops per (query, key) pair, head dim and q head
    assert bench.prefill_flops(w) == 4 * d * hq * sum(pairs[s] for s in tiled)


def test_reference_arm_sample_is_bounded():
    # as many sequences per process as fit 0.8 of the step's budget at the contended time ...
    assert bench.reference_sample_size(num_seqs=64, cores=16, budget_s=6.0, seq_s=0.7) == 6
    # ... but never more than twice the workload's sequences over all processes, however fast
    # one sequence is (an uncapped sample only repeats sequences and grows every process)
    assert bench.reference_sample_size(num_seqs=64, cores=16, budget_s=50.0, seq_s=0.01) == 8
    assert bench.reference_sample_size(num_seqs=64, cores=8, budget_s=50.0, seq_s=0.01) == 16
    # and always at least one
    assert bench.reference_sample_size(num_seqs=4, cores=16, budget_s=0.1, seq_s=5.0) == 1
    assert bench.reference_sample_size(num_seqs=64, cores=16, budget_s=1.0, seq_s=0.0) == 8
