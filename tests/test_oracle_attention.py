"""Pins of the fp64 attention oracle against what the pages and the mathematics fix:

* the contiguous special case equals torch's float64 scaled_dot_product_attention (a library
  routine sharing no code with the oracle), for decode, GQA and a causal chunk;
* paging invariance: a random permutation of the physical blocks (tables rewritten) gives the
  identical result ("Serving LLMs with vLLM ...", "Attention Over Scattered Blocks");
* prefix sharing: shared prefix blocks give the same result as private copies ("Shared Prefixes")
  and as a copy made before a write ("Copy-on-Write");
* special cases: one key returns its value exactly; equal keys return the mean of the values;
  two keys with score gap ln 3 weigh 1/4 and 3/4;
* chunked-prefill invariance: one chunk equals two chunks with a cached prefix ("Chunked
  Prefill"); causality: keys after a token's position do not change its output;
* split invariance: the log-sum-exp merge of any key partition equals the unsplit softmax.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import (attention_partial, bf16_bits_to_f64, cache_append, e4m3_decode,
                    gather_context, lse_merge, paged_attention, run_step)
from synthetic import make_workload


def _pools(w):
    return run_step(w)[:2]


def _attn(w, kp, vp, tables=None):
    return paged_attention(w.q_bits, kp, vp, w.block_tables if tables is None else tables,
                           w.context_lens, w.query_start_loc, w.num_q_heads, w.num_kv_heads,
                           w.head_dim, w.scale, w.block_size, w.cache_dtype, w.k_scale,
                           w.v_scale)


def _sdpa_seq(w, kp, vp, s, causal=False):
    """torch fp64 SDPA on the sequence's contiguous K/V (rebuilt by slicing the raw token
    arrays, not through the oracle's gather)."""
    L = int(w.context_lens[s])
    t0, t1 = int(w.query_start_loc[s]), int(w.query_start_loc[s + 1])
    # contiguous keys of sequence s straight from the drawn tokens (pool not involved)
    prior_idx = [i for i, sl in enumerate(w.slot_prior.tolist())
                 if sl // w.block_size in set(w.block_tables[s].tolist())]
    k = np.concatenate([w.k_prior_bits[prior_idx], w.k_new_bits[t0:t1]])
    v = np.concatenate([w.v_prior_bits[prior_idx], w.v_new_bits[t0:t1]])
    assert k.shape[0] == L
    q = torch.from_numpy(bf16_bits_to_f64(w.q_bits[t0:t1])).permute(1, 0, 2)[None]
    kt = torch.from_numpy(bf16_bits_to_f64(k)).permute(1, 0, 2)[None]
    vt = torch.from_numpy(bf16_bits_to_f64(v)).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(q, kt, vt, scale=w.scale, is_causal=causal,
                                       enable_gqa=w.num_q_heads != w.num_kv_heads)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (8, 2, 32), (6, 3, 16)])
def test_decode_matches_torch_sdpa(hq, hkv, d):
    w = make_workload([10, 40, 33, 80], [1, 1, 1, 1], num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=d, seed=11)
    kp, vp = _pools(w)
    out = _attn(w, kp, vp)
    for s in range(w.num_seqs):
        t0, t1 = w.query_start_loc[s], w.query_start_loc[s + 1]
        np.testing.assert_allclose(out[t0:t1], _sdpa_seq(w, kp, vp, s), rtol=0, atol=1e-12)


def test_causal_chunk_without_prefix_matches_torch_sdpa():
    w = make_workload([37, 5], [37, 5], num_q_heads=4, num_kv_heads=2, head_dim=16, seed=12)
    kp, vp = _pools(w)
    out = _attn(w, kp, vp)
    for s in range(2):
        t0, t1 = w.query_start_loc[s], w.query_start_loc[s + 1]
        np.testing.assert_allclose(out[t0:t1], _sdpa_seq(w, kp, vp, s, causal=True), rtol=0,
                                   atol=1e-12)


def test_fp8_cache_matches_torch_sdpa_on_dequantised_values():
    w = make_workload([21, 50], [1, 1], num_q_heads=4, num_kv_heads=2, head_dim=32,
                      cache_dtype="fp8_e4m3", seed=13)
    kp, vp = _pools(w)
    out = _attn(w, kp, vp)
    for s in range(2):
        L = int(w.context_lens[s])
        nb = -(-L // 16)
        blocks = w.block_tables[s, :nb]
        # dequantise with torch's float8 decode, independently of the oracle's gather
        def seq(pool, scale):
            codes = torch.from_numpy(np.ascontiguousarray(pool[blocks]))   # [nb][H][bs][D]
            x = codes.view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(scale))
            return x.permute(1, 0, 2, 3).reshape(w.num_kv_heads, nb * 16, -1)[:, :L][None]
        t0 = w.query_start_loc[s]
        q = torch.from_numpy(bf16_bits_to_f64(w.q_bits[t0:t0 + 1])).permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(q, seq(kp, w.k_scale), seq(vp, w.v_scale),
                                           scale=w.scale, enable_gqa=True)
        np.testing.assert_allclose(out[t0:t0 + 1], o[0].permute(1, 0, 2).numpy(), rtol=0,
                                   atol=1e-12)


def test_paging_invariance_is_exact():
    w = make_workload([5, 16, 17, 64, 99], [1, 1, 3, 1, 7], num_q_heads=4, num_kv_heads=2,
                      head_dim=16, seed=14)
    kp, vp = _pools(w)
    ref = _attn(w, kp, vp)
    perm = np.random.default_rng(5).permutation(w.num_blocks)     # new position of block b
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    assert np.array_equal(_attn(w, kp2, vp2, tables), ref)


def test_prefix_sharing_equals_private_copies_and_copy_on_write():
    w = make_workload([70, 90, 65], [1, 2, 1], num_q_heads=4, num_kv_heads=1, head_dim=16,
                      shared_prefix_blocks=4, seed=15, pool_factor=3.0)
    kp, vp = _pools(w)
    ref = _attn(w, kp, vp)
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    free = [b for b in range(w.num_blocks) if b not in used]
    tables = w.block_tables.copy()
    kp2, vp2 = kp.copy(), vp.copy()
    for s in range(1, w.num_seqs):       # give sequences 1.. private copies of the prefix
        for j in range(4):
            b = free.pop()
            kp2[b], vp2[b] = kp[tables[s, j]], vp[tables[s, j]]
            tables[s, j] = b
    assert np.array_equal(_attn(w, kp2, vp2, tables), ref)
    assert len(set(tables[:, :4].ravel().tolist())) == 12


def test_single_key_returns_value_exactly():
    w = make_workload([1, 1], [1, 1], num_q_heads=4, num_kv_heads=2, head_dim=8, seed=16)
    kp, vp = _pools(w)
    out = _attn(w, kp, vp)
    for t in range(2):
        for h in range(4):
            assert np.array_equal(out[t, h], bf16_bits_to_f64(w.v_new_bits[t, h // 2]))


def test_equal_keys_return_mean_of_values():
    w = make_workload([23], [1], num_q_heads=2, num_kv_heads=1, head_dim=8, seed=17)
    kp, vp = _pools(w)
    for b in w.block_tables[0, :2]:
        kp[b] = kp[w.block_tables[0, 0], :, 0:1, :]     # every key equal to key 0
    out = _attn(w, kp, vp)
    V = gather_context(vp, w.block_tables[0], 23, 16)
    np.testing.assert_allclose(out[0, 0], V[:, 0].mean(0), rtol=0, atol=1e-14)


def test_two_keys_with_score_gap_ln3_weigh_quarter_and_three_quarters():
    w = make_workload([2], [1], num_q_heads=1, num_kv_heads=1, head_dim=4, seed=18,
                      scale=1.0)
    kp, vp = _pools(w)
    # q = (1,0,0,0); k0 = (0,...), k1 = (ln 3 rounded to bf16, ...) -> weights 1/(1+r), r/(1+r)
    q = np.zeros_like(w.q_bits)
    q[0, 0, 0] = 0x3F80                                  # 1.0
    w.q_bits = q
    b = w.block_tables[0, 0]
    kp[b, 0, 0, :] = 0
    kp[b, 0, 1, :] = 0
    kp[b, 0, 1, 0] = 0x3F8D                              # bf16 1.1015625 ~ ln 3
    out = _attn(w, kp, vp)
    r = math.exp(1.1015625)
    V = bf16_bits_to_f64(vp[b, 0, :2])
    np.testing.assert_allclose(out[0, 0], (V[0] + r * V[1]) / (1 + r), rtol=0, atol=1e-14)


def test_chunked_prefill_equals_one_chunk():
    """A 96-token prompt processed whole equals 64 tokens then a 32-token chunk on top of the
    cached 64 (the same keys, positions and values)."""
    whole = make_workload([96], [96], num_q_heads=4, num_kv_heads=2, head_dim=16, seed=19)
    kp, vp = _pools(whole)
    out_whole = _attn(whole, kp, vp)
    # second chunk: the same pool, 32 queries at positions 64..95
    qsl = np.array([0, 32], dtype=np.int32)
    out_tail = paged_attention(whole.q_bits[64:], kp, vp, whole.block_tables, whole.context_lens,
                               qsl, 4, 2, 16, whole.scale, 16)
    np.testing.assert_array_equal(out_tail, out_whole[64:])
    # first chunk: a 64-key context with its 64 queries
    out_head = paged_attention(whole.q_bits[:64], kp, vp, whole.block_tables,
                               np.array([64], dtype=np.int32), np.array([0, 64], dtype=np.int32),
                               4, 2, 16, whole.scale, 16)
    np.testing.assert_array_equal(out_head, out_whole[:64])


def test_causality_later_keys_do_not_matter():
    w = make_workload([48], [20], num_q_heads=2, num_kv_heads=1, head_dim=8, seed=20)
    kp, vp = _pools(w)
    ref = _attn(w, kp, vp)
    # change key/value at position 40 (query token i = 40 - 28 = 12 is the first to see it)
    b, o = w.block_tables[0, 40 // 16], 40 % 16
    kp[b, 0, o, :] ^= 0x0100
    vp[b, 0, o, :] ^= 0x0100
    out = _attn(w, kp, vp)
    assert np.array_equal(out[:12], ref[:12])
    assert not np.allclose(out[12:], ref[12:])


@pytest.mark.parametrize("cuts", [[0, 100], [0, 1, 100], [0, 16, 33, 64, 100], [0, 99, 100]])
def test_lse_merge_of_any_partition_equals_unsplit(cuts):
    rng = np.random.default_rng(21)
    K, V, q = rng.standard_normal((100, 32)), rng.standard_normal((100, 32)), \
        rng.standard_normal(32) * 3
    full, _ = attention_partial(q, K, V, slice(0, 100), 0.3)
    parts = [attention_partial(q, K, V, slice(a, b), 0.3) for a, b in zip(cuts, cuts[1:])]
    merged = lse_merge(np.array([p[0] for p in parts]), np.array([p[1] for p in parts]))
    np.testing.assert_allclose(merged, full, rtol=0, atol=1e-13)
    # and the unsplit lse is the log of the full normaliser
    a = 0.3 * K @ q
    assert abs(attention_partial(q, K, V, slice(0, 100), 0.3)[1]
               - math.log(np.exp(a).sum())) < 1e-12


def test_fp8_append_codes_match_torch_conversion():
    w = make_workload([40, 3], [40, 3], num_q_heads=2, num_kv_heads=2, head_dim=16,
                      cache_dtype="fp8_e4m3", seed=22)
    kp, vp = cache_append(w.empty_pool(), w.empty_pool(), w.k_new_bits, w.v_new_bits,
                          w.slot_mapping, 16, "fp8_e4m3", w.k_scale, w.v_scale)
    x = torch.from_numpy(w.k_new_bits.view(np.int16)).view(torch.bfloat16).float()
    ref = (x / torch.tensor(w.k_scale, dtype=torch.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()
    slots = w.slot_mapping
    got = kp[slots // 16, :, slots % 16, :]
    assert np.array_equal(got, ref)
    assert np.abs(e4m3_decode(got)).max() <= 448


def test_parallel_oracle_gives_the_serial_result_bitwise():
    """paged_attention_parallel runs paged_attention itself on shares of the sequences in
    spawned processes: its output must be the serial output, bit for bit, with the left-out
    sequences' rows NaN in both."""
    from oracle import paged_attention, paged_attention_parallel
    from synthetic import make_workload
    w = make_workload([40, 1, 300, 77, 16, 129], [1, 1, 9, 1, 16, 3], num_q_heads=8,
                      num_kv_heads=2, head_dim=16, seed=11)
    kp, vp = cache_append(w.empty_pool(), w.empty_pool(), w.k_prior_bits, w.v_prior_bits,
                          w.slot_prior, w.block_size)
    kp, vp = cache_append(kp, vp, w.k_new_bits, w.v_new_bits, w.slot_mapping, w.block_size)
    args = (w.q_bits, kp, vp, w.block_tables, w.context_lens, w.query_start_loc, w.num_q_heads,
            w.num_kv_heads, w.head_dim, w.scale, w.block_size)
    for seqs in (None, [0, 2, 5]):
        a = paged_attention(*args, seqs=seqs)
        b = paged_attention_parallel(*args, seqs=seqs, processes=3)
        assert np.array_equal(np.isnan(a), np.isnan(b))
        assert np.array_equal(np.nan_to_num(a), np.nan_to_num(b))


def test_parallel_e4m3_append_gives_the_serial_pools_bitwise():
    from oracle import cache_append_parallel
    from synthetic import make_workload
    w = make_workload([300, 41, 700], [1, 1, 1], num_q_heads=4, num_kv_heads=2, head_dim=16,
                      cache_dtype="fp8_e4m3", seed=12, pool_fill="nan")
    args = (w.empty_pool(), w.empty_pool(), w.k_prior_bits, w.v_prior_bits, w.slot_prior,
            w.block_size, w.cache_dtype, w.k_scale, w.v_scale)
    a = cache_append(*args)
    b = cache_append_parallel(*args, processes=3, rows_per_task=100)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
