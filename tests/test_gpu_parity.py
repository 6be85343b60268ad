"""Parity of the CUDA library (through its C ABI) with the fp64 oracle.

Append: bit-exact against the oracle's scatter, for bf16 and E4M3 pools, untouched slots
included.  Attention: max |gpu - oracle| <= 2e-3 for bf16 K/V and 2e-2 for E4M3 K/V (fp32
output), element by element, on cases that span several partitions and a ragged last block, on
the six named workloads (every row of each, the full-size ones in the same launch
configuration the benchmark times), and on edge cases.  GPU invariants:
permuting the physical blocks and sharing vs duplicating a prefix give bitwise-identical output.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import cache_append, e4m3_encode_f32, paged_attention, run_step  # noqa: E402
from synthetic import make_config, make_workload  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_286_gb300 import build
    build.build()


def _h():
    import gpu_harness
    return gpu_harness


def _oracle_pools(w):
    """The oracle's pools after the set-up and step appends (E4M3 encoding spread over the
    host cores: cache_append_parallel gives cache_append's result)."""
    from oracle import cache_append_parallel
    kp, vp = cache_append_parallel(w.empty_pool(), w.empty_pool(), w.k_prior_bits,
                                   w.v_prior_bits, w.slot_prior, w.block_size, w.cache_dtype,
                                   w.k_scale, w.v_scale)
    return cache_append(kp, vp, w.k_new_bits, w.v_new_bits, w.slot_mapping, w.block_size,
                        w.cache_dtype, w.k_scale, w.v_scale)


def _check_small(w, out_dtype=torch.float32):
    h = _h()
    d, out = h.run_gpu(w, out_dtype)
    kp, vp, ref = run_step(w)
    gk, gv = d.pools_numpy()
    assert np.array_equal(gk, kp) and np.array_equal(gv, vp), "append is not bit-exact"
    return h.assert_close_to_oracle(w, out, ref)


# ---- the tiny named workload, every row ----------------------------------------------------
def test_config1_all_rows():
    _check_small(make_config(1))


@pytest.mark.parametrize("fill", ["zero", "nan"])
def test_config1_stale_slots_do_not_leak(fill):
    """Unwritten slots of a sequence's last block hold NaN patterns; they must be masked."""
    _check_small(make_config(1, pool_fill=fill))


# ---- small cases spanning partitions and ragged tails ------------------------------------
EDGE_CTX = [1, 15, 16, 17, 32, 33, 100, 511, 512, 513, 2000]


@pytest.mark.parametrize("hq,hkv,d,dtype", [
    (4, 4, 128, "bf16"), (8, 4, 128, "bf16"), (16, 4, 128, "bf16"), (32, 4, 128, "bf16"),
    (4, 4, 64, "bf16"), (16, 2, 64, "bf16"),
    (8, 8, 128, "fp8_e4m3"), (16, 4, 128, "fp8_e4m3"), (32, 4, 128, "fp8_e4m3"),
    (64, 4, 128, "bf16"), (32, 2, 64, "bf16"), (64, 4, 128, "fp8_e4m3"),     # groups of 16
    (12, 3, 128, "fp8_e4m3"),   # group of 4 over an odd number of kv heads: one head per item
])
def test_decode_edge_lengths(hq, hkv, d, dtype):
    w = make_workload(EDGE_CTX, [1] * len(EDGE_CTX), num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=d, cache_dtype=dtype, seed=hq * 131 + d, pool_fill="nan",
                      extra_table_cols=3)
    _check_small(w)


@pytest.mark.parametrize("qlens,ctx", [
    ([2, 3, 7, 16], [40, 3, 200, 16]),            # short multi-query runs (speculative verify)
    ([37, 1, 64], [37, 900, 300]),                # chunk with no prior context; chunk on prefix
    ([0, 5, 0, 1], [10, 70, 33, 1]),              # sequences with nothing to do
])
@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_multi_query_causal(qlens, ctx, dtype):
    w = make_workload(ctx, qlens, num_q_heads=16, num_kv_heads=4, head_dim=128,
                      cache_dtype=dtype, seed=sum(ctx), pool_fill="nan")
    _check_small(w)


@pytest.mark.parametrize("hq,hkv,qlens,ctx", [
    (8, 8, [9, 16, 3, 1], [9, 700, 40, 2000]),        # MHA: up to 16 tokens in one 16-row tile
    (8, 2, [5, 5, 1, 3], [517, 64, 1500, 3]),         # 4 x 4 rows, tail tile of one token
    (64, 4, [1, 2, 5, 16], [33, 1000, 5, 300]),       # group of 16: one token per tile
    (32, 2, [100, 1, 40], [2000, 77, 40]),            # group of 16 with long chunks
    (24, 8, [7, 2, 11], [7, 260, 900]),               # group of 3: 5 tokens (15 rows) a tile
    (16, 2, [3, 2, 1], [70, 900, 33]),                # group of 8: 24 rows to the tensor-core
                                                      # tiles, 16 and 8 rows to the split-KV path
    (8, 4, [9, 8, 1], [9, 500, 1200]),                # group of 2: 18 rows vs 16
    (16, 4, [16, 9, 1], [16, 700, 300]),              # 64 and 36 rows: two lane quarters,
                                                      # rows split over two warps
    (16, 4, [20, 3], [900, 50]),                      # 80 rows: whole-row softmax warps
])
@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_multi_query_row_tiles(hq, hkv, qlens, ctx, dtype):
    """Multi-query runs whose (token x head) rows fill 16-row decode tiles, groups of up to 16
    q heads per kv head, and groups that do not divide the tile."""
    w = make_workload(ctx, qlens, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                      cache_dtype=dtype, seed=hq + sum(ctx), pool_fill="nan")
    _check_small(w)


PF_CTX = [700, 17, 300, 1000, 129, 2100]
PF_QL = [200, 17, 300, 33, 129, 64]


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8)])
def test_prefill_chunks_on_tensor_core_tiles(hq, hkv):
    """Chunks with more than 16 queries take the tcgen05 tile path (bf16, head_dim 128):
    several 128-row tiles and 128-key slices, chunks with and without a cached prefix, ragged
    last blocks holding NaN patterns, GQA groups 1, 2, 4, 8, mixed with decode sequences."""
    w = make_workload(PF_CTX + [90, 3000], PF_QL + [1, 1], num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=128, seed=hq * 7 + 1, pool_fill="nan")
    _check_small(w)


@pytest.mark.parametrize("hq,hkv,out", [(32, 8, "f32"), (8, 8, "f32"), (64, 8, "f32"),
                                         (32, 8, "bf16")])
def test_prefill_tiles_split_along_the_keys(hq, hkv, out):
    """Tiles whose keys span many 128-key slices are cut along the keys into up to four items;
    each writes a normalised partial and its log-sum-exp, and the last to finish merges them.
    Runs here: a 200-token chunk after a 4,800-token prefix (four splits), a 96-token chunk
    after 1,200 (two), a short chunk with no prefix (none), beside decodes; sharp scores
    (scale 1) make the partials' maxima differ widely."""
    w = make_workload([5000, 1296, 700, 3000, 40], [200, 96, 130, 1, 1], num_q_heads=hq,
                      num_kv_heads=hkv, head_dim=128, seed=hq + 13, pool_fill="nan")
    _check_small(w, torch.bfloat16 if out == "bf16" else torch.float32)
    w = make_workload([5000, 1296], [200, 96], num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                      seed=hq + 14, pool_fill="nan", scale=1.0)
    _check_small(w)


def test_verify_tiles_split_along_the_keys():
    """Speculative-verify runs (rows split over two softmax warps) over long contexts are cut
    along the keys as well; every row of every split tile is merged and compared."""
    w = make_workload([4096, 3000, 1100, 512], [5, 5, 5, 5], num_q_heads=32, num_kv_heads=8,
                      head_dim=128, seed=57, pool_fill="nan")
    _check_small(w)


@pytest.mark.parametrize("qlens,ctx,dtype", [
    ([1, 1, 1, 1], [4000, 2000, 513, 100], "bf16"),        # split-KV decode
    ([1, 1, 1, 1], [4000, 2000, 513, 100], "fp8_e4m3"),
    ([3, 2], [3000, 700], "bf16"),                          # 16-row split-KV tiles
    ([100, 40], [2000, 600], "bf16"),                       # tensor-core tiles, whole rows
    ([5, 16], [1500, 900], "bf16"),                         # tensor-core tiles, split rows
])
def test_sharp_scores_rescale_the_running_max(qlens, ctx, dtype):
    """Unscaled q.k (scale 1: scores of sd ~11 nats) make the running max of a row grow by
    more than 2^8 as the keys stream in, so the accumulated output is rescaled on the way."""
    w = make_workload(ctx, qlens, num_q_heads=16, num_kv_heads=4, head_dim=128,
                      cache_dtype=dtype, seed=sum(ctx) + len(qlens), scale=1.0)
    _check_small(w)


def test_prefill_chunks_bf16_output():
    w = make_workload(PF_CTX, PF_QL, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=91)
    _check_small(w, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("hq,hkv,out", [(8, 8, "f32"), (16, 4, "f32"), (32, 4, "f32"),
                                         (16, 2, "f32"), (32, 4, "bf16")])
def test_prefill_chunks_head_dim_64(hq, hkv, out):
    """head_dim 64 chunks on the tensor-core tiles (one 64-column q half, 2 KiB block tiles by
    2-D copies, 64 O columns): chunks with and without a cached prefix, a tile long enough to
    be cut along the keys (7,000 keys: two splits, merged), a five-token verify run, and
    decodes beside them; stale slots hold NaN patterns."""
    w = make_workload([700, 17, 7000, 300, 90, 3000], [200, 17, 200, 5, 1, 1], num_q_heads=hq,
                      num_kv_heads=hkv, head_dim=64, seed=hq * 5 + hkv, pool_fill="nan")
    _check_small(w, torch.bfloat16 if out == "bf16" else torch.float32)


@pytest.mark.parametrize("hq,hkv,scale,out", [(32, 8, None, "f32"), (16, 16, None, "f32"),
                                               (32, 4, 1.0, "f32"), (32, 8, None, "bf16")])
def test_prefill_chunks_e4m3(hq, hkv, scale, out):
    """E4M3 pools' chunks on the tensor-core tiles (f8f6f4 MMAs: q in three E4M3 parts with a
    per-row scale, P in two parts scaled by 2^8, K and V as stored): chunks with and without a
    cached prefix, a tile cut along the keys (7,000 keys), a five-token verify run and decodes
    beside them; stale slots hold NaN patterns; scale 1 gives scores of sd ~11 nats."""
    w = make_workload([700, 17, 7000, 300, 90, 3000], [200, 17, 200, 5, 1, 1], num_q_heads=hq,
                      num_kv_heads=hkv, head_dim=128, cache_dtype="fp8_e4m3", seed=hq + hkv + 3,
                      pool_fill="nan", scale=scale)
    _check_small(w, torch.bfloat16 if out == "bf16" else torch.float32)


def test_large_v_values_keep_their_precision():
    """V values far outside the N(0,1) range (+-65536, beyond what fp16 can hold, and 65280)
    in tensor-core tiles: P V stays exact (bf16 hi + lo parts of P against bf16 V), so the
    output is finite and the dims holding them are within 2^-13 of their size, the rest
    within 2e-3."""
    w = make_workload([600, 300], [200, 100], num_q_heads=32, num_kv_heads=8, head_dim=128,
                      seed=77)
    # prior rows: sequence 0 positions 0..399, then sequence 1 positions 0..199
    planted = {(10, 0, 5): 0x4780,    # +65536: keys 0-63 of slice 0 of sequence 0, head 0
               (300, 3, 7): 0xC780,   # -65536: keys 0-63 of slice 2, head 3
               (405, 2, 9): 0x477F}   # 65280: sequence 1, head 2
    for (i, hk, d), bits in planted.items():
        w.v_prior_bits[i, hk, d] = bits
    dev, out = _h().run_gpu(w, torch.float32)
    _, _, ref = run_step(w)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), "non-finite output"
    G = w.num_q_heads // w.num_kv_heads
    mask = np.zeros(ref.shape, dtype=bool)
    err = np.abs(got - ref)
    for (_, hk, d), bits in planted.items():
        mask[:, hk * G:(hk + 1) * G, d] = True
        e, r = err[:, hk * G:(hk + 1) * G, d], np.abs(ref[:, hk * G:(hk + 1) * G, d])
        assert np.all(e <= 2e-3 + 2.0 ** -13 * r), (hex(bits), float((e - 2.0 ** -13 * r).max()))
    assert err[~mask].max() <= 2e-3, err[~mask].max()


def test_prefill_block_permutation_is_bitwise_invariant():
    h = _h()
    args = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, seed=92, pool_factor=1.5)
    w = make_workload([600, 300], [400, 300], **args)
    _, out1 = h.run_gpu(w)
    out1 = out1.clone()
    perm = np.random.default_rng(2).permutation(w.num_blocks)
    w2 = make_workload([600, 300], [400, 300], **args)
    w2.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1) \
        .astype(np.int32)
    w2.slot_mapping = perm[w.slot_mapping // 16] * 16 + w.slot_mapping % 16
    w2.slot_prior = perm[w.slot_prior // 16] * 16 + w.slot_prior % 16
    _, out2 = h.run_gpu(w2)
    assert torch.equal(out1, out2)


def test_single_sequence_long_context_splits():
    w = make_workload([9000], [1], num_q_heads=8, num_kv_heads=2, head_dim=128, seed=5)
    _check_small(w)


@pytest.mark.parametrize("qlen_long", [1, 3])
@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_many_sequences_with_splits_past_the_first_thousand(qlen_long, dtype):
    """1,100 sequences, most of them short; the long ones (split into partitions) sit at the
    first and last index, at the 32- and 1024-sequence boundaries and in between, so the
    merge finds each row's sequence in more than one round of its 32-way search."""
    rng = np.random.default_rng(4100 + qlen_long)
    n = 1100
    ctx = rng.integers(1, 48, size=n)
    qlen = np.ones(n, dtype=np.int64)
    for s in (0, 31, 32, 517, 1023, 1024, 1099):
        ctx[s] = 6000 + s
        qlen[s] = qlen_long
    w = make_workload(list(ctx), list(qlen), num_q_heads=8, num_kv_heads=2, head_dim=128,
                      cache_dtype=dtype, seed=41 + qlen_long, pool_fill="nan")
    _check_small(w)


def test_bf16_output():
    w = make_workload(EDGE_CTX, [1] * len(EDGE_CTX), num_q_heads=8, num_kv_heads=2,
                      head_dim=128, seed=77)
    _check_small(w, out_dtype=torch.bfloat16)


# ---- append -------------------------------------------------------------------------------
def test_append_skips_negative_slots():
    h = _h()
    w = make_workload([50, 20], [50, 20], num_q_heads=4, num_kv_heads=4, head_dim=64, seed=8)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[::3] = -1
    d = h.DeviceStep(w)
    d.append_new()
    assert __import__("paged_kv_cache_286_gb300").check_error(d.ws) == 0
    kp, vp = cache_append(w.empty_pool(), w.empty_pool(), w.k_new_bits, w.v_new_bits,
                          w.slot_mapping, 16)
    gk, gv = d.pools_numpy()
    assert np.array_equal(gk, kp) and np.array_equal(gv, vp)


@pytest.mark.parametrize("scale", [1.0, 0.012904576, 3.7, 2.0 ** -20])
def test_e4m3_append_every_bf16_value(scale):
    """Every one of the 65536 bf16 bit patterns quantised on append equals the oracle's OCP
    encoding of fl32(x) / scale (round to nearest even, saturating; NaN -> 0x7F)."""
    import paged_kv_cache_286_gb300 as pa
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 1, 128)
    slots = np.arange(512, dtype=np.int64)
    k = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    kc = torch.zeros((32, 1, 16, 128), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ws = pa.new_workspace(256)
    pa.cache_append(k, k, torch.from_numpy(slots).cuda(), kc, vc, ws, k_scale=scale,
                    v_scale=scale)
    assert pa.check_error(ws) == 0
    got = kc.cpu().numpy()[slots // 16, 0, slots % 16, :]
    x = (bits.astype(np.uint32) << 16).view(np.float32)[:, 0, :]
    want = e4m3_encode_f32(np.divide(x, np.float32(scale), dtype=np.float32))
    nan_in = np.isnan(x)
    assert np.array_equal(got[~nan_in], want[~nan_in])
    assert np.all((got[nan_in] & 0x7F) == 0x7F)        # NaN stays NaN


# ---- invariants on the GPU ---------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_block_permutation_is_bitwise_invariant(dtype):
    h = _h()
    w = make_workload([300, 1000, 17, 4000], [1, 1, 1, 1], num_q_heads=16, num_kv_heads=4,
                      head_dim=128, seed=9, pool_factor=1.5, cache_dtype=dtype)
    d1, out1 = h.run_gpu(w)
    out1 = out1.clone()
    perm = np.random.default_rng(1).permutation(w.num_blocks)
    w2 = make_workload([300, 1000, 17, 4000], [1, 1, 1, 1], num_q_heads=16, num_kv_heads=4,
                       head_dim=128, seed=9, pool_factor=1.5, cache_dtype=dtype)
    w2.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1) \
        .astype(np.int32)
    w2.slot_mapping = perm[w.slot_mapping // 16] * 16 + w.slot_mapping % 16
    w2.slot_prior = perm[w.slot_prior // 16] * 16 + w.slot_prior % 16
    d2, out2 = h.run_gpu(w2)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_shared_prefix_equals_duplicated_prefix_bitwise(dtype):
    h = _h()
    ctx = [2000, 1700, 1300]
    w = make_workload(ctx, [1, 1, 1], num_q_heads=8, num_kv_heads=2, head_dim=128, seed=10,
                      shared_prefix_blocks=20, pool_factor=2.0, cache_dtype=dtype)
    d, out_shared = h.run_gpu(w)
    out_shared = out_shared.clone()
    # duplicate the 20 shared blocks into private copies for sequences 1 and 2
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    free = [b for b in range(w.num_blocks) if b not in used]
    tables = w.block_tables.copy()
    for s in (1, 2):
        for j in range(20):
            b = free.pop()
            d.k_cache[b] = d.k_cache[tables[s, j]]
            d.v_cache[b] = d.v_cache[tables[s, j]]
            tables[s, j] = b
    assert len(set(tables[:, :20].ravel().tolist())) == 60
    d.tables = torch.from_numpy(tables).cuda()
    out_dup = d.attend()
    assert torch.equal(out_shared, out_dup)


# ---- device-side errors (bounds checks; nothing is read out of bounds) -------------------
def test_out_of_range_block_id_sets_error_word():
    import paged_kv_cache_286_gb300 as pa
    h = _h()
    w = make_workload([100, 50], [1, 1], num_q_heads=4, num_kv_heads=4, head_dim=64, seed=3)
    d = h.DeviceStep(w)
    d.append_prior()
    d.append_new()
    bad = w.block_tables.copy()
    bad[0, 2] = w.num_blocks + 5
    bad[1, 0] = -7
    d.tables = torch.from_numpy(bad).cuda()
    d.attend()
    word = pa.check_error(d.ws, raise_on_error=False)
    assert word & pa._lib.PA_DEVERR_BLOCK_ID
    assert pa.check_error(d.ws) == 0        # reading clears it


def test_out_of_range_slot_sets_error_word():
    import paged_kv_cache_286_gb300 as pa
    h = _h()
    w = make_workload([10], [10], num_q_heads=4, num_kv_heads=4, head_dim=64, seed=4)
    d = h.DeviceStep(w)
    d.slots[3] = w.num_blocks * 16
    d.append_new()
    with pytest.raises(pa.PagedAttnError):
        pa.check_error(d.ws)


def test_inconsistent_lengths_set_error_word():
    import paged_kv_cache_286_gb300 as pa
    h = _h()
    w = make_workload([10, 40], [1, 1], num_q_heads=4, num_kv_heads=4, head_dim=64, seed=6)
    d = h.DeviceStep(w)
    d.append_prior()
    d.append_new()
    d.ctx[0] = 0                      # n_s = 1 > context_len = 0
    d.attend()
    word = pa.check_error(d.ws, raise_on_error=False)
    assert word & pa._lib.PA_DEVERR_LENGTHS


# ---- the full-size named workloads (launch configuration of the benchmark) ---------------
def _full(cid):
    """Every row of a full-size named workload against the oracle, element by element; the
    oracle runs sharded over the host cores (paged_attention_parallel runs paged_attention
    itself on shares of the sequences)."""
    from oracle import paged_attention_parallel
    h = _h()
    w = make_config(cid)
    d, out = h.run_gpu(w)
    kp, vp = _oracle_pools(w)
    gk, gv = d.pools_numpy()
    assert np.array_equal(gk, kp) and np.array_equal(gv, vp), "append is not bit-exact"
    del gk, gv
    ref = paged_attention_parallel(w.q_bits, kp, vp, w.block_tables, w.context_lens,
                                   w.query_start_loc, w.num_q_heads, w.num_kv_heads,
                                   w.head_dim, w.scale, w.block_size, w.cache_dtype,
                                   w.k_scale, w.v_scale)
    assert not np.isnan(ref).any()
    return h.assert_close_to_oracle(w, out, ref)


@pytest.mark.slow
def test_config2_full_size_every_row():
    _full(2)


@pytest.mark.slow
def test_config3_full_size_every_row():
    _full(3)


@pytest.mark.slow
def test_config4_full_size_every_row():
    _full(4)


@pytest.mark.slow
def test_config5_full_size_every_row():
    _full(5)


@pytest.mark.slow
def test_speculative_verify_workload_every_row():
    """Multi-query verify step (1 accepted + 4 draft tokens per sequence, causal among them)."""
    _full(6)


def test_step_replays_from_a_cuda_graph():
    """The library's calls are stream-ordered with no host synchronisation: a whole step
    (append + attention) captured in a CUDA graph and replayed gives the eager result."""
    h = _h()
    w = make_workload([300, 1000, 2500, 40], [1, 1, 37, 1], num_q_heads=16, num_kv_heads=4,
                      head_dim=128, seed=123)
    d, out_eager = h.run_gpu(w)
    out_eager = out_eager.clone()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        d.step()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=cap):
        d.step()
    d.out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(d.out, out_eager)


def test_concurrent_callers_on_their_own_streams():
    """Two host threads run attention steps with prefill chunks (which fork the prefill tiles to
    a per-thread side stream) on their own streams and workspaces over one shared pool; each
    result equals the single-caller one bitwise."""
    import threading
    import paged_kv_cache_286_gb300 as pa
    h = _h()
    w = make_workload([300, 1000, 2500, 40], [1, 1, 37, 1], num_q_heads=16, num_kv_heads=4,
                      head_dim=128, seed=321)
    d, ref = h.run_gpu(w)
    ref = ref.clone()
    outs, errors = {}, []

    def caller(tag):
        try:
            stream = torch.cuda.Stream()
            ws = pa.new_workspace(d.ws.numel())
            out = torch.empty_like(d.out)
            with torch.cuda.stream(stream):
                for _ in range(5):
                    pa.attention(d.q, d.k_cache, d.v_cache, d.tables, d.ctx, d.qsl, ws,
                                 scale=w.scale, max_context_len=w.max_context_len,
                                 max_query_len=w.max_query_len, out=out, stream=stream)
            stream.synchronize()
            assert pa.check_error(ws, stream=stream) == 0
            outs[tag] = out
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=caller, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for tag in (0, 1):
        assert torch.equal(outs[tag], ref)


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_poisoned_workspace_gives_the_same_output(dtype):
    """Every byte of the workspace past its header filled with 0xFF (fp32 NaN) before the step:
    the partials, item tables and plan arrays are all written before they are read, so the
    output equals the one from a clean workspace bitwise."""
    import paged_kv_cache_286_gb300 as pa
    h = _h()
    w = make_workload([5000, 3100, 700, 1], [1, 1, 1, 1], num_q_heads=8, num_kv_heads=2,
                      head_dim=128, seed=77, cache_dtype=dtype)
    d, ref = h.run_gpu(w)
    ref = ref.clone()
    ws = pa.new_workspace(d.ws.numel())
    ws[pa.PA_WORKSPACE_HEADER_BYTES:].fill_(255)
    out = torch.full_like(d.out, float("nan"))
    pa.attention(d.q, d.k_cache, d.v_cache, d.tables, d.ctx, d.qsl, ws, scale=w.scale,
                 max_context_len=w.max_context_len, max_query_len=w.max_query_len, out=out,
                 k_scale=w.k_scale, v_scale=w.v_scale)
    assert pa.check_error(ws) == 0
    assert torch.equal(out, ref)


def test_pipelined_host_loop_reads_back_every_step_output():
    """bench.py's end-to-end loop (packed inputs copied in, output copied back, double-buffered
    against the compute on a copy stream) hands back the step's output in both host buffers."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    w = make_config(4)
    dw = bench.DeviceWorkload(w, torch.device("cuda", 0))
    dw.step()
    torch.cuda.synchronize()
    ref = dw.out.cpu()
    for t in (dw.out, dw.out2):
        t.fill_(float("nan"))
    for t in (dw.out_host, dw.out_host2):
        t.fill_(float("nan"))
    dw.steps_from_host(4, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.equal(dw.out_host, ref) and torch.equal(dw.out_host2, ref)
