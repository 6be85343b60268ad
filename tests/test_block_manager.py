"""The native block manager (free list, tables, reference counts, copy-on-write, prefix cache)
against the pages' worked examples and against the plain Python model in oracle/.
Host-only: runs without a GPU."""

import random

import numpy as np
import pytest

from conftest import load_golden
from oracle.block_manager import BlockManagerModel, NoSpace as ModelNoSpace

pa_build = pytest.importorskip("paged_kv_cache_286_gb300.build")
G = load_golden("page_arithmetic.txt")


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()


def _bm(nb, bs=16):
    from paged_kv_cache_286_gb300.block_manager import BlockManager
    return BlockManager(nb, bs)


def test_blocks_are_taken_only_when_the_last_one_fills():
    """P2 "Worked Example: Fragmentation Saved" / "Growing During Decode": 300 tokens appended
    one per step hold 19 blocks, the last with 12 tokens; a block is taken on token 16k+1."""
    bm = _bm(64)
    taken_at = []
    for t in range(int(G["frag_tokens"])):
        before = bm.num_free()
        slots, pairs = bm.append(7, 1)
        assert pairs == []
        if bm.num_free() < before:
            taken_at.append(t)
    table = bm.block_table(7)
    assert len(table) == int(G["frag_blocks"])
    assert taken_at == [16 * k for k in range(19)]
    assert bm.num_tokens(7) == 300 and bm.num_tokens(7) % 16 == 12
    bm.free(7)                                  # finished: all blocks return at once
    assert bm.num_free() == 64


def test_prefix_shared_by_eight_requests_costs_ten_blocks():
    """P2 "Shared Prefixes" / "The Savings in Numbers": a 160-token prompt is 10 blocks; 8
    requests share one copy (refcount 8) instead of 80 blocks: 70 saved."""
    bm = _bm(200)
    prompt = list(range(1000, 1000 + int(G["prefix_tokens"])))
    cached = []
    for r in range(int(G["prefix_requests"])):
        slots, pairs, c = bm.append_tokens(r, prompt + [r, r + 1, r + 2])
        cached.append(c)
    assert cached == [0] + [160] * 7
    tables = [bm.block_table(r) for r in range(8)]
    prefix = {tuple(t[:10].tolist()) for t in tables}
    assert len(prefix) == 1                     # one physical copy
    assert all(bm.refcount(int(b)) == 8 for b in tables[0][:10])
    used = 200 - bm.num_free()
    assert used == 10 + 8                       # the prefix once + one tail block per request
    assert 8 * 10 - 10 == int(G["prefix_saved_blocks"])


def test_parallel_sampling_copies_only_the_last_block():
    """P2 "Copy-on-Write": samples forked from one prompt share its blocks and diverge by
    copying only the shared last block when they first write into it."""
    bm = _bm(32)
    bm.append_tokens(0, list(range(40)))        # 2 full blocks + 8 tokens
    for c in (1, 2, 3):
        bm.fork(0, c)
    base = bm.block_table(0)
    assert all(bm.refcount(int(b)) == 4 for b in base)
    copies = []
    for c in (1, 2, 3):
        slots, pairs, _ = bm.append_tokens(c, [99])
        copies.append(pairs)
        t = bm.block_table(c)
        assert t[:2].tolist() == base[:2].tolist()      # full blocks stay shared
        assert t[2] != base[2] and pairs == [(int(base[2]), int(t[2]))]
        assert slots[0] == t[2] * 16 + 8
    assert bm.refcount(int(base[2])) == 1               # only the parent still holds it
    slots, pairs, _ = bm.append_tokens(0, [5])          # the parent now writes in place
    assert pairs == [] and bm.block_table(0).tolist() == base.tolist()


def test_changing_the_first_token_breaks_every_prefix_match():
    """P1 "Prefix caching" (and its quiz): a block's identity covers all tokens before it, so a
    different first token matches nothing even if later tokens agree."""
    bm = _bm(64)
    prompt = list(range(64))
    bm.append_tokens(0, prompt)
    _, _, c_same = bm.append_tokens(1, prompt)
    _, _, c_diff = bm.append_tokens(2, [777] + prompt[1:])
    assert c_same == 64 and c_diff == 0


def test_unused_cached_blocks_are_evicted_least_recently_released_first():
    bm = _bm(6)
    bm.append_tokens(0, list(range(32)))        # blocks 0,1
    bm.append_tokens(1, list(range(100, 132)))  # blocks 2,3
    bm.free(0)
    bm.free(1)                                  # cached, evictable: 0,1 then 2,3
    assert bm.num_free() == 6
    bm.append(9, 16 * 4)                        # free 4,5 then evicts 0,1
    assert bm.block_table(9).tolist() == [4, 5, 0, 1]
    _, _, c = bm.append_tokens(10, list(range(100, 132)))   # 2,3 still cached
    assert c == 32 and bm.block_table(10).tolist() == [2, 3]
    bm.free(9)
    _, _, c = bm.append_tokens(11, list(range(32)))          # 0,1 were evicted
    assert c == 0


def test_no_space_changes_nothing():
    from paged_kv_cache_286_gb300.block_manager import NoSpace
    bm = _bm(4)
    bm.append(0, 40)
    with pytest.raises(NoSpace):
        bm.append(1, 40)
    assert bm.num_free() == 1 and bm.block_table(0).tolist() == [0, 1, 2]
    with pytest.raises(ValueError):
        bm.block_table(1)                       # the failed call created nothing


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_the_model(seed):
    rng = random.Random(seed)
    nb, bs = rng.choice([(24, 4), (40, 16), (12, 8)])
    bm, model = _bm(nb, bs), BlockManagerModel(nb, bs)
    from paged_kv_cache_286_gb300.block_manager import NoSpace
    live, next_id = [], 0
    vocab = [rng.randrange(3) for _ in range(6)]   # few prompts -> many prefix hits
    prompts = [[rng.randrange(50) for _ in range(rng.randrange(1, 5 * bs))] for _ in vocab]
    for _ in range(300):
        op = rng.random()
        if op < 0.35 or not live:
            seq = next_id
            next_id += 1
            toks = list(rng.choice(prompts)) if rng.random() < 0.8 else None
            n = len(toks) if toks else rng.randrange(1, 3 * bs)
            try:
                exp = model.append(seq, n, toks)
            except ModelNoSpace:
                exp = None
            try:
                got = bm.append_tokens(seq, toks) if toks else bm.append(seq, n) + (0,)
            except NoSpace:
                got = None
            assert (exp is None) == (got is None)
            if got is not None:
                assert got[0].tolist() == exp[0] and got[1] == exp[1] and got[2] == exp[2]
                live.append(seq)
        elif op < 0.7:
            seq = rng.choice(live)
            with_tokens = model.seqs[seq].hashing and rng.random() < 0.7
            k = rng.randrange(1, bs + 3)
            toks = [rng.randrange(50) for _ in range(k)] if with_tokens else None
            try:
                exp = model.append(seq, k, toks)
            except ModelNoSpace:
                exp = None
            try:
                got = bm.append_tokens(seq, toks) if toks else bm.append(seq, k) + (0,)
            except NoSpace:
                got = None
            assert (exp is None) == (got is None)
            if got is not None:
                assert got[0].tolist() == exp[0] and got[1] == exp[1]
        elif op < 0.8:
            parent = rng.choice(live)
            child = next_id
            next_id += 1
            model.fork(parent, child)
            bm.fork(parent, child)
            live.append(child)
        else:
            seq = live.pop(rng.randrange(len(live)))
            model.free_seq(seq)
            bm.free(seq)
        assert bm.num_free() == model.num_free()
        for s in live:
            assert bm.block_table(s).tolist() == model.table(s)
        for b in range(nb):
            assert bm.refcount(b) == model.ref[b]
