"""Copy-on-write and prefix caching on the GPU: pa_copy_blocks is bit-exact, and a step the
native block manager plans (forked samples that copy their shared last block, a request that
reuses a cached prefix) gives the oracle's attention on the oracle's pool."""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import cache_append, paged_attention  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_286_gb300 import build
    build.build()


@pytest.mark.parametrize("fp8", [False, True])
def test_copy_blocks_is_bit_exact(fp8):
    import paged_kv_cache_286_gb300 as pa
    from paged_kv_cache_286_gb300 import _lib
    rng = np.random.default_rng(3)
    shape = (40, 4, 16, 128)
    dt = np.uint8 if fp8 else np.uint16
    kp = rng.integers(0, np.iinfo(dt).max, size=shape, dtype=dt)
    vp = rng.integers(0, np.iinfo(dt).max, size=shape, dtype=dt)
    perm = rng.permutation(40)
    pairs = np.stack([perm[:12], perm[12:24]], axis=1).astype(np.int32)   # disjoint
    tk = torch.from_numpy(kp if fp8 else kp.view(np.int16)).cuda()
    tv = torch.from_numpy(vp if fp8 else vp.view(np.int16)).cuda()
    ws = pa.new_workspace(256)
    desc = _lib.CacheDesc(40, 16, 4, 128, 1 if fp8 else 0, 1.0, 1.0)
    tp = torch.from_numpy(pairs).cuda()
    _lib.check(pa.library().pa_copy_blocks(ctypes.c_void_p(tk.data_ptr()),
                                           ctypes.c_void_p(tv.data_ptr()), ctypes.byref(desc),
                                           ctypes.c_void_p(tp.data_ptr()), 12,
                                           ctypes.c_void_p(ws.data_ptr()), None))
    assert pa.check_error(ws) == 0
    ek, ev = kp.copy(), vp.copy()
    ek[pairs[:, 1]] = kp[pairs[:, 0]]
    ev[pairs[:, 1]] = vp[pairs[:, 0]]
    gk = tk.cpu().numpy().view(dt)
    gv = tv.cpu().numpy().view(dt)
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


def test_step_planned_by_the_block_manager():
    import paged_kv_cache_286_gb300 as pa
    from paged_kv_cache_286_gb300 import _lib
    from paged_kv_cache_286_gb300.block_manager import BlockManager
    NB, BS, HKV, HQ, D = 64, 16, 2, 8, 128
    g = torch.Generator().manual_seed(5)
    bm = BlockManager(NB, BS)
    kp = np.zeros((NB, HKV, BS, D), np.uint16)
    vp = np.zeros_like(kp)
    tk = torch.zeros((NB, HKV, BS, D), dtype=torch.bfloat16, device="cuda")
    tv = torch.zeros_like(tk)
    ws = pa.new_workspace(1 << 20)
    desc = _lib.CacheDesc(NB, BS, HKV, D, 0, 1.0, 1.0)

    def kv(n):
        k = torch.randn(n, HKV, D, generator=g).bfloat16()
        v = torch.randn(n, HKV, D, generator=g).bfloat16()
        return k, v

    def write(slots, k, v):
        nonlocal kp, vp
        pa.cache_append(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), tk, tv, ws)
        kp, vp = cache_append(kp, vp, k.view(torch.int16).numpy().view(np.uint16),
                              v.view(torch.int16).numpy().view(np.uint16), slots, BS)

    def copy(pairs):
        nonlocal kp, vp
        if not pairs:
            return
        arr = torch.tensor(pairs, dtype=torch.int32, device="cuda")
        _lib.check(pa.library().pa_copy_blocks(ctypes.c_void_p(tk.data_ptr()),
                                               ctypes.c_void_p(tv.data_ptr()),
                                               ctypes.byref(desc), ctypes.c_void_p(arr.data_ptr()),
                                               len(pairs), ctypes.c_void_p(ws.data_ptr()), None))
        for s, d in pairs:
            kp[d], vp[d] = kp[s], vp[s]

    prompt = list(range(500, 540))                     # 40 tokens: 2 full blocks + 8
    slots, pairs, cached = bm.append_tokens(0, prompt)
    assert cached == 0 and pairs == []
    write(slots, *kv(40))
    for c in (1, 2, 3):                                 # three samples of the same prompt
        bm.fork(0, c)
    step_tokens = {}
    for c in (1, 2, 3):                                 # each writes its first sampled token
        slots, pairs, _ = bm.append_tokens(c, [900 + c])
        assert len(pairs) == 1                          # its shared last block is copied first
        copy(pairs)
        k, v = kv(1)
        write(slots, k, v)
        step_tokens[c] = 1
    slots, pairs, cached = bm.append_tokens(4, prompt[:32] + [7] * 5)   # a new request
    assert cached == 32                                 # two cached blocks reused
    write(slots[cached:], *kv(5))
    seqs = [1, 2, 3, 4]
    ctx = np.array([bm.num_tokens(s) for s in seqs], dtype=np.int32)
    qlen = np.array([1, 1, 1, 5], dtype=np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    tables = bm.tables(seqs)
    q = torch.randn(int(qsl[-1]), HQ, D, generator=g).bfloat16()
    scale = 1 / np.sqrt(D)
    out = pa.attention(q.cuda(), tk, tv, torch.from_numpy(tables).cuda(),
                       torch.from_numpy(ctx).cuda(), torch.from_numpy(qsl).cuda(), ws,
                       scale=scale, max_context_len=int(ctx.max()), max_query_len=5)
    assert pa.check_error(ws) == 0
    gk = tk.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gk, kp)
    ref = paged_attention(q.view(torch.int16).numpy().view(np.uint16), kp, vp, tables, ctx, qsl,
                          HQ, HKV, D, scale, BS)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref).max()
    assert err <= 2e-3, err


def test_scheduler_driven_steps_match_oracle():
    """Steps planned by the continuous-batching simulator (chunked prefill on the tensor-core
    tile path, decodes, preemptions, prefix-cache hits) run through pa_cache_append and
    pa_attention; every step's output matches the oracle on the oracle's own pool."""
    import paged_kv_cache_286_gb300 as pa
    from paged_kv_cache_286_gb300.scheduler import Request, Scheduler
    NB, BS, HKV, HQ, D = 96, 16, 2, 8, 128
    sch = Scheduler(num_blocks=NB, block_size=BS, max_num_seqs=6, token_budget=160,
                    prefix_caching=True)
    shared = list(range(7000, 7000 + 48))
    rng = np.random.default_rng(11)
    reqs = {}
    for i in range(10):
        pl = int(rng.integers(20, 260))
        toks = shared + [int(x) for x in rng.integers(0, 5000, pl)] if i % 2 == 0 else None
        r = Request(i, prompt_len=len(toks) if toks else pl, output_len=int(rng.integers(2, 12)),
                    arrival=1 + 2 * i, prompt_tokens=toks)
        reqs[i] = r
        sch.submit(r)
    kp = np.zeros((NB, HKV, BS, D), np.uint16)
    vp = np.zeros_like(kp)
    tk = torch.zeros((NB, HKV, BS, D), dtype=torch.bfloat16, device="cuda")
    tv = torch.zeros_like(tk)
    ws = pa.new_workspace(64 << 20)

    def kv_of(token, pos, salt):
        g = np.random.default_rng([token & 0x7FFFFFFF, pos, salt])
        x = torch.from_numpy(g.standard_normal((HKV, D)).astype(np.float32))
        return x.bfloat16()

    worst = [0.0]

    def execute(sb):
        nonlocal kp, vp
        ks, vs, qs = [], [], []
        for i, sid in enumerate(sb.seq_ids):
            toks = reqs[sid].token_ids()
            n = int(sb.query_lens[i])
            for pos in range(int(sb.context_lens[i]) - n, int(sb.context_lens[i])):
                ks.append(kv_of(toks[pos], pos, 1))
                vs.append(kv_of(toks[pos], pos, 2))
                qs.append(torch.cat([kv_of(toks[pos], pos, 3 + j) for j in range(HQ // HKV)]))
        k = torch.stack(ks)
        v = torch.stack(vs)
        q = torch.stack(qs)
        pa.cache_append(k.cuda(), v.cuda(), torch.from_numpy(sb.slot_mapping).cuda(), tk, tv, ws)
        kp, vp = cache_append(kp, vp, k.view(torch.int16).numpy().view(np.uint16),
                              v.view(torch.int16).numpy().view(np.uint16), sb.slot_mapping, BS)
        out = pa.attention(q.cuda(), tk, tv, torch.from_numpy(sb.block_tables).cuda(),
                           torch.from_numpy(sb.context_lens).cuda(),
                           torch.from_numpy(sb.query_start_loc).cuda(), ws, scale=D ** -0.5,
                           max_context_len=int(sb.context_lens.max()),
                           max_query_len=int(sb.query_lens.max()))
        ref = paged_attention(q.view(torch.int16).numpy().view(np.uint16), kp, vp,
                              sb.block_tables, sb.context_lens, sb.query_start_loc, HQ, HKV, D,
                              D ** -0.5, BS)
        err = float(np.abs(out.cpu().numpy().astype(np.float64) - ref).max())
        worst[0] = max(worst[0], err)
        assert err <= 2e-3, (sb.step, err)

    sch.run(executor=execute)
    assert pa.check_error(ws) == 0
    assert len(sch.done) == 10
    assert any(int(b.query_lens.max()) > 16 for b in sch.history)      # prefill tile path used
    assert sum(r.cached_tokens for r in sch.done) > 0                   # prefix cache hits
