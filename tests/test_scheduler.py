"""The continuous-batching step simulator against the pages' scheduling examples (host-only)."""

import numpy as np
import pytest

from conftest import load_golden

pa_build = pytest.importorskip("paged_kv_cache_286_gb300.build")
G = load_golden("page_arithmetic.txt")


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()


def _sched(**kw):
    from paged_kv_cache_286_gb300.scheduler import Scheduler
    return Scheduler(**kw)


def _req(*a, **kw):
    from paged_kv_cache_286_gb300.scheduler import Request
    return Request(*a, **kw)


def test_worked_timeline_slots_refill_on_the_next_step():
    """P2 "Worked Timeline": A-D need 10, 40, 20 and 80 tokens, E and F wait; A ends at step 10
    and E joins at once; C ends at step 20 and F joins."""
    lens = [int(x) for x in G["static_lengths"].split(",")]
    s = _sched(num_blocks=64, max_num_seqs=4, token_budget=64)
    for i, n in enumerate(lens + [30, 30]):
        s.submit(_req(i, prompt_len=1, output_len=n))
    s.run()
    by = {r.rid: r for r in s.done}
    assert [by[i].finish_step for i in range(4)] == [10, 40, 20, 80]
    assert by[4].admitted_step == 11 and by[5].admitted_step == 21
    # every step runs as many sequences as there are slots while work remains
    busy = [len(b.seq_ids) for b in s.history[:40]]
    assert all(b == 4 for b in busy)


def test_static_batching_wastes_slots():
    """P2 "Worked Example: Wasted Slots": 150 useful of 320 paid slot-steps, about 47 percent;
    continuous batching finishes the same four requests with every slot used until the queue
    drains."""
    from paged_kv_cache_286_gb300.scheduler import static_batch_steps
    lens = [int(x) for x in G["static_lengths"].split(",")]
    steps, useful, paid = static_batch_steps(lens, 4)
    assert (steps, useful, paid) == (80, int(G["static_useful"]), int(G["static_paid"]))
    assert round(100 * useful / paid) == int(G["static_utilization_pct"])
    s = _sched(num_blocks=64, max_num_seqs=4, token_budget=64)
    for i, n in enumerate(lens):
        s.submit(_req(i, prompt_len=1, output_len=n))
    s.run()
    assert sum(len(b.seq_ids) for b in s.history) == useful   # no idle slot-steps are paid


def test_chunked_prefill_keeps_decodes_moving():
    """P1 "Continuous batching": a long prompt is split across steps by the token budget, and
    the decoding sequences get a token in every one of those steps."""
    s = _sched(num_blocks=512, max_num_seqs=8, token_budget=256)
    for i in range(3):
        s.submit(_req(i, prompt_len=8, output_len=40))
    s.run(max_steps=2)
    s.submit(_req(9, prompt_len=3000, output_len=2, arrival=3))
    s.run(max_steps=20)
    chunks = [int(b.query_lens[b.seq_ids.index(9)]) for b in s.history if 9 in b.seq_ids]
    assert len(chunks) >= 3000 // 256 and max(chunks) <= 256 - 3
    for b in s.history[2:14]:
        assert {0, 1, 2} <= set(b.seq_ids)                 # decodes never stall
        assert sum(b.query_lens) <= 256


def test_batches_are_valid_attention_inputs():
    s = _sched(num_blocks=256, max_num_seqs=16, token_budget=128)
    rng = np.random.default_rng(0)
    for i in range(24):
        s.submit(_req(i, prompt_len=int(rng.integers(1, 300)), output_len=int(rng.integers(1, 40)),
                      arrival=int(rng.integers(1, 30))))
    s.run()
    assert len(s.done) == 24
    for b in s.history:
        assert np.all(b.query_lens >= 1) and np.all(b.query_lens <= b.context_lens)
        assert b.query_start_loc[-1] == len(b.slot_mapping) == b.query_lens.sum()
        for i in range(len(b.seq_ids)):
            nb = -(-int(b.context_lens[i]) // 16)
            assert np.all(b.block_tables[i, :nb] >= 0)
            # the step's new tokens sit at the tail positions of the sequence
            t0, t1 = b.query_start_loc[i], b.query_start_loc[i + 1]
            pos = np.arange(b.context_lens[i] - (t1 - t0), b.context_lens[i])
            want = b.block_tables[i, pos // 16].astype(np.int64) * 16 + pos % 16
            assert np.array_equal(b.slot_mapping[t0:t1], want)


def test_preemption_when_memory_runs_out():
    """P2 "What the Scheduler Does": if memory runs short mid-flight a sequence is preempted,
    its cache freed, and it is recomputed later; every request still completes."""
    s = _sched(num_blocks=12, max_num_seqs=8, token_budget=64)
    for i in range(6):
        s.submit(_req(i, prompt_len=10, output_len=40))
    s.run()
    assert len(s.done) == 6
    assert any(b.preempted for b in s.history)
    assert sum(r.preemptions for r in s.done) >= 1
    assert s.bm.num_free() == 12


def test_shared_system_prompt_prefills_once_with_prefix_caching():
    """"08 serving many users", exercise: with prefix caching a shared 1,500-token system prompt
    (here 1504 tokens = 94 blocks) is prefilled once; requests arriving after it is cached
    prefill only their own suffix.  (Requests admitted in the same step as the first one cannot
    reuse it yet and compute it too.)"""
    sys_prompt = list(range(1504))

    def run(caching, arrival):
        s = _sched(num_blocks=2000, max_num_seqs=8, token_budget=4096, prefix_caching=caching)
        for i in range(8):
            s.submit(_req(i, prompt_len=1504 + 20, output_len=4, arrival=arrival(i),
                          prompt_tokens=sys_prompt + [9000 + 20 * i + j for j in range(20)]))
        s.run()
        return sum(r.prefill_tokens for r in s.done), sum(r.cached_tokens for r in s.done)

    staggered = lambda i: 1 + i  # noqa: E731
    cold, cached0 = run(False, staggered)
    warm, cached1 = run(True, staggered)
    assert cached0 == 0 and cold == 8 * 1524
    assert cached1 == 7 * 1504 and warm == 1504 + 8 * 20
    together, cached2 = run(True, lambda i: 1)
    assert cached2 > 0 and warm < together < cold
