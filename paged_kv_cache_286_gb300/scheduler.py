"""Continuous-batching step simulator that plans each step's ragged batch.

Host-only.  It reproduces the scheduling the pages describe and produces, for every step, the
inputs of the attention step: the slot mapping of the step's new tokens, query_start_loc,
context_lens and block tables.

* "Why a Second Kind of Engine: Batching, Paged Attention and Throughput", "Continuous batching":
  every step the scheduler forms the batch from the running sequences plus as many waiting
  prompts as the token budget and free KV blocks allow; a finished sequence leaves and releases
  its blocks in the same step; long prompts are cut into chunks ("chunked prefill") so that no
  step is spent on one prompt.
* "Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained", "Schedule Per
  Step", "Worked Timeline", "What the Scheduler Does": admission when memory allows; when memory
  runs out mid-flight a sequence is preempted (its cache is freed, it is recomputed later).
* Same page, "Static Batching", "Worked Example: Wasted Slots": a static batch runs until its
  longest member ends (static_batch_steps, for comparison).
* "08 serving many users", "Exercises": with prefix caching a shared system prompt costs its
  prefill once.

Request model: `prompt_len` prompt tokens, then `output_len` generated tokens.  The step that
completes the prompt yields the first token; each later step appends the previous token and
yields the next.  A preempted request recomputes its prompt and the tokens it had generated.
"""

from __future__ import annotations

import dataclasses
from collections import deque
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

from .block_manager import BlockManager


@dataclasses.dataclass
class Request:
    rid: int
    prompt_len: int
    output_len: int
    arrival: int = 1                      # first step at which it may be admitted
    prompt_tokens: Optional[Sequence[int]] = None
    computed: int = 0                     # tokens whose K/V are in the cache
    generated: int = 0
    admitted_step: Optional[int] = None
    first_token_step: Optional[int] = None
    finish_step: Optional[int] = None
    preemptions: int = 0
    cached_tokens: int = 0                # prompt tokens served by the prefix cache
    prefill_tokens: int = 0               # tokens it computed (prompt and recompute)

    def known(self) -> int:
        return self.prompt_len + self.generated

    def token_ids(self) -> List[int]:
        base = list(self.prompt_tokens) if self.prompt_tokens is not None else \
            [(self.rid * 1_000_003 + i) % 50_000 for i in range(self.prompt_len)]
        return base + [50_000 + (self.rid * 7919 + i) % 1000 for i in range(self.generated)]


@dataclasses.dataclass
class StepBatch:
    step: int
    seq_ids: List[int]
    query_lens: np.ndarray          # int32 [S]
    context_lens: np.ndarray        # int32 [S]
    query_start_loc: np.ndarray     # int32 [S+1]
    slot_mapping: np.ndarray        # int64 [T]
    block_tables: np.ndarray        # int32 [S, max_blocks]
    finished: List[int]
    preempted: List[int]


class Scheduler:
    def __init__(self, num_blocks: int, block_size: int = 16, max_num_seqs: int = 256,
                 token_budget: int = 2048, prefix_caching: bool = False):
        self.bm = BlockManager(num_blocks, block_size)
        self.bs = block_size
        self.max_num_seqs = max_num_seqs
        self.token_budget = token_budget
        self.prefix_caching = prefix_caching
        self.waiting: deque = deque()
        self.running: List[Request] = []
        self.done: List[Request] = []
        self.step_no = 0
        self.history: List[StepBatch] = []

    def submit(self, req: Request) -> None:
        self.waiting.append(req)

    def _blocks_needed(self, r: Request, n: int) -> int:
        cur = r.computed
        return -(-(cur + n) // self.bs) - (-(-cur // self.bs))

    def _preempt(self, r: Request) -> None:
        if r.computed or r in self.running:
            try:
                self.bm.free(r.rid)
            except ValueError:
                pass
        r.computed = 0
        r.preemptions += 1
        self.running.remove(r)
        self.waiting.appendleft(r)

    def _probe(self, r: Request) -> int:
        """Prompt tokens a fresh request would find in the prefix cache (at least the last
        known token is always computed, so that the step can yield a token)."""
        if not self.prefix_caching or r.computed:
            return 0
        return self.bm.cached_prefix(r.token_ids()[:r.known() - 1])

    def _reserve(self, r: Request, cached: int, n: int) -> np.ndarray:
        """Reuse `cached` leading tokens from the prefix cache (fresh requests only), then
        slots for the next n tokens of r; only the latter are queries of this step."""
        toks = r.token_ids()
        if not self.prefix_caching:
            slots, _ = self.bm.append(r.rid, n)
            r.computed += n
            return slots
        if r.computed == 0:
            _, _, hit = self.bm.append_tokens(r.rid, toks[:cached])
            r.cached_tokens += hit
            r.computed = hit
        lo, hi = r.computed, r.computed + n
        slots, _, _ = self.bm.append_tokens(r.rid, toks[lo:hi])
        r.computed = hi
        return slots

    def step(self) -> Optional[StepBatch]:
        self.step_no += 1
        t = self.step_no
        budget = self.token_budget
        plan: Dict[int, int] = {}
        hits: Dict[int, int] = {}
        for r in self.running:                      # running first: decodes, then prompt chunks
            n = min(r.known() - r.computed, budget)
            if n > 0:
                plan[r.rid] = n
                budget -= n
        while (self.waiting and len(self.running) < self.max_num_seqs and budget > 0
               and self.waiting[0].arrival <= t):
            r = self.waiting[0]
            c = self._probe(r)                      # cached prompt tokens cost no budget
            n = min(r.known() - r.computed - c, budget)
            if self._blocks_needed(r, c + n) > self.bm.num_free():
                break                               # admit only when memory allows
            self.waiting.popleft()
            self.running.append(r)
            if r.admitted_step is None:
                r.admitted_step = t
            plan[r.rid] = n
            hits[r.rid] = c
            budget -= n
        slots: Dict[int, np.ndarray] = {}
        preempted: List[int] = []
        for r in list(self.running):
            if r.rid not in plan or r not in self.running:
                continue
            n = plan[r.rid]
            c = hits.get(r.rid, 0)
            while self._blocks_needed(r, c + n) > self.bm.num_free() and r in self.running:
                victim = self.running[-1]           # the most recently admitted goes first
                self._preempt(victim)
                preempted.append(victim.rid)
                plan.pop(victim.rid, None)
                slots.pop(victim.rid, None)
            if r not in self.running:
                continue
            s = self._reserve(r, c, n)
            if r.first_token_step is None:
                r.prefill_tokens += len(s)
            if len(s):
                slots[r.rid] = s
        batch = [r for r in self.running if r.rid in slots]
        finished = []
        for r in self.running:
            if r.computed >= r.known() and r.rid in plan:   # the step yields a token
                r.generated += 1
                if r.first_token_step is None:
                    r.first_token_step = t
        if not batch:
            return None
        tables = self.bm.tables([r.rid for r in batch])
        qlens = np.array([len(slots[r.rid]) for r in batch], dtype=np.int32)
        ctx = np.array([r.computed for r in batch], dtype=np.int32)
        for r in list(self.running):
            if r.generated >= r.output_len:
                r.finish_step = t
                self.bm.free(r.rid)
                self.running.remove(r)
                self.done.append(r)
                finished.append(r.rid)
        sb = StepBatch(step=t, seq_ids=[r.rid for r in batch], query_lens=qlens, context_lens=ctx,
                       query_start_loc=np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32),
                       slot_mapping=np.concatenate([slots[r.rid] for r in batch]).astype(np.int64),
                       block_tables=tables, finished=finished, preempted=preempted)
        self.history.append(sb)
        return sb

    def run(self, max_steps: int = 100_000,
            executor: Optional[Callable[[StepBatch], None]] = None) -> None:
        while (self.waiting or self.running) and self.step_no < max_steps:
            sb = self.step()
            if sb is not None and executor is not None:
                executor(sb)


def static_batch_steps(output_lens: Sequence[int], slots: int):
    """Static batching: groups of `slots` requests run until their longest member ends.
    Returns (steps, useful slot-steps, paid slot-steps)."""
    steps = useful = paid = 0
    lens = list(output_lens)
    for i in range(0, len(lens), slots):
        group = lens[i:i + slots]
        steps += max(group)
        useful += sum(group)
        paid += max(group) * slots
    return steps, useful, paid
