"""Reference model of the KV block manager, written from the pages with plain Python containers.

Test infrastructure only (see the package docstring).  It fixes what the native manager must
do, operation by operation:

* "Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained":
  "Blocks and Block Tables" - a sequence takes a new block from the free list only when its
  current block is full; "Growing During Decode" - tokens go into the last block; a finished
  sequence returns all its blocks; "Shared Prefixes" / "The Savings in Numbers" - tables may
  point at the same block, counted by a reference count; "Copy-on-Write" - before a sequence
  writes into a block whose count is above one, the block is copied to a fresh one that only
  this sequence's table points at.
* "Why a Second Kind of Engine: Batching, Paged Attention and Throughput", "Prefix caching": a
  full block is identified by its tokens and all tokens before it; a new request reuses cached
  blocks for the longest such prefix; unused cached blocks are evicted least recently used
  first when space is needed.

Here a cached block is keyed by the whole token prefix up to its end (a tuple), which is what a
chained block hash identifies when it has no collisions.  Allocation order: free blocks in
first-in-first-out order starting from 0..N-1, then the least recently released cached block.
"""

from __future__ import annotations

from collections import OrderedDict, deque
from typing import Dict, List, Optional, Sequence


class NoSpace(Exception):
    pass


class _Seq:
    def __init__(self):
        self.blocks: List[int] = []
        self.ntok = 0
        self.hashing = True
        self.tokens: List[int] = []   # every token id so far (while hashing)


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int):
        self.bs = block_size
        self.ref = [0] * num_blocks
        self.free = deque(range(num_blocks))
        self.cache: Dict[tuple, int] = {}      # full prefix -> block
        self.key_of: Dict[int, tuple] = {}     # block -> its prefix key (cached blocks)
        self.lru: "OrderedDict[int, None]" = OrderedDict()
        self.seqs: Dict[int, _Seq] = {}

    def num_free(self) -> int:
        return len(self.free) + len(self.lru)

    def _take(self) -> int:
        if self.free:
            b = self.free.popleft()
        else:
            b, _ = self.lru.popitem(last=False)
            key = self.key_of.pop(b)
            if self.cache.get(key) == b:
                del self.cache[key]
        self.ref[b] = 1
        return b

    def _drop(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            if b in self.key_of:
                self.lru[b] = None
            else:
                self.free.append(b)

    def append(self, seq: int, n: int, tokens: Optional[Sequence[int]] = None):
        """Returns (slots, copy pairs, cached tokens); raises NoSpace with no change."""
        bs = self.bs
        s = self.seqs.get(seq, _Seq())
        hits = []
        if tokens is not None and s.ntok == 0:
            for off in range(0, n - bs + 1, bs):
                b = self.cache.get(tuple(tokens[:off + bs]))
                if b is None:
                    break
                hits.append(b)
        revived = sum(1 for b in hits if self.ref[b] == 0 and b in self.lru)
        cur = s.ntok + len(hits) * bs
        rest = n - len(hits) * bs
        partial = cur % bs != 0
        cow = rest > 0 and partial and bool(s.blocks) and self.ref[s.blocks[-1]] > 1
        room = bs - cur % bs if partial else 0
        new_blocks = -(-(rest - room) // bs) if rest > room else 0
        if new_blocks + (1 if cow else 0) > self.num_free() - revived:
            raise NoSpace()
        self.seqs[seq] = s
        slots, pairs = [], []
        for b in hits:
            if self.ref[b] == 0:
                self.lru.pop(b, None)
            self.ref[b] += 1
            s.blocks.append(b)
            slots.extend(b * bs + o for o in range(bs))
            s.ntok += bs
        if hits:
            s.tokens = list(tokens[:len(hits) * bs])
        if cow:
            old = s.blocks[-1]
            new = self._take()
            pairs.append((old, new))
            self._drop(old)
            s.blocks[-1] = new
        if tokens is None and rest > 0:
            s.hashing = False
        for i in range(rest):
            if s.ntok % bs == 0:
                s.blocks.append(self._take())
            b = s.blocks[s.ntok // bs]
            slots.append(b * bs + s.ntok % bs)
            s.ntok += 1
            if s.hashing and tokens is not None:
                s.tokens.append(int(tokens[len(hits) * bs + i]))
                if s.ntok % bs == 0:
                    key = tuple(s.tokens)
                    if key not in self.cache and b not in self.key_of:
                        self.cache[key] = b
                        self.key_of[b] = key
        return slots, pairs, len(hits) * bs

    def fork(self, parent: int, child: int) -> None:
        p = self.seqs[parent]
        assert child not in self.seqs
        c = _Seq()
        c.blocks, c.ntok, c.hashing, c.tokens = list(p.blocks), p.ntok, p.hashing, list(p.tokens)
        for b in c.blocks:
            self.ref[b] += 1
        self.seqs[child] = c

    def free_seq(self, seq: int) -> None:
        for b in self.seqs.pop(seq).blocks:
            self._drop(b)

    def table(self, seq: int) -> List[int]:
        return list(self.seqs[seq].blocks)
