"""Python handle on the native block manager (include/pa_block_manager.h).

Host-only: the manager never touches the GPU, so it works without one.  It hands out the slots
that pa_cache_append writes, the block tables pa_attention reads, and the (source, destination)
pairs pa_copy_blocks must copy before a shared block is written.
"""

from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import numpy as np

from . import _lib

NO_SPACE = -1
BAD_ARG = -2


class NoSpace(RuntimeError):
    """Not enough free or evictable blocks; the manager is unchanged."""


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int = 16):
        self._L = _lib.load()
        self._h = self._L.pa_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._L.pa_bm_destroy(h)
            self._h = None

    @staticmethod
    def _check(rc: int) -> int:
        if rc == NO_SPACE:
            raise NoSpace("not enough free blocks")
        if rc < 0:
            raise ValueError("bad argument (unknown or duplicate sequence, bad count)")
        return rc

    def num_free(self) -> int:
        return int(self._L.pa_bm_num_free(self._h))

    def append(self, seq: int, n: int) -> Tuple[np.ndarray, List[Tuple[int, int]]]:
        """Reserve slots for n new tokens; returns (slots, copy-on-write pairs)."""
        slots = np.empty(max(n, 1), dtype=np.int64)
        pairs = np.empty(2, dtype=np.int32)
        rc = self._check(self._L.pa_bm_append(self._h, int(seq), int(n),
                                               slots.ctypes.data, pairs.ctypes.data, 1))
        return slots[:n], [(int(pairs[0]), int(pairs[1]))] if rc else []

    def append_tokens(self, seq: int, tokens: Sequence[int]
                      ) -> Tuple[np.ndarray, List[Tuple[int, int]], int]:
        """Like append, with token ids (makes full blocks cacheable; a new sequence reuses the
        longest cached prefix).  Returns (slots, copy pairs, tokens already cached)."""
        toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = int(toks.shape[0])
        slots = np.empty(max(n, 1), dtype=np.int64)
        pairs = np.empty(2, dtype=np.int32)
        cached = ctypes.c_int32(0)
        rc = self._check(self._L.pa_bm_append_tokens(self._h, int(seq), toks.ctypes.data, n,
                                                      slots.ctypes.data, pairs.ctypes.data, 1,
                                                      ctypes.byref(cached)))
        return slots[:n], ([(int(pairs[0]), int(pairs[1]))] if rc else []), int(cached.value)

    def cached_prefix(self, tokens: Sequence[int]) -> int:
        """Leading tokens a new sequence with these ids would find in the prefix cache."""
        toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return self._check(self._L.pa_bm_cached_prefix(self._h, toks.ctypes.data,
                                                        int(toks.shape[0])))

    def fork(self, parent: int, child: int) -> None:
        self._check(self._L.pa_bm_fork(self._h, int(parent), int(child)))

    def free(self, seq: int) -> None:
        self._check(self._L.pa_bm_free(self._h, int(seq)))

    def block_table(self, seq: int) -> np.ndarray:
        n = self._check(self._L.pa_bm_block_table(self._h, int(seq), None, 0))
        out = np.empty(max(n, 1), dtype=np.int32)
        self._L.pa_bm_block_table(self._h, int(seq), out.ctypes.data, n)
        return out[:n]

    def num_tokens(self, seq: int) -> int:
        return int(self._check(self._L.pa_bm_num_tokens(self._h, int(seq))))

    def refcount(self, block: int) -> int:
        return int(self._check(self._L.pa_bm_refcount(self._h, int(block))))

    def tables(self, seqs: Sequence[int], width: Optional[int] = None) -> np.ndarray:
        """Block tables of several sequences as one int32 array padded with -1."""
        rows = [self.block_table(s) for s in seqs]
        w = max([len(r) for r in rows] + [1]) if width is None else width
        out = np.full((len(rows), w), -1, dtype=np.int32)
        for i, r in enumerate(rows):
            out[i, :len(r)] = r
        return out
