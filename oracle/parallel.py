"""The oracle's ragged attention and E4M3 append spread over host processes (test
infrastructure only).

``paged_attention_parallel`` returns exactly what ``paged_attention`` returns: every worker runs
that same function, unchanged, on a share of the sequences, and the rows are put back in place.
``cache_append_parallel`` returns exactly what ``cache_append`` returns: the per-element
encoding runs on row chunks in the workers, the scatter in the caller.  Only the scheduling
differs.  The pools and queries go to the workers through shared memory (no
copy per worker); workers are started with ``spawn`` and use one BLAS thread each, so the
helper is safe to call from a process that has already initialised CUDA.
"""

from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory
from typing import Iterable, Optional

import numpy as np

from .paged_kv import _encode_cache, cache_append, paged_attention, scatter_codes

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _attach(spec):
    name, shape, dtype = spec
    shm = shared_memory.SharedMemory(name=name)
    return shm, np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)


def _worker(args):
    specs, meta, seqs = args
    handles = [_attach(s) for s in specs]
    try:
        q, kp, vp = (h[1] for h in handles)
        out = paged_attention(q, kp, vp, seqs=seqs, **meta)
        qsl = meta["query_start_loc"]
        return [(int(qsl[s]), np.array(out[int(qsl[s]):int(qsl[s + 1])])) for s in seqs]
    finally:
        for shm, _ in handles:
            shm.close()


def _shards(seqs, context_lens, query_start_loc, count):
    """Sequences dealt to `count` shards, largest work (queries x keys) first, each to the
    lightest shard so far."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    cost = {s: (int(qsl[s + 1] - qsl[s]) + 1) * int(context_lens[s]) for s in seqs}
    load = [0] * count
    out = [[] for _ in range(count)]
    for s in sorted(seqs, key=lambda s: -cost[s]):
        i = int(np.argmin(load))
        out[i].append(s)
        load[i] += cost[s]
    return [sorted(x) for x in out if x]


def paged_attention_parallel(q_bits: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                             block_tables: np.ndarray, context_lens: np.ndarray,
                             query_start_loc: np.ndarray, num_q_heads: int, num_kv_heads: int,
                             head_dim: int, scale: float, block_size: int,
                             cache_dtype: str = "bf16", k_scale: float = 1.0,
                             v_scale: float = 1.0, seqs: Optional[Iterable[int]] = None,
                             processes: Optional[int] = None) -> np.ndarray:
    """``paged_attention`` over ``processes`` host processes (default: every core this process
    may run on); same arguments, same result (rows of sequences left out of ``seqs`` are NaN)."""
    S = len(context_lens)
    seqs = list(range(S)) if seqs is None else [int(s) for s in seqs]
    if processes is None:
        try:
            processes = len(os.sched_getaffinity(0))
        except AttributeError:  # pragma: no cover
            processes = os.cpu_count() or 1
    processes = max(1, min(int(processes), len(seqs)))
    meta = dict(block_tables=np.asarray(block_tables), context_lens=np.asarray(context_lens),
                query_start_loc=np.asarray(query_start_loc), num_q_heads=num_q_heads,
                num_kv_heads=num_kv_heads, head_dim=head_dim, scale=scale,
                block_size=block_size, cache_dtype=cache_dtype, k_scale=k_scale,
                v_scale=v_scale)
    T = int(np.asarray(query_start_loc)[-1])
    out = np.full((T, num_q_heads, head_dim), np.nan, dtype=np.float64)
    if processes == 1 or not seqs:
        part = paged_attention(q_bits, k_pool, v_pool, seqs=seqs, **meta)
        mask = ~np.isnan(part[:, 0, 0])
        out[mask] = part[mask]
        return out
    shms, specs = [], []
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    try:
        for a in (q_bits, k_pool, v_pool):
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            shms.append(shm)
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            specs.append((shm.name, a.shape, a.dtype.str))
        for v in _THREAD_VARS:
            os.environ[v] = "1"
        shards = _shards(seqs, context_lens, query_start_loc, 4 * processes)
        with mp.get_context("spawn").Pool(processes) as pool:
            for rows in pool.imap_unordered(_worker, [(specs, meta, sh) for sh in shards]):
                for t0, block in rows:
                    out[t0:t0 + block.shape[0]] = block
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
        for shm in shms:
            shm.close()
            shm.unlink()
    return out


def _encode_rows(args):
    bits, cache_dtype, scale = args
    return _encode_cache(bits, cache_dtype, scale)


def cache_append_parallel(k_pool: np.ndarray, v_pool: np.ndarray, k_bits: np.ndarray,
                          v_bits: np.ndarray, slot_mapping: np.ndarray, block_size: int,
                          cache_dtype: str = "bf16", k_scale: float = 1.0, v_scale: float = 1.0,
                          processes: Optional[int] = None, rows_per_task: int = 4096):
    """``cache_append`` with the E4M3 encoding of the new rows spread over host processes;
    bf16 pools (no encoding) go straight to ``cache_append``."""
    if cache_dtype == "bf16" or len(slot_mapping) <= rows_per_task:
        return cache_append(k_pool, v_pool, k_bits, v_bits, slot_mapping, block_size,
                            cache_dtype, k_scale, v_scale)
    if processes is None:
        try:
            processes = len(os.sched_getaffinity(0))
        except AttributeError:  # pragma: no cover
            processes = os.cpu_count() or 1
    T = len(slot_mapping)
    tasks = [(np.asarray(bits[a:a + rows_per_task]), cache_dtype, scale)
             for bits, scale in ((k_bits, k_scale), (v_bits, v_scale))
             for a in range(0, T, rows_per_task)]
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    try:
        for v in _THREAD_VARS:
            os.environ[v] = "1"
        with mp.get_context("spawn").Pool(max(1, int(processes))) as pool:
            codes = pool.map(_encode_rows, tasks, chunksize=1)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    half = len(codes) // 2
    return scatter_codes(k_pool, v_pool, np.concatenate(codes[:half]),
                         np.concatenate(codes[half:]), slot_mapping, block_size)
