"""fp64 oracle: slot-mapped cache append and ragged paged attention.

Test infrastructure only (see the package docstring).  Plain and slow on purpose: sequences are
processed one by one, each sequence's keys and values are rebuilt as one contiguous array from
its block table, and attention is the textbook formula evaluated in float64.

Layout conventions (the pages fix none; these are the harness's):

* pool tensors ``k_pool``/``v_pool``: ``[num_blocks][num_kv_heads][block_size][head_dim]`` of raw
  codes (uint16 bf16 bit patterns, or uint8 OCP E4M3 codes with a per-tensor fp32 scale);
* ``slot = physical_block * block_size + offset``; a negative slot is padding and is skipped;
* ``context_lens[s]`` counts the keys of sequence s after this step's append; its ``n_s`` query
  tokens are the last ``n_s`` positions ``p_i = L_s - n_s + i``, and token i attends keys
  ``0..p_i`` (a decode token sees the whole history including itself; a prefill chunk is
  causal within itself and sees the cached prefix in full);
* q head h reads kv head ``h // (num_q_heads // num_kv_heads)``.
"""

from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from .e4m3 import decode as _e4m3_decode, encode_f32 as _e4m3_encode


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact float64 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32) \
        .astype(np.float64)


def _decode_cache(codes: np.ndarray, cache_dtype: str, scale: float) -> np.ndarray:
    if cache_dtype == "bf16":
        return bf16_bits_to_f64(codes)
    if cache_dtype == "fp8_e4m3":
        return _e4m3_decode(codes) * float(np.float32(scale))
    raise ValueError(cache_dtype)


def _encode_cache(bits: np.ndarray, cache_dtype: str, scale: float) -> np.ndarray:
    """Stored code of each new bf16 value: the bits themselves, or E4M3 of fl32(fl32(x)/scale)
    where the division is IEEE fp32 rounded to nearest."""
    if cache_dtype == "bf16":
        return np.asarray(bits, dtype=np.uint16)
    x = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return _e4m3_encode(np.divide(x, np.float32(scale), dtype=np.float32))


def cache_append(k_pool: np.ndarray, v_pool: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray,
                 slot_mapping: np.ndarray, block_size: int, cache_dtype: str = "bf16",
                 k_scale: float = 1.0, v_scale: float = 1.0):
    """Write each new token's k/v into its slot; returns new pool arrays.

    "Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained", section "Growing
    During Decode": each step appends the token into the last block of the sequence, at the next
    free offset; section "Blocks and Block Tables": the block is found through the table.  Here
    the table lookup has been folded into the slot: token t goes to block ``slot // block_size``
    at offset ``slot % block_size``, for every kv head.  Negative slots are skipped.
    """
    return scatter_codes(k_pool, v_pool, _encode_cache(k_bits, cache_dtype, k_scale),
                         _encode_cache(v_bits, cache_dtype, v_scale), slot_mapping, block_size)


def scatter_codes(k_pool: np.ndarray, v_pool: np.ndarray, k_codes: np.ndarray,
                  v_codes: np.ndarray, slot_mapping: np.ndarray, block_size: int):
    """The write half of ``cache_append``: already encoded per-token codes ``[T][H][D]`` go to
    block ``slot // block_size``, offset ``slot % block_size``; negative slots are skipped.
    Returns new pool arrays."""
    k_out = k_pool.copy()
    v_out = v_pool.copy()
    slots = np.asarray(slot_mapping, dtype=np.int64)
    total = k_pool.shape[0] * block_size
    if np.any(slots >= total):
        raise IndexError(f"slot outside a pool of {total} slots")
    keep = np.nonzero(slots >= 0)[0]
    b = slots[keep] // block_size
    o = slots[keep] % block_size
    # one assignment per (token, kv head); a slot written twice in one call is undefined
    k_out[b, :, o, :] = np.asarray(k_codes)[keep]
    v_out[b, :, o, :] = np.asarray(v_codes)[keep]
    return k_out, v_out


def gather_context(pool: np.ndarray, table_row: np.ndarray, context_len: int, block_size: int,
                   cache_dtype: str = "bf16", scale: float = 1.0) -> np.ndarray:
    """Rebuild one sequence's contiguous ``[L][num_kv_heads][head_dim]`` fp64 keys (or values).

    Same page, section "Attention Over Scattered Blocks": the kernel reads the block table and
    fetches each block from its physical location; logical block j of the sequence is physical
    block ``table_row[j]``, and its slot o holds position ``j * block_size + o``.
    """
    nblk = -(-context_len // block_size)
    ids = np.asarray(table_row[:nblk], dtype=np.int64)
    if np.any(ids < 0) or np.any(ids >= pool.shape[0]):
        raise IndexError("block table entry outside the pool")
    blocks = pool[ids]                                   # [nblk][H][bs][D]
    seq = np.transpose(blocks, (0, 2, 1, 3)).reshape(nblk * block_size, pool.shape[1],
                                                     pool.shape[3])
    return _decode_cache(seq[:context_len], cache_dtype, scale)


def _attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, first_pos: int, scale: float,
            group: int) -> np.ndarray:
    """Causal attention of n queries at positions first_pos..first_pos+n-1 over K/V [L][Hkv][D].

    Query i at position p attends keys 0..p:  a_j = scale * q . k_j,
    w = exp(a - max a) / sum exp(a - max a),  out = sum_j w_j v_j.
    """
    n, Hq, D = q.shape
    out = np.empty((n, Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        Kg = K[:, g, :]
        Vg = V[:, g, :]
        for i in range(n):
            p = first_pos + i
            a = scale * (Kg[:p + 1] @ q[i, h])
            w = np.exp(a - a.max())
            w /= w.sum()
            out[i, h] = w @ Vg[:p + 1]
    return out


def paged_attention(q_bits: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                    block_tables: np.ndarray, context_lens: np.ndarray,
                    query_start_loc: np.ndarray, num_q_heads: int, num_kv_heads: int,
                    head_dim: int, scale: float, block_size: int, cache_dtype: str = "bf16",
                    k_scale: float = 1.0, v_scale: float = 1.0,
                    seqs: Optional[Iterable[int]] = None) -> np.ndarray:
    """Attention of a ragged step batch over the paged pool, in fp64.

    Same page, section "Attention Over Scattered Blocks": the mathematics is that of ordinary
    attention, softmax of the query times the keys over the whole history; only the addressing
    changed.  Section "Prefill Versus Decode" and "Chunked Prefill": one step mixes decode
    tokens with prompt chunks, which attend causally to their cached prefix and to themselves.
    Returns ``[T][num_q_heads][head_dim]`` float64; rows of sequences left out of ``seqs`` are NaN.
    """
    assert num_q_heads % num_kv_heads == 0
    group = num_q_heads // num_kv_heads
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    T = int(qsl[-1])
    out = np.full((T, num_q_heads, head_dim), np.nan, dtype=np.float64)
    S = len(context_lens)
    for s in (range(S) if seqs is None else seqs):
        L = int(context_lens[s])
        t0, t1 = int(qsl[s]), int(qsl[s + 1])
        n = t1 - t0
        if n == 0:
            continue
        assert 0 < n <= L
        K = gather_context(k_pool, block_tables[s], L, block_size, cache_dtype, k_scale)
        V = gather_context(v_pool, block_tables[s], L, block_size, cache_dtype, v_scale)
        q = bf16_bits_to_f64(q_bits[t0:t1])
        out[t0:t1] = _attend(q, K, V, L - n, scale, group)
    return out


def attention_partial(q: np.ndarray, K: np.ndarray, V: np.ndarray, keys: slice, scale: float):
    """Softmax restricted to a key range: (normalised output, natural-log sum of exponentials).

    For one query vector q [D] over contiguous K/V [L][D]: a_j = scale q.k_j for j in ``keys``;
    returns (sum_j e^{a_j - m} v_j / sum_j e^{a_j - m},  m + ln sum_j e^{a_j - m}).
    """
    a = scale * (K[keys] @ q)
    m = a.max()
    e = np.exp(a - m)
    return (e @ V[keys]) / e.sum(), m + np.log(e.sum())


def lse_merge(outs: np.ndarray, lses: np.ndarray) -> np.ndarray:
    """Combine softmax partials over disjoint key ranges into the full-range result.

    With l_p = e^{lse_p}: out = sum_p l_p o_p / sum_p l_p, evaluated against the largest lse.
    """
    lses = np.asarray(lses, dtype=np.float64)
    w = np.exp(lses - lses.max())
    return (w[:, None] * np.asarray(outs)).sum(0) / w.sum()


def run_step(w, seqs: Optional[Iterable[int]] = None):
    """Whole step for a ``synthetic.Workload``: set-up append of the prior context, the step's
    append, then attention.  Returns (k_pool, v_pool, out)."""
    k_pool, v_pool = w.empty_pool(), w.empty_pool()
    k_pool, v_pool = cache_append(k_pool, v_pool, w.k_prior_bits, w.v_prior_bits, w.slot_prior,
                                  w.block_size, w.cache_dtype, w.k_scale, w.v_scale)
    k_pool, v_pool = cache_append(k_pool, v_pool, w.k_new_bits, w.v_new_bits, w.slot_mapping,
                                  w.block_size, w.cache_dtype, w.k_scale, w.v_scale)
    out = paged_attention(w.q_bits, k_pool, v_pool, w.block_tables, w.context_lens,
                          w.query_start_loc, w.num_q_heads, w.num_kv_heads, w.head_dim, w.scale,
                          w.block_size, w.cache_dtype, w.k_scale, w.v_scale, seqs=seqs)
    return k_pool, v_pool, out
