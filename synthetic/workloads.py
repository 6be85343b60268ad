"""Seeded synthetic workloads for one paged-attention step.

A workload is everything one continuous-batching step hands to the attention layer:

* the ragged step batch: ``context_lens[s]`` (keys visible to the last query of sequence s,
  including the tokens appended in this step) and ``query_start_loc`` (exclusive prefix sum of
  the per-sequence query counts ``n_s``);
* a block pool of ``num_blocks`` physical blocks of ``block_size`` token slots and a per-sequence
  block table mapping logical block j to a physical block id, with the ids drawn from a random
  permutation of the pool (blocks "need not be neighbors", vLLM page, "Blocks and Block Tables");
  optionally the first blocks of every table point at one shared copy of a common prefix
  (vLLM page, "Shared Prefixes");
* the prior context that the cache holds before the step (written by a set-up append), and the
  step's new tokens: q for every query token, k/v for every new token, and the slot mapping
  ``slot = physical_block * block_size + offset`` that says where each new token's k/v goes.

Values are fp32 N(0,1) draws from a CPU ``torch.Generator`` cast to bf16 (round to nearest
even); lengths and permutations come from ``numpy.random.default_rng``.  Everything is returned
as raw bit patterns (``uint16`` for bf16) so that both sides start from identical bytes.
This module contains no attention, quantisation or gather arithmetic.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

E4M3_MAX = 448.0  # largest finite OCP E4M3 magnitude; used only to pick the per-tensor scale

CONFIG_NAMES = {
    1: "tiny paged decode: Hq=Hkv=4, D=64, bs=16, 4 seqs with contexts 10/40/20/80, 32-block pool",
    2: "7B-class MHA decode: Hq=Hkv=32, D=128, bs=16, 64 seqs, contexts U[512,4096], bf16 KV",
    3: "GQA decode, fp8 e4m3 KV: Hq=32, Hkv=8, D=128, bs=16, 256 seqs, lognormal contexts "
       "(median 1000, sigma 0.8, clamp [16,8192])",
    4: "mixed step: Hq=32, Hkv=8, D=128, bs=16, 48 decodes U[256,4096] + prefill chunks "
       "(512 new, no prefix) and (512 new after a 2048-token prefix), bf16 KV",
    5: "long-context decode, shared prefix: Hq=32, Hkv=8, D=128, bs=16, 16 seqs at 32768 "
       "tokens sharing a 1504-token (94-block) prefix, bf16 KV",
    6: "speculative verify step: Hq=32, Hkv=8, D=128, bs=16, 64 seqs with contexts U[512,4096], "
       "5 causal query tokens each (1 accepted + 4 draft), bf16 KV",
}

_CHUNK = 1 << 24  # elements per generator draw; fixed so that draws are reproducible


def f32_to_bf16_bits(x: torch.Tensor) -> np.ndarray:
    """fp32 tensor -> bf16 bit patterns (uint16), round to nearest even (torch's cast)."""
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _randn_bf16(gen: torch.Generator, shape: Sequence[int]) -> np.ndarray:
    """Draw N(0,1) fp32 values in fixed-size chunks and cast them to bf16 bits."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    for start in range(0, n, _CHUNK):
        m = min(_CHUNK, n - start)
        out[start:start + m] = f32_to_bf16_bits(torch.randn(m, generator=gen, dtype=torch.float32))
    return out.reshape(shape)


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    cache_dtype: str            # "bf16" or "fp8_e4m3"
    scale: float                # softmax scale applied to q.k
    context_lens: np.ndarray    # int32 [S]
    query_start_loc: np.ndarray  # int32 [S+1]
    num_blocks: int
    block_tables: np.ndarray    # int32 [S, max_blocks_per_seq], -1 past the last used block
    q_bits: np.ndarray          # uint16 (bf16) [T, Hq, D]
    k_new_bits: np.ndarray      # uint16 (bf16) [T, Hkv, D]
    v_new_bits: np.ndarray      # uint16 (bf16) [T, Hkv, D]
    slot_mapping: np.ndarray    # int64 [T]
    k_prior_bits: np.ndarray    # uint16 (bf16) [P, Hkv, D]  context present before the step
    v_prior_bits: np.ndarray    # uint16 (bf16) [P, Hkv, D]
    slot_prior: np.ndarray      # int64 [P]
    k_scale: float = 1.0        # fp32 per-tensor scales of an fp8 cache (1.0 for bf16)
    v_scale: float = 1.0
    pool_fill: str = "zero"     # initial contents of every slot: "zero" or "nan" bit patterns
    shared_prefix_blocks: int = 0
    seed: int = 0

    # ---- derived sizes -------------------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def query_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc).astype(np.int32)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0

    @property
    def cache_elem_bytes(self) -> int:
        return 1 if self.cache_dtype == "fp8_e4m3" else 2

    @property
    def cache_np_dtype(self):
        return np.uint8 if self.cache_dtype == "fp8_e4m3" else np.uint16

    @property
    def pool_shape(self):
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    def empty_pool(self) -> np.ndarray:
        """One pool tensor (K or V) holding the initial fill pattern in every slot."""
        if self.pool_fill == "zero":
            fill = 0
        elif self.pool_fill == "nan":
            fill = 0x7F if self.cache_dtype == "fp8_e4m3" else 0x7FC0
        else:
            raise ValueError(self.pool_fill)
        return np.full(self.pool_shape, fill, dtype=self.cache_np_dtype)

    def attended_tokens(self) -> int:
        """Sum over query tokens of the keys each attends (decode: L_s; chunk: sum of p_i+1)."""
        total = 0
        for L, n in zip(self.context_lens.tolist(), self.query_lens.tolist()):
            # positions L-n .. L-1 attend L-n+1 .. L keys
            total += n * L - n * (n - 1) // 2
        return total

    def unique_blocks(self, seqs: Optional[Sequence[int]] = None) -> int:
        """Physical blocks referenced by the step, or by the sequences `seqs` (a shared block
        counts once)."""
        ids = set()
        for s in (range(self.num_seqs) if seqs is None else seqs):
            nb = -(-int(self.context_lens[s]) // self.block_size)
            ids.update(self.block_tables[s, :nb].tolist())
        return len(ids)

    def algorithmic_bytes(self, out_bytes_per_elem: int = 4,
                          seqs: Optional[Sequence[int]] = None) -> int:
        """Bytes a perfect implementation moves for the attention: unique K/V blocks touched
        (whole blocks, shared ones once), q read, out written, and the metadata read; over all
        sequences or only over `seqs`."""
        idx = list(range(self.num_seqs)) if seqs is None else list(seqs)
        kv = 2 * self.unique_blocks(idx) * self.num_kv_heads * self.block_size * \
            self.head_dim * self.cache_elem_bytes
        T = int(sum(int(self.query_lens[s]) for s in idx))
        qo = T * self.num_q_heads * self.head_dim * (2 + out_bytes_per_elem)
        meta = 4 * (len(idx) * 2 + 1) + 4 * sum(
            -(-int(self.context_lens[s]) // self.block_size) for s in idx)
        return int(kv + qo + meta)

    def append_bytes(self) -> int:
        """Bytes the step's append moves: bf16 k/v read, cache written, slots read."""
        T = self.num_tokens
        per = self.num_kv_heads * self.head_dim
        return int(T * per * 2 * 2 + T * per * self.cache_elem_bytes * 2 + T * 8)


def make_workload(context_lens: Sequence[int], query_lens: Sequence[int], *, num_q_heads: int,
                  num_kv_heads: int, head_dim: int, block_size: int = 16,
                  cache_dtype: str = "bf16", seed: int = 0, pool_factor: float = 1.25,
                  num_blocks: Optional[int] = None, shared_prefix_blocks: int = 0,
                  pool_fill: str = "zero", scale: Optional[float] = None,
                  name: str = "custom", permute: bool = True,
                  extra_table_cols: int = 0) -> Workload:
    """Build a seeded workload.

    ``context_lens[s]`` counts the keys of sequence s after this step's append;
    ``query_lens[s]`` (n_s <= context_lens[s]) of them are new this step.  The pool has
    ``num_blocks`` blocks (default ``ceil(pool_factor * blocks needed)``); physical ids are a
    random permutation of the pool unless ``permute`` is False.  With
    ``shared_prefix_blocks = m`` the first m logical blocks of every sequence map to the same m
    physical blocks, whose tokens are written once.
    """
    ctx = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    assert ctx.shape == ql.shape and ctx.ndim == 1
    assert np.all(ql >= 0) and np.all(ql <= ctx), "n_s must be in [0, L_s]"
    assert num_q_heads % num_kv_heads == 0
    S = ctx.shape[0]
    bs = block_size
    nblk = (ctx + bs - 1) // bs
    m = shared_prefix_blocks
    if m:
        assert np.all(ctx - ql >= m * bs), "new tokens must not land in shared prefix blocks"
    needed = m + int(np.sum(nblk - m)) if S else 0
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_factor * needed)))
    assert num_blocks >= needed, "pool too small"
    rng = np.random.default_rng(seed)
    ids = rng.permutation(num_blocks) if permute else np.arange(num_blocks)
    max_blocks = max(1, int(nblk.max()) if S else 1) + extra_table_cols
    tables = np.full((S, max_blocks), -1, dtype=np.int32)
    cursor = m
    for s in range(S):
        tables[s, :m] = ids[:m]
        k = int(nblk[s]) - m
        tables[s, m:m + k] = ids[cursor:cursor + k]
        cursor += k

    qsl = np.zeros(S + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(ql)
    T = int(qsl[-1])

    def slot_of(s: int, pos: int) -> int:
        return int(tables[s, pos // bs]) * bs + pos % bs

    slots_new = np.array([slot_of(s, int(ctx[s] - ql[s] + i))
                          for s in range(S) for i in range(int(ql[s]))], dtype=np.int64)
    prior = []
    for p in range(m * bs):  # shared prefix, written once
        prior.append(slot_of(0, p))
    for s in range(S):
        prior.extend(slot_of(s, p) for p in range(m * bs, int(ctx[s] - ql[s])))
    slots_prior = np.array(prior, dtype=np.int64)
    P = slots_prior.shape[0]

    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (T, num_q_heads, head_dim))
    k_new = _randn_bf16(gen, (T, num_kv_heads, head_dim))
    v_new = _randn_bf16(gen, (T, num_kv_heads, head_dim))
    k_prior = _randn_bf16(gen, (P, num_kv_heads, head_dim))
    v_prior = _randn_bf16(gen, (P, num_kv_heads, head_dim))

    k_scale = v_scale = 1.0
    if cache_dtype == "fp8_e4m3":
        def amax(*arrs):
            vals = [float(np.abs(bf16_bits_to_f32(a)).max()) for a in arrs if a.size]
            return max(vals) if vals else 1.0
        k_scale = float(np.float32(amax(k_new, k_prior)) / np.float32(E4M3_MAX))
        v_scale = float(np.float32(amax(v_new, v_prior)) / np.float32(E4M3_MAX))
    elif cache_dtype != "bf16":
        raise ValueError(cache_dtype)

    return Workload(
        name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=bs, cache_dtype=cache_dtype,
        scale=float(np.float32(1.0 / math.sqrt(head_dim))) if scale is None else float(scale),
        context_lens=ctx.astype(np.int32), query_start_loc=qsl, num_blocks=num_blocks,
        block_tables=tables, q_bits=q, k_new_bits=k_new, v_new_bits=v_new,
        slot_mapping=slots_new, k_prior_bits=k_prior, v_prior_bits=v_prior,
        slot_prior=slots_prior, k_scale=k_scale, v_scale=v_scale, pool_fill=pool_fill,
        shared_prefix_blocks=m, seed=seed)


def config_lengths(config_id: int):
    """(context_lens, query_lens, extra kwargs) of the five named workloads."""
    seed = 1000 + config_id
    rng = np.random.default_rng(seed)
    if config_id == 1:
        # the four request lengths of the vLLM page's static-batching example (10, 40, 20, 80)
        return [10, 40, 20, 80], [1, 1, 1, 1], dict(
            num_q_heads=4, num_kv_heads=4, head_dim=64, num_blocks=32)
    if config_id == 2:
        ctx = rng.integers(512, 4096, size=64, endpoint=True)
        return ctx.tolist(), [1] * 64, dict(num_q_heads=32, num_kv_heads=32, head_dim=128)
    if config_id == 3:
        ctx = np.clip(np.rint(rng.lognormal(mean=math.log(1000.0), sigma=0.8, size=256)),
                      16, 8192).astype(np.int64)
        return ctx.tolist(), [1] * 256, dict(num_q_heads=32, num_kv_heads=8, head_dim=128,
                                             cache_dtype="fp8_e4m3")
    if config_id == 4:
        ctx = rng.integers(256, 4096, size=48, endpoint=True).tolist()
        return ctx + [512, 2560], [1] * 48 + [512, 512], dict(
            num_q_heads=32, num_kv_heads=8, head_dim=128)
    if config_id == 5:
        return [32768] * 16, [1] * 16, dict(num_q_heads=32, num_kv_heads=8, head_dim=128,
                                            shared_prefix_blocks=94)
    if config_id == 6:
        ctx = rng.integers(512, 4096, size=64, endpoint=True)
        return ctx.tolist(), [5] * 64, dict(num_q_heads=32, num_kv_heads=8, head_dim=128)
    raise ValueError(f"no workload {config_id}")


def make_config(config_id: int, pool_fill: str = "zero") -> Workload:
    """One of the five named workloads, seeded with 1000 + config id."""
    ctx, ql, kw = config_lengths(config_id)
    return make_workload(ctx, ql, seed=1000 + config_id, pool_fill=pool_fill,
                         name=f"cfg{config_id}: {CONFIG_NAMES[config_id]}", **kw)
