"""Runs a synthetic workload through the CUDA library (C ABI via the Python binding) and, on
the oracle side, through ``oracle.run_step``; used by the GPU parity tests and smoke()."""

from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_286_gb300 as pa

BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F


def _bits_to_dev(bits: np.ndarray) -> torch.Tensor:
    """Raw bit patterns (uint16 = bf16, uint8 = E4M3) to a CUDA tensor of the matching dtype."""
    bits = np.ascontiguousarray(bits)
    if bits.dtype == np.uint16:
        t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(bits)
    return t.cuda()


def new_pools(w):
    """k/v pool tensors on the device holding the workload's initial fill."""
    shape = w.pool_shape
    if w.cache_dtype == "fp8_e4m3":
        fill = 0 if w.pool_fill == "zero" else E4M3_NAN
        k = torch.full(shape, fill, dtype=torch.uint8, device="cuda")
    else:
        fill = 0 if w.pool_fill == "zero" else BF16_NAN
        k = torch.full(shape, fill, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    return k, k.clone()


class DeviceStep:
    """Device copies of a workload's tensors plus pools and workspace."""

    def __init__(self, w, out_dtype=torch.float32):
        self.w = w
        self.q = _bits_to_dev(w.q_bits)
        self.k_new = _bits_to_dev(w.k_new_bits)
        self.v_new = _bits_to_dev(w.v_new_bits)
        self.slots = torch.from_numpy(w.slot_mapping).cuda()
        self.tables = torch.from_numpy(w.block_tables).cuda()
        self.ctx = torch.from_numpy(w.context_lens).cuda()
        self.qsl = torch.from_numpy(w.query_start_loc).cuda()
        self.k_cache, self.v_cache = new_pools(w)
        self.out = torch.empty((w.num_tokens, w.num_q_heads, w.head_dim), dtype=out_dtype,
                               device="cuda")
        nbytes = pa.attention_workspace_size(w.num_seqs, w.num_tokens, w.num_q_heads,
                                             w.num_kv_heads, w.head_dim,
                                             max(1, w.max_context_len), max(1, w.max_query_len))
        self.ws = pa.new_workspace(nbytes)

    def append_prior(self, chunk_tokens: int = 1 << 16):
        """Set-up: write the context that exists before the step, in chunks."""
        w = self.w
        P = w.slot_prior.shape[0]
        for a in range(0, P, chunk_tokens):
            b = min(P, a + chunk_tokens)
            k = _bits_to_dev(w.k_prior_bits[a:b])
            v = _bits_to_dev(w.v_prior_bits[a:b])
            s = torch.from_numpy(w.slot_prior[a:b]).cuda()
            pa.cache_append(k, v, s, self.k_cache, self.v_cache, self.ws, k_scale=w.k_scale,
                            v_scale=w.v_scale)

    def append_new(self):
        w = self.w
        pa.cache_append(self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache, self.ws,
                        k_scale=w.k_scale, v_scale=w.v_scale)

    def attend(self):
        w = self.w
        return pa.attention(self.q, self.k_cache, self.v_cache, self.tables, self.ctx, self.qsl,
                            self.ws, scale=w.scale, max_context_len=max(1, w.max_context_len),
                            max_query_len=max(1, w.max_query_len), out=self.out,
                            k_scale=w.k_scale, v_scale=w.v_scale)

    def step(self):
        self.append_new()
        return self.attend()

    def pools_numpy(self):
        if self.k_cache.dtype == torch.bfloat16:
            f = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
        else:
            f = lambda t: t.cpu().numpy()  # noqa: E731
        return f(self.k_cache), f(self.v_cache)


def run_gpu(w, out_dtype=torch.float32):
    """Set-up append, the step's append and attention on the GPU; returns (DeviceStep, out)."""
    d = DeviceStep(w, out_dtype)
    d.append_prior()
    out = d.step()
    word = pa.check_error(d.ws, raise_on_error=False)
    assert word == 0, f"device error word 0x{word:x}"
    return d, out


def tolerance(w) -> float:
    return 2e-2 if w.cache_dtype == "fp8_e4m3" else 2e-3


def assert_close_to_oracle(w, out_gpu: torch.Tensor, ref: np.ndarray, rows=None):
    """max |gpu - oracle| within the workload's tolerance, over the rows the oracle computed."""
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    mask = ~np.isnan(ref[:, 0, 0]) if rows is None else rows
    assert mask.any()
    g, r = got[mask], ref[mask]
    assert np.isfinite(g).all(), "non-finite output"
    tol = tolerance(w)
    if out_gpu.dtype == torch.bfloat16:
        # bf16 output: allow half an ulp of the rounded result on top
        bound = tol + np.abs(r) * 2.0 ** -8
        err = np.abs(g - r) - bound
        assert err.max() <= 0, f"max excess {err.max():.3g}"
    else:
        err = np.abs(g - r).max()
        assert err <= tol, f"max abs error {err:.3g} > {tol}"
    return float(np.abs(g - r).max())
