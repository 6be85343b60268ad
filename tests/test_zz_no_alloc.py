"""pa_attention_noalloc: the attention entry point for callers that cannot allocate device
memory (for example code running under a memory manager that owns the whole device, or code
that must not grow its footprint after start-up).  It keeps its scratch in an array built into
the library instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row, on two different steps (the second one
smaller, so that stale scratch from the first call would show), and compares each output with
the workspace-taking pa_attention on the same inputs, within the parity tolerance.  This file
is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from synthetic import make_config, make_workload


def _lib():
    from paged_kv_cache_286_gb300 import _lib, build
    build.build()
    return _lib, _lib.load()


def _call_noalloc(lib, d, error_word):
    from paged_kv_cache_286_gb300 import cache_desc
    w = d.w
    out = torch.full_like(d.out, float("nan"))
    desc = cache_desc(d.k_cache, w.k_scale, w.v_scale)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.pa_attention_noalloc(
        p(d.q), w.num_tokens, p(d.k_cache), p(d.v_cache), ctypes.byref(desc), p(d.tables),
        w.max_blocks_per_seq, p(d.ctx), p(d.qsl), w.num_seqs, w.max_context_len,
        w.max_query_len, w.num_q_heads, w.num_kv_heads, w.head_dim, w.scale, p(out),
        2 if out.dtype == torch.float32 else 0, p(error_word),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    import gpu_harness as h
    _l, lib = _lib()
    first = make_workload([9000, 300, 17], [1, 1, 1], num_q_heads=32, num_kv_heads=8,
                          head_dim=128, seed=41, pool_fill="nan")       # split-KV + merge path
    second = make_config(1, pool_fill="nan")                             # smaller, no split
    error_word = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    for w in (first, second):
        d, ref = h.run_gpu(w)                  # pa_attention with a caller workspace
        ref = ref.clone()
        st, out = _call_noalloc(lib, d, error_word)
        assert st == _l.PA_OK, lib.pa_last_error_string().decode()
        torch.cuda.synchronize()
        assert int(error_word.item()) == 0
        diff = (out - ref).abs().max().item()
        assert np.isfinite(diff) and diff <= h.tolerance(w), diff


def test_noalloc_rejects_steps_beyond_its_scratch():
    _l, lib = _lib()
    from paged_kv_cache_286_gb300 import _lib as L
    desc = L.CacheDesc(1 << 20, 16, 8, 128, 0, 1.0, 1.0)
    fake = ctypes.c_void_p(0x100000)       # never dereferenced: rejected on the host first
    # 1024 sequences of 131072 tokens need far more than the built-in scratch
    need = lib.pa_attention_workspace_size(1024, 1024, 32, 8, 128, 16, 131072, 1)
    assert need > L.PA_NOALLOC_SCRATCH_BYTES
    st = lib.pa_attention_noalloc(fake, 1024, fake, fake, ctypes.byref(desc), fake, 8192, fake,
                                  fake, 1024, 131072, 1, 32, 8, 128, 0.088, fake, 2, None, None)
    assert st == L.PA_ERR_INVALID_ARG
    assert "scratch" in lib.pa_last_error_string().decode()
