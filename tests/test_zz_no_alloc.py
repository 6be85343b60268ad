"""pa_attention_noalloc: the attention entry point for callers that cannot allocate device
memory (for example code running under a memory manager that owns the whole device, or code
that must not grow its footprint after start-up).  It keeps its scratch in an array built into
the library instead of a caller workspace.

The GPU test calls it through the C ABI three times in a row, on different steps (split-KV
with a merge, chunked-prefill tiles, and a smaller step last, so that stale scratch from the
calls before would show), and checks each output against the fp64 oracle within the parity
tolerance, and bit for bit against the workspace-taking pa_attention on the same inputs (the
same kernels, with their scratch elsewhere).  This file is named so that pytest collects it
last.
"""

import ctypes

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
def test_noalloc_matches_the_oracle_on_three_calls_in_a_row():
    import gpu_harness as h
    from oracle import run_step
    _l, lib = _lib()
    steps = [
        make_workload([9000, 300, 17], [1, 1, 1], num_q_heads=32, num_kv_heads=8,
                      head_dim=128, seed=41, pool_fill="nan"),       # split-KV + merge path
        make_workload([600, 90, 2000], [130, 1, 1], num_q_heads=32, num_kv_heads=8,
                      head_dim=128, seed=43, pool_fill="nan"),       # prefill tiles + decode
        make_config(1, pool_fill="nan"),                             # smaller, no split
    ]
    error_word = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    for w in steps:
        d, ws_out = h.run_gpu(w)               # pa_attention with a caller workspace
        ws_out = ws_out.clone()
        st, out = _call_noalloc(lib, d, error_word)
        assert st == _l.PA_OK, lib.pa_last_error_string().decode()
        torch.cuda.synchronize()
        assert int(error_word.item()) == 0
        _, _, ref = run_step(w)
        h.assert_close_to_oracle(w, out, ref)
        assert torch.equal(out, ws_out), "noalloc and workspace entry points differ"


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
