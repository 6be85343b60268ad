"""The device-side failure signal: a bounded wait that expires.

Every mbarrier wait of the library's kernels gives up after a limit (1 s by default, settable
per thread with pa_set_wait_limit_ns), records PA_DEVERR_TIMEOUT in the workspace's error word,
lets the copies it still has in flight land and returns, so the context stays usable and
pa_check_error reports PA_ERR_TIMEOUT.  These tests make such waits expire on purpose, with no
fault of any kind: the self-test waits on a barrier phase nothing completes, and the test hook
pa_test_skip_one_copy leaves out one tile copy whose bytes the barrier still expects.  Each
forced expiry is followed by a clean call on the same device whose output must match the oracle.
"""

import ctypes
import time

import pytest
import torch

from oracle import run_step
from synthetic import make_workload

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000  # 2 ms


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_286_gb300 import build, _lib
    build.build()
    return _lib.load()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _status_of_check(lib, ws):
    word = ctypes.c_uint32(0)
    st = lib.pa_check_error(ctypes.c_void_p(ws.data_ptr()), _stream(), ctypes.byref(word))
    return st, int(word.value)


def test_selftest_wait_expires_and_reports_timeout(lib):
    import paged_kv_cache_286_gb300 as pa
    ws = pa.new_workspace(256)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    assert lib.pa_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), LIMIT_NS, _stream()) == 0
    st, word = _status_of_check(lib, ws)
    dt = time.monotonic() - t0
    assert st == pa._lib.PA_ERR_TIMEOUT and word & pa._lib.PA_DEVERR_TIMEOUT, (st, word)
    assert dt < 0.5, dt
    assert _status_of_check(lib, ws) == (0, 0)   # the check cleared the word


CASES = {
    # single-token decode, bf16, GQA 4: split-KV kernel (one kv head per item) and the merge
    "decode_bf16": dict(ctx=[2000, 700, 33], ql=[1, 1, 1], hq=8, hkv=2, dtype="bf16"),
    # single-token decode, E4M3, GQA 4: the two-heads-per-item instance
    "decode_e4m3": dict(ctx=[2000, 700, 33], ql=[1, 1, 1], hq=8, hkv=2, dtype="fp8_e4m3"),
    # a 300-token chunk after a prefix beside a decode: both kernels time out
    "chunk_bf16": dict(ctx=[900, 600], ql=[300, 1], hq=8, hkv=2, dtype="bf16"),
    # speculative-verify runs of 20 rows: the tensor-core tiles with rows split over two warps
    "verify_bf16": dict(ctx=[600, 900], ql=[5, 5], hq=8, hkv=2, dtype="bf16"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_missing_copy_times_out_then_the_next_call_is_correct(lib, name):
    import gpu_harness as h
    import paged_kv_cache_286_gb300 as pa
    c = CASES[name]
    w = make_workload(c["ctx"], c["ql"], num_q_heads=c["hq"], num_kv_heads=c["hkv"],
                      head_dim=128, cache_dtype=c["dtype"], seed=97, pool_fill="nan")
    d = h.DeviceStep(w)
    d.append_prior()
    d.append_new()
    assert pa.check_error(d.ws) == 0
    lib.pa_set_wait_limit_ns(LIMIT_NS)
    lib.pa_test_skip_one_copy(1)
    try:
        t0 = time.monotonic()
        d.attend()
        st, word = _status_of_check(lib, d.ws)
        dt = time.monotonic() - t0
    finally:
        lib.pa_test_skip_one_copy(0)
        lib.pa_set_wait_limit_ns(0)
    assert st == pa._lib.PA_ERR_TIMEOUT, (st, word)
    assert word & pa._lib.PA_DEVERR_TIMEOUT
    assert dt < 1.0, dt       # a few limits at most, far below the default 1 s per wait
    # the same context, the same pools: a clean call gives the oracle's result
    out = d.attend()
    assert pa.check_error(d.ws) == 0
    _, _, ref = run_step(w)
    h.assert_close_to_oracle(w, out, ref)
