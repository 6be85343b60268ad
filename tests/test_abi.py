"""The C-ABI library builds for sm_103a, loads without a GPU, exports every function that
include/pa.h declares, and rejects bad arguments on the host before launching anything."""

import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

pa_build = pytest.importorskip("paged_kv_cache_286_gb300.build")


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    from paged_kv_cache_286_gb300 import _lib
    return _lib.load()


def header_functions():
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    for n in ("pa_cache_append", "pa_attention", "pa_attention_workspace_size",
              "pa_check_error", "pa_last_error_string"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pa_build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pa_[a-z_0-9]+)$", out, flags=re.M))
    missing = [n for n in header_functions() if n not in exported]
    assert not missing, missing
    for n in header_functions():
        assert hasattr(lib, n)


def test_block_manager_header_is_exported(lib):
    with open(os.path.join(ROOT, "include", "pa_block_manager.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = sorted(set(re.findall(r"\b(pa_bm_[a-z_0-9]+)\s*\(", text)))
    from paged_kv_cache_286_gb300 import _lib
    assert names == sorted(_lib.EXPORTED_BM)
    out = subprocess.run(["nm", "-D", "--defined-only", pa_build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pa_bm_[a-z_0-9]+)$", out, flags=re.M))
    assert set(names) <= exported


def test_copy_blocks_rejects_bad_arguments(lib):
    d = _desc()
    assert lib.pa_copy_blocks(FAKE, FAKE, ctypes.byref(d), FAKE, -1, FAKE, None) == 1
    assert lib.pa_copy_blocks(FAKE, FAKE, ctypes.byref(d), FAKE, 70000, FAKE, None) == 1
    assert lib.pa_copy_blocks(FAKE, FAKE, ctypes.byref(d), None, 3, FAKE, None) == 1
    assert lib.pa_copy_blocks(FAKE, FAKE, ctypes.byref(d), FAKE, 0, FAKE, None) == 0


def test_binding_lists_every_export():
    from paged_kv_cache_286_gb300 import _lib
    assert sorted(_lib.EXPORTED) == header_functions()


def test_version_and_workspace_size(lib):
    from paged_kv_cache_286_gb300 import _lib
    assert lib.pa_version().decode().count(".") == 2
    hdr = _lib.PA_WORKSPACE_HEADER_BYTES
    small = lib.pa_attention_workspace_size(4, 4, 4, 4, 64, 16, 80, 1)
    assert small >= hdr
    # a long single-partition-per-sequence problem needs split partials: grows with context
    a = lib.pa_attention_workspace_size(16, 16, 32, 8, 128, 16, 32768, 1)
    b = lib.pa_attention_workspace_size(16, 16, 32, 8, 128, 16, 65536, 1)
    assert b > a > hdr


def _desc(**kw):
    from paged_kv_cache_286_gb300 import _lib
    d = dict(num_blocks=32, block_size=16, num_kv_heads=4, head_dim=64, cache_dtype=0,
             k_scale=1.0, v_scale=1.0)
    d.update(kw)
    return _lib.CacheDesc(**d)


FAKE = ctypes.c_void_p(0x100000)   # never dereferenced: every case fails validation first


@pytest.mark.parametrize("desc_kw,status", [
    (dict(block_size=32), 2), (dict(head_dim=72), 2), (dict(cache_dtype=7), 2),
    (dict(num_blocks=0), 1), (dict(cache_dtype=1, k_scale=0.0), 1),
])
def test_append_rejects_bad_cache_descriptors(lib, desc_kw, status):
    d = _desc(**desc_kw)
    st = lib.pa_cache_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), FAKE, None)
    assert st == status
    assert lib.pa_last_error_string().decode()


def test_append_rejects_null_and_negative(lib):
    d = _desc()
    assert lib.pa_cache_append(FAKE, FAKE, FAKE, -1, FAKE, FAKE, ctypes.byref(d), FAKE, None) == 1
    assert lib.pa_cache_append(None, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), FAKE, None) == 1
    assert lib.pa_cache_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, None, FAKE, None) == 1
    assert lib.pa_cache_append(FAKE, FAKE, FAKE, 0, FAKE, FAKE, ctypes.byref(d), None, None) == 1
    misaligned = ctypes.c_void_p(0x100008)  # 8 bytes past a 16-byte boundary
    assert lib.pa_cache_append(misaligned, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), FAKE,
                               None) == 1
    # zero tokens with valid arguments is a no-op that touches nothing
    assert lib.pa_cache_append(FAKE, FAKE, FAKE, 0, FAKE, FAKE, ctypes.byref(d), FAKE, None) == 0


def _attn(lib, **kw):
    d = kw.pop("desc", _desc())
    args = dict(q=FAKE, T=4, k=FAKE, v=FAKE, tables=FAKE, maxb=5, ctx=FAKE, qsl=FAKE, S=4,
                maxctx=80, maxq=1, hq=4, hkv=4, dim=64, scale=0.125, out=FAKE, odt=2,
                ws=ctypes.c_void_p(0x100000), wsb=1 << 30)
    args.update(kw)
    return lib.pa_attention(args["q"], args["T"], args["k"], args["v"], ctypes.byref(d),
                            args["tables"], args["maxb"], args["ctx"], args["qsl"], args["S"],
                            args["maxctx"], args["maxq"], args["hq"], args["hkv"], args["dim"],
                            args["scale"], args["out"], args["odt"], args["ws"], args["wsb"],
                            None)


@pytest.mark.parametrize("kw,status", [
    (dict(hq=6, hkv=4), 1),                 # not a multiple
    (dict(hq=128, hkv=4), 2),               # group of 32 not built
    (dict(dim=128), 1),                     # disagrees with the descriptor
    (dict(odt=1), 2),                       # fp8 output not built
    (dict(scale=float("nan")), 1),
    (dict(q=None), 1),
    (dict(maxctx=0), 1),
    (dict(wsb=300), 1),                     # workspace too small
    (dict(ws=ctypes.c_void_p(0x100010)), 1),  # workspace not 256-byte aligned
    (dict(S=-1), 1),
    (dict(desc=_desc(cache_dtype=1, head_dim=64)), 2),   # fp8 attention needs head_dim 128
    (dict(q=ctypes.c_void_p(0x100002)), 1),  # q not 16-byte aligned
    (dict(maxq=0), 1),                       # host hints must be positive
    (dict(maxb=0), 1),
    (dict(hkv=0), 1),                        # no kv heads
    (dict(desc=_desc(num_blocks=1 << 26)), 1),  # 2^32 pool rows: beyond the 32-bit row index
    (dict(desc=_desc(num_blocks=1 << 25)), 1),  # 2^31 pool rows: one past the signed index
])
def test_attention_rejects_bad_arguments(lib, kw, status):
    assert _attn(lib, **kw) == status
    assert lib.pa_last_error_string().decode()


def test_attention_with_nothing_to_do_is_ok(lib):
    assert _attn(lib, S=0) == 0
    assert _attn(lib, T=0) == 0
    assert lib.pa_last_error_string().decode() == ""


def test_python_binding_fails_loudly_without_cuda_tensors():
    torch = pytest.importorskip("torch")
    import paged_kv_cache_286_gb300 as pa
    x = torch.zeros(4, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        pa.cache_append(x, x, torch.zeros(4, dtype=torch.int64),
                        torch.zeros(32, 4, 16, 64, dtype=torch.bfloat16),
                        torch.zeros(32, 4, 16, 64, dtype=torch.bfloat16),
                        torch.zeros(256, dtype=torch.uint8))
