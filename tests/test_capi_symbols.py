"""The C-ABI library loads without a GPU and exports every function that
include/pagedkv.h declares; host-side argument checks reject bad calls before
anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(pkv_\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__  # noqa: F401  (puts the repo on sys.path)
    from paged_kv_cache_252_gb300 import build
    build.build()
    return ctypes.CDLL(build.LIB)


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["pkv_kv_cache_write", "pkv_paged_attention_decode", "pkv_decode_workspace_bytes",
              "pkv_error_string", "pkv_version"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_error_strings_and_version(lib):
    lib.pkv_error_string.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert lib.pkv_error_string(code)
    assert lib.pkv_version() >= 100


def test_host_validation_rejects_bad_arguments_without_a_device(lib):
    from paged_kv_cache_252_gb300.api import _CacheDesc
    vp = ctypes.c_void_p
    good = _CacheDesc(32, 16, 2, 64)
    bad_block = _CacheDesc(32, 8, 2, 64)
    bad_head = _CacheDesc(32, 16, 2, 96)
    fake = vp(0x1000)
    w = lib.pkv_kv_cache_write
    w.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int32, vp, vp, vp, ctypes.c_int,
                  ctypes.POINTER(_CacheDesc), vp, vp]
    assert w(fake, fake, 0, 4, fake, fake, fake, 0, ctypes.byref(bad_block), None, None) == -1
    assert w(fake, fake, 0, 4, fake, fake, fake, 0, ctypes.byref(bad_head), None, None) == -1
    assert w(fake, fake, 0, 4, fake, fake, fake, 0, None, None, None) == -1
    assert w(fake, fake, 1, 4, fake, fake, fake, 2, ctypes.byref(good), None, None) == -2  # bf16 -> fp8
    assert w(fake, fake, 0, -1, fake, fake, fake, 0, ctypes.byref(good), None, None) == -1
    assert w(None, fake, 0, 4, fake, fake, fake, 0, ctypes.byref(good), None, None) == -1
    assert w(vp(0x1001), fake, 0, 4, fake, fake, fake, 0, ctypes.byref(good), None, None) == -1
    assert w(None, None, 0, 0, None, None, None, 0, ctypes.byref(good), None, None) == 0  # no-op
    d = lib.pkv_paged_attention_decode
    d.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp, ctypes.c_int,
                  ctypes.POINTER(_CacheDesc), vp, ctypes.c_int32, vp, ctypes.c_float, vp,
                  ctypes.c_size_t, vp, vp]
    args = [fake, fake, 4, 4, 1, fake, fake, 0, ctypes.byref(good), fake, 4, fake, 0.125, fake,
            1 << 20, None, None]
    a = list(args); a[3] = 3                       # 3 q heads over 2 KV heads
    assert d(*a) == -1
    a = list(args); a[3] = 2 * 65                  # group x tokens > 64
    assert d(*a) == -2
    a = list(args); a[7] = 5                       # unknown dtype
    assert d(*a) == -2
    a = list(args); a[4] = 0                       # q_per_seq 0
    assert d(*a) == -1
    a = list(args); a[0] = None
    assert d(*a) == -1
    a = list(args); a[2] = 0                       # empty batch: no-op
    assert d(*a) == 0


def test_chunked_call_checks_its_host_arrays_without_a_device(lib):
    """The chunked entry point reads the query counts and lengths from host memory and
    rejects an empty sequence or a context shorter than its query tokens before any
    device work."""
    from paged_kv_cache_252_gb300.api import _CacheDesc
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    good = _CacheDesc(32, 16, 2, 64)
    fake = vp(0x1000)
    c = lib.pkv_paged_attention_decode_chunked
    c.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, ctypes.c_int, ctypes.POINTER(_CacheDesc), vp, i32,
                  ctypes.c_float, vp, ctypes.c_size_t, vp, vp]

    def call(q_lens, ctx, heads=4, mbs=8):
        ql = (i32 * len(q_lens))(*q_lens)
        cl = (i32 * len(ctx))(*ctx)
        return c(fake, fake, ctypes.cast(ql, vp), ctypes.cast(cl, vp), len(q_lens), heads, fake, fake, None, 0,
                 ctypes.byref(good), fake, mbs, 0.125, vp(0x10000), 1 << 20, None, None)

    assert call([1, 0, 3], [4, 4, 4]) == -1            # a sequence without query tokens
    assert call([1, 5, 3], [4, 4, 4]) == -1            # context shorter than its tokens
    assert call([1, 2], [4, 4], heads=3) == -1         # 3 query heads over 2 KV heads
    assert call([1, 2], [4, 4], mbs=0) == -1
    assert c(fake, fake, None, None, 0, 4, fake, fake, None, 0, ctypes.byref(good), fake, 8, 0.125, None, 0,
             None, None) == 0                           # empty batch: no-op
    ws = lib.pkv_decode_chunked_workspace_bytes
    ws.argtypes = [vp, i32, i32, i32, ctypes.POINTER(_CacheDesc)]
    ws.restype = ctypes.c_size_t
    bad = (i32 * 2)(1, 0)
    assert ws(ctypes.cast(bad, vp), 2, 4, 8, ctypes.byref(good)) == 0


def test_bounded_wait_selftest_checks_its_arguments_without_a_device(lib):
    vp = ctypes.c_void_p
    f = lib.pkv_selftest_bounded_wait
    f.argtypes = [vp, ctypes.c_uint64, vp, vp]
    assert f(None, 1000, vp(0x1000), None) == -1
    assert f(vp(0x1000), 1000, None, None) == -1
    assert f(vp(0x1002), 1000, vp(0x1000), None) == -1     # misaligned status word
    assert f(vp(0x1000), 0, vp(0x1000), None) == -1        # no limit
    assert f(vp(0x1000), 3_000_000_000, vp(0x1000), None) == -1
