"""The allocation-free decode entry point (for callers that cannot allocate
device memory when they run attention: its scratch is a buffer built into the
library). Called through the C ABI, its output must match the regular entry
point's within the tolerance the parity tests use, on two calls in a row (the
second call reuses the shared buffer with the first call's contents in it).

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_252_gb300 import workloads as wl

import _gpu

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _noalloc_call(lib, out, q, kc, vc, kv_code, desc, bt, cl, n, scale, status):
    fn = lib.pkv_paged_attention_decode_noalloc
    vp = ctypes.c_void_p
    return fn(vp(out.data_ptr()), vp(q.data_ptr()), int(cl.shape[0]), int(q.shape[1]), int(n),
              vp(kc.data_ptr()), vp(vc.data_ptr()), kv_code, ctypes.byref(desc), vp(bt.data_ptr()),
              int(bt.shape[1]), vp(cl.data_ptr()), ctypes.c_float(scale), vp(status.data_ptr()),
              vp(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("key", ["8b", "70b_spec"])
def test_noalloc_matches_regular_entry_point_twice(dev, key):
    import paged_kv_cache_252_gb300 as pkv
    from paged_kv_cache_252_gb300.api import _CacheDesc, load_library
    lib = load_library()
    w = wl.reduced(wl.by_name(key), num_seqs=16)
    vals = wl.token_values(w, device=dev)
    kc, vc = pkv.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, w.kv_dtype, dev)
    pkv.kv_cache_write(vals["k_all"], vals["v_all"], vals["slot_all"], kc, vc)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    q = vals["q"]
    ref = torch.empty_like(q)
    pkv.paged_attention_decode(ref, q, kc, vc, bt, cl, w.q_per_seq, w.scale)
    desc = _CacheDesc(w.num_blocks, 16, w.num_kv_heads, w.head_size)
    kv_code = {"fp16": 0, "bf16": 1, "e5m2": 2}[w.kv_dtype]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _noalloc_call(lib, out, q, kc, vc, kv_code, desc, bt, cl, w.q_per_seq, w.scale, status)
        assert rc == 0, rc
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        r = ref.float().cpu().numpy().astype(np.float64)
        _gpu.compare(out, r, label=f"no-alloc {key} call {call}")


def test_noalloc_rejects_problems_beyond_its_buffer(dev):
    from paged_kv_cache_252_gb300.api import _CacheDesc, load_library
    lib = load_library()
    limit = 32 << 20
    desc = _CacheDesc(1024, 16, 8, 128)
    # 64 rows per unit and enough sequences that the split-KV scratch exceeds the buffer
    S = 4096
    need = lib.pkv_decode_workspace_bytes(S, 64, 8, ctypes.byref(desc))
    assert need > limit
    fake = ctypes.c_void_p(256)
    rc = lib.pkv_paged_attention_decode_noalloc(fake, fake, S, 64, 8, fake, fake, 0, ctypes.byref(desc),
                                                fake, 4, fake, ctypes.c_float(0.1), None, None)
    assert rc == -3   # PKV_ERR_WORKSPACE_TOO_SMALL, nothing launched


@pytest.mark.parametrize("case", ["rows_over_64", "heads_not_divisible", "bad_head_size"])
def test_noalloc_refused_shapes_get_the_regular_status(dev, case):
    """A shape the library refuses gets the same status from the no-alloc entry
    point as from the regular one (nothing is launched by either)."""
    from paged_kv_cache_252_gb300.api import _CacheDesc, load_library
    lib = load_library()
    Hq, Hkv, D, n = {"rows_over_64": (128, 1, 128, 1), "heads_not_divisible": (12, 8, 128, 1),
                     "bad_head_size": (8, 2, 96, 1)}[case]
    desc = _CacheDesc(64, 16, Hkv, D)
    fake = ctypes.c_void_p(256)
    ws = ctypes.c_void_p(1 << 20)
    reg = lib.pkv_paged_attention_decode(fake, fake, 4, Hq, n, fake, fake, 0, ctypes.byref(desc), fake, 4,
                                         fake, ctypes.c_float(0.1), ws, ctypes.c_size_t(1 << 30), None, None)
    na = lib.pkv_paged_attention_decode_noalloc(fake, fake, 4, Hq, n, fake, fake, 0, ctypes.byref(desc),
                                                fake, 4, fake, ctypes.c_float(0.1), None, None)
    assert reg < 0 and na == reg, (reg, na)
