"""The Python binding checks tensor shapes before any pointer reaches the
library (which sees only pointers and sizes and cannot check them). Runs on the
CPU: the device check is stubbed and the library is never loaded."""
import pytest
import torch

import paged_kv_cache_252_gb300.api as api


class _Reached(Exception):
    pass


@pytest.fixture
def stub(monkeypatch):
    monkeypatch.setattr(api, "_need_cuda_contig", lambda name, t: None)

    def no_library():
        raise _Reached()
    monkeypatch.setattr(api, "load_library", no_library)


def _case(S=3, n=2, Hq=8, Hkv=2, D=64, nb=10, mbs=4, kv=torch.float16):
    q = torch.zeros(S * n, Hq, D, dtype=torch.float16)
    kc = torch.zeros(nb, Hkv, 16, D, dtype=kv)
    return dict(out=q.clone(), q=q, k_cache=kc, v_cache=kc.clone(),
                block_tables=torch.zeros(S, mbs, dtype=torch.int32),
                context_lens=torch.ones(S, dtype=torch.int32), q_per_seq=n, scale=0.125)


def test_consistent_decode_call_reaches_the_library(stub):
    with pytest.raises(_Reached):
        api.paged_attention_decode(**_case())


@pytest.mark.parametrize("bad", ["q_rows", "out_shape", "head_size", "bt_rows", "v_shape", "ctx_dim"])
def test_inconsistent_decode_call_is_refused(stub, bad):
    c = _case()
    if bad == "q_rows":
        c["q"], c["out"] = c["q"][:5].contiguous(), c["out"][:5].contiguous()
    elif bad == "out_shape":
        c["out"] = torch.zeros(6, 8, 32, dtype=torch.float16)
    elif bad == "head_size":
        c["q"] = torch.zeros(6, 8, 128, dtype=torch.float16)
        c["out"] = c["q"].clone()
    elif bad == "bt_rows":
        c["block_tables"] = torch.zeros(2, 4, dtype=torch.int32)
    elif bad == "v_shape":
        c["v_cache"] = torch.zeros(9, 2, 16, 64, dtype=torch.float16)
    elif bad == "ctx_dim":
        c["context_lens"] = torch.ones(3, 1, dtype=torch.int32)
    with pytest.raises(api.PagedKVError):
        api.paged_attention_decode(**c)
    with pytest.raises(api.PagedKVError):
        api.paged_attention_decode_noalloc(**c)


def test_varlen_and_tree_row_counts(stub):
    c = _case()
    del c["q_per_seq"]
    cu = torch.tensor([0, 1, 3, 4], dtype=torch.int32)
    q = torch.zeros(4, 8, 64, dtype=torch.float16)
    args = dict(c, q=q, out=q.clone())
    with pytest.raises(_Reached):
        api.paged_attention_decode_varlen(cu_q_lens=cu, max_q_per_seq=2, **args)
    big = torch.zeros(7, 8, 64, dtype=torch.float16)        # more rows than 3 sequences x 2
    with pytest.raises(api.PagedKVError):
        api.paged_attention_decode_varlen(cu_q_lens=cu, max_q_per_seq=2, **dict(args, q=big, out=big.clone()))
    with pytest.raises(api.PagedKVError):
        api.paged_attention_decode_varlen(cu_q_lens=cu[:3].contiguous(), max_q_per_seq=2, **args)
    masks = torch.zeros(6, dtype=torch.int64)
    full = torch.zeros(6, 8, 64, dtype=torch.float16)
    with pytest.raises(_Reached):
        api.paged_attention_decode_tree(tree_masks=masks, max_q_per_seq=2, **dict(args, q=full, out=full.clone()))
    with pytest.raises(api.PagedKVError):
        api.paged_attention_decode_tree(tree_masks=masks[:5].contiguous(), max_q_per_seq=2,
                                        **dict(args, q=full, out=full.clone()))
    with pytest.raises(api.PagedKVError):        # without cu_q_lens: exactly num_seqs x max_q_per_seq rows
        api.paged_attention_decode_tree(tree_masks=masks[:4].contiguous(), max_q_per_seq=2, **args)


def test_cache_write_and_int8_shapes(stub):
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.float16)
    key = torch.zeros(5, 2, 64, dtype=torch.float16)
    slots = torch.zeros(5, dtype=torch.int32)
    with pytest.raises(_Reached):
        api.kv_cache_write(key, key.clone(), slots, kc, kc.clone())
    with pytest.raises(api.PagedKVError):
        api.kv_cache_write(key, key.clone(), slots[:4].contiguous(), kc, kc.clone())
    with pytest.raises(api.PagedKVError):
        api.kv_cache_write(torch.zeros(5, 2, 32, dtype=torch.float16), torch.zeros(5, 2, 32, dtype=torch.float16),
                           slots, kc, kc.clone())
    k8 = torch.zeros(4, 2, 16, 64, dtype=torch.int8)
    sc = torch.zeros(4, 2, 2, 16, dtype=torch.float32)
    with pytest.raises(_Reached):
        api.kv_cache_write_int8(key, key.clone(), slots, k8, k8.clone(), sc)
    with pytest.raises(api.PagedKVError):   # the old two-array shape
        api.kv_cache_write_int8(key, key.clone(), slots, k8, k8.clone(), sc[:, :, 0].contiguous())
    c = _case(kv=torch.int8)
    with pytest.raises(api.PagedKVError):   # scales of another pool size
        api.paged_attention_decode_int8(c["out"], c["q"], c["k_cache"], c["v_cache"], sc,
                                        c["block_tables"], c["context_lens"], 2, 0.125)


def test_int8_scales_go_with_an_int8_cache_only():
    """The varlen and tree calls take scales exactly when the cache is INT8 (checked
    before anything reaches the library)."""
    import paged_kv_cache_252_gb300 as pkv
    import pytest as _pt
    q = torch.zeros(2, 4, 64, dtype=torch.float16)
    kc8 = torch.zeros(4, 2, 16, 64, dtype=torch.int8)
    with _pt.raises(pkv.PagedKVError):
        pkv.api._int8_scales(pkv.api.KV_INT8, kc8, None)
    with _pt.raises(pkv.PagedKVError):
        pkv.api._int8_scales(pkv.api.KV_FP16, kc8, torch.zeros(4, 2, 2, 16))
    pkv.api._int8_scales(pkv.api.KV_FP16, kc8, None)


def test_int8_cache_bytes_are_offset_binary_codes():
    """A fresh INT8 cache holds code 0 (byte 0x80); int8_codes reads byte u as u - 128."""
    kc, vc = api.alloc_kv_cache(2, 1, 64, "int8", "cpu")
    assert kc.dtype == torch.int8 and int(kc.view(torch.uint8)[0, 0, 0, 0]) == 0x80
    assert int(api.int8_codes(kc).abs().max()) == 0 and int(api.int8_codes(vc).abs().max()) == 0
    raw = torch.tensor([0x01, 0x7F, 0x80, 0x81, 0xFF], dtype=torch.uint8).view(torch.int8)
    assert api.int8_codes(raw).tolist() == [-127, -1, 0, 1, 127]
    with pytest.raises(api.PagedKVError):
        api.int8_codes(torch.zeros(4, dtype=torch.uint8))
    e, _ = api.alloc_kv_cache(2, 1, 64, "e5m2", "cpu")
    assert e.dtype == torch.uint8 and int(e.max()) == 0


def _chunked_case(q_lens=(1, 40, 3), ctx=(5, 60, 3), Hq=8, Hkv=2, D=64, nb=10, mbs=4):
    rows = sum(q_lens)
    q = torch.zeros(rows, Hq, D, dtype=torch.float16)
    kc = torch.zeros(nb, Hkv, 16, D, dtype=torch.float16)
    return dict(out=q.clone(), q=q, q_lens=list(q_lens), context_lens=torch.tensor(ctx, dtype=torch.int32),
                k_cache=kc, v_cache=kc.clone(), block_tables=torch.zeros(len(q_lens), mbs, dtype=torch.int32),
                scale=0.125)


def test_chunked_call_reaches_the_library_and_checks_its_host_arrays(stub):
    with pytest.raises(_Reached):
        api.paged_attention_decode_chunked(**_chunked_case())
    for bad in ("rows", "ctx_short", "zero_tokens", "ctx_len", "bt_rows"):
        c = _chunked_case()
        if bad == "rows":
            c["q"], c["out"] = c["q"][:40].contiguous(), c["out"][:40].contiguous()
        elif bad == "ctx_short":
            c["context_lens"] = torch.tensor([5, 39, 3], dtype=torch.int32)
        elif bad == "zero_tokens":
            c["q_lens"] = [1, 0, 3]
        elif bad == "ctx_len":
            c["context_lens"] = torch.tensor([5, 60], dtype=torch.int32)
        elif bad == "bt_rows":
            c["block_tables"] = torch.zeros(2, 4, dtype=torch.int32)
        with pytest.raises(api.PagedKVError):
            api.paged_attention_decode_chunked(**c)
