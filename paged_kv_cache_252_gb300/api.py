"""Python binding of libpagedkv.so: argument marshalling only.

Every function here turns torch tensors into device pointers and sizes and
calls the C ABI declared in ``include/pagedkv.h``; the computation happens in
the library's CUDA kernels. There is no fallback: if the library is missing or
a call fails, a :class:`PagedKVError` is raised.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import numpy as np
import torch

KV_FP16, KV_BF16, KV_E5M2, KV_INT8 = 0, 1, 2, 3
_NAMES = {"fp16": KV_FP16, "bf16": KV_BF16, "e5m2": KV_E5M2, "fp8_e5m2": KV_E5M2, "int8": KV_INT8}
_TORCH = {torch.float16: KV_FP16, torch.bfloat16: KV_BF16, torch.uint8: KV_E5M2,
          torch.float8_e5m2: KV_E5M2, torch.int8: KV_INT8}
BLOCK_SIZE = 16

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None
_workspaces: dict = {}
_ws_bytes_cache: dict = {}


class PagedKVError(RuntimeError):
    pass


class _CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_size", ctypes.c_int32)]


def library_path() -> str:
    return os.path.join(_HERE, "libpagedkv.so")


def load_library(path: str | None = None):
    """Load libpagedkv.so (built in-tree by ``__graft_entry__.build()``). A profiling
    tool may pass the path of a variant build of the same library instead; the
    first load wins for the rest of the process."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or library_path()
        if not os.path.exists(path):
            raise PagedKVError(f"{path} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, i32, P = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER
        lib.pkv_kv_cache_write.argtypes = [vp, vp, ctypes.c_int, i32, vp, vp, vp, ctypes.c_int,
                                           P(_CacheDesc), vp, vp]
        lib.pkv_kv_cache_write.restype = ctypes.c_int
        lib.pkv_decode_workspace_bytes.argtypes = [i32, i32, i32, P(_CacheDesc)]
        lib.pkv_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.pkv_paged_attention_decode.argtypes = [
            vp, vp, i32, i32, i32, vp, vp, ctypes.c_int, P(_CacheDesc), vp, i32, vp,
            ctypes.c_float, vp, ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode.restype = ctypes.c_int
        lib.pkv_paged_attention_decode_varlen.argtypes = [
            vp, vp, vp, i32, i32, i32, i32, vp, vp, ctypes.c_int, P(_CacheDesc), vp, i32, vp,
            ctypes.c_float, vp, ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode_varlen.restype = ctypes.c_int
        lib.pkv_paged_attention_decode_tree.argtypes = [
            vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, ctypes.c_int, P(_CacheDesc), vp, i32, vp,
            ctypes.c_float, vp, ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode_tree.restype = ctypes.c_int
        lib.pkv_paged_attention_decode_noalloc.argtypes = [
            vp, vp, i32, i32, i32, vp, vp, ctypes.c_int, P(_CacheDesc), vp, i32, vp,
            ctypes.c_float, vp, vp]
        lib.pkv_paged_attention_decode_noalloc.restype = ctypes.c_int
        i64 = ctypes.c_int64
        lib.pkv_allocator_create.argtypes = [i32]
        lib.pkv_allocator_create.restype = vp
        lib.pkv_allocator_destroy.argtypes = [vp]
        lib.pkv_allocator_destroy.restype = None
        for fn in ("pkv_allocator_free_blocks", "pkv_allocator_evictable"):
            getattr(lib, fn).argtypes = [vp]
            getattr(lib, fn).restype = i32
        lib.pkv_allocator_refcount.argtypes = [vp, i32]
        lib.pkv_allocator_refcount.restype = i32
        lib.pkv_seq_add.argtypes = [vp, i64]
        lib.pkv_seq_add.restype = ctypes.c_int
        lib.pkv_seq_fork.argtypes = [vp, i64, i64]
        lib.pkv_seq_fork.restype = ctypes.c_int
        lib.pkv_seq_release.argtypes = [vp, i64]
        lib.pkv_seq_release.restype = ctypes.c_int
        lib.pkv_seq_length.argtypes = [vp, i64]
        lib.pkv_seq_length.restype = i32
        lib.pkv_seq_block_table.argtypes = [vp, i64, vp, i32]
        lib.pkv_seq_block_table.restype = i32
        lib.pkv_seq_append.argtypes = [vp, i64, i32, vp, vp, vp, vp]
        lib.pkv_seq_append.restype = ctypes.c_int
        lib.pkv_prefix_insert.argtypes = [vp, i64, vp, i32]
        lib.pkv_prefix_insert.restype = i32
        lib.pkv_seq_add_cached.argtypes = [vp, i64, vp, i32, vp]
        lib.pkv_seq_add_cached.restype = ctypes.c_int
        lib.pkv_copy_blocks.argtypes = [vp, vp, vp, ctypes.c_int, P(_CacheDesc), vp, vp, i32, vp, vp]
        lib.pkv_copy_blocks.restype = ctypes.c_int
        lib.pkv_kv_cache_write_int8.argtypes = [vp, vp, i32, vp, vp, vp, vp, P(_CacheDesc), vp, vp]
        lib.pkv_kv_cache_write_int8.restype = ctypes.c_int
        lib.pkv_paged_attention_decode_int8.argtypes = [
            vp, vp, i32, i32, i32, vp, vp, vp, P(_CacheDesc), vp, i32, vp, ctypes.c_float, vp,
            ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode_int8.restype = ctypes.c_int
        lib.pkv_paged_attention_decode_int8_varlen.argtypes = [
            vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, P(_CacheDesc), vp, i32, vp, ctypes.c_float, vp,
            ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode_int8_varlen.restype = ctypes.c_int
        lib.pkv_paged_attention_decode_int8_tree.argtypes = [
            vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, P(_CacheDesc), vp, i32, vp, ctypes.c_float, vp,
            ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode_int8_tree.restype = ctypes.c_int
        lib.pkv_decode_chunked_workspace_bytes.argtypes = [vp, i32, i32, i32, P(_CacheDesc)]
        lib.pkv_decode_chunked_workspace_bytes.restype = ctypes.c_size_t
        lib.pkv_paged_attention_decode_chunked.argtypes = [
            vp, vp, vp, vp, i32, i32, vp, vp, vp, ctypes.c_int, P(_CacheDesc), vp, i32, ctypes.c_float, vp,
            ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode_chunked.restype = ctypes.c_int
        lib.pkv_selftest_bounded_wait.argtypes = [vp, ctypes.c_uint64, vp, vp]
        lib.pkv_selftest_bounded_wait.restype = ctypes.c_int
        lib.pkv_error_string.argtypes = [ctypes.c_int]
        lib.pkv_error_string.restype = ctypes.c_char_p
        lib.pkv_version.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load_library().pkv_error_string(rc).decode()
        raise PagedKVError(f"{what} failed: {msg} ({rc})")


def _kv_code(kv_dtype, cache: torch.Tensor) -> int:
    if kv_dtype is None:
        return _TORCH[cache.dtype]
    if isinstance(kv_dtype, str):
        return _NAMES[kv_dtype]
    if isinstance(kv_dtype, torch.dtype):
        return _TORCH[kv_dtype]
    return int(kv_dtype)


def _src_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return KV_FP16
    if t.dtype == torch.bfloat16:
        return KV_BF16
    raise PagedKVError(f"unsupported key/value/query dtype {t.dtype}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _desc(cache: torch.Tensor) -> _CacheDesc:
    if cache.dim() != 4 or cache.shape[2] != BLOCK_SIZE:
        raise PagedKVError(f"cache must be [num_blocks, num_kv_heads, 16, head_size], got {tuple(cache.shape)}")
    return _CacheDesc(cache.shape[0], cache.shape[2], cache.shape[1], cache.shape[3])


def _pair(k_cache, v_cache) -> _CacheDesc:
    d = _desc(k_cache)
    if tuple(v_cache.shape) != tuple(k_cache.shape) or v_cache.dtype != k_cache.dtype:
        raise PagedKVError("k_cache and v_cache must have the same shape and dtype")
    return d


def _decode_shapes(out, q, k_cache, v_cache, block_tables, context_lens, rows=None, max_rows=None):
    """The library sees only pointers: check here that every tensor is as large as
    the call will read or write. Returns (cache descriptor, num_seqs)."""
    d = _pair(k_cache, v_cache)
    if q.dim() != 3 or tuple(out.shape) != tuple(q.shape):
        raise PagedKVError(f"q and out must both be [rows, num_q_heads, head_size], got "
                           f"{tuple(q.shape)} and {tuple(out.shape)}")
    if int(q.shape[2]) != int(k_cache.shape[3]):
        raise PagedKVError(f"query head size {int(q.shape[2])} != cache head size {int(k_cache.shape[3])}")
    if context_lens.dim() != 1:
        raise PagedKVError("context_lens must be 1-D [num_seqs]")
    S = int(context_lens.shape[0])
    if block_tables.dim() != 2 or int(block_tables.shape[0]) < S:
        raise PagedKVError(f"block_tables must be [num_seqs, max_blocks_per_seq], got {tuple(block_tables.shape)}")
    if rows is not None and int(q.shape[0]) != rows:
        raise PagedKVError(f"q must have num_seqs * q_per_seq = {rows} rows, got {int(q.shape[0])}")
    if max_rows is not None and not (S <= int(q.shape[0]) <= max_rows):
        raise PagedKVError(f"q must have between num_seqs and num_seqs * max_q_per_seq rows, got {int(q.shape[0])}")
    return d, S


def _scales_shape(k_cache, scales):
    want = (int(k_cache.shape[0]), int(k_cache.shape[1]), 2, BLOCK_SIZE)
    if tuple(scales.shape) != want or scales.dtype != torch.float32:
        raise PagedKVError(f"scales must be float32 {want} (K then V row scales)")


def _write_shapes(key, value, slot_mapping, k_cache, v_cache) -> _CacheDesc:
    d = _pair(k_cache, v_cache)
    want = (int(k_cache.shape[1]), int(k_cache.shape[3]))
    if key.dim() != 3 or tuple(value.shape) != tuple(key.shape) or tuple(key.shape[1:]) != want:
        raise PagedKVError(f"key and value must both be [T, {want[0]}, {want[1]}], got "
                           f"{tuple(key.shape)} and {tuple(value.shape)}")
    if slot_mapping.dim() != 1 or int(slot_mapping.shape[0]) != int(key.shape[0]):
        raise PagedKVError("slot_mapping must be 1-D with one slot per token")
    return d


def _need_cuda_contig(name, t):
    if not t.is_cuda:
        raise PagedKVError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PagedKVError(f"{name} must be contiguous")


def alloc_kv_cache(num_blocks: int, num_kv_heads: int, head_size: int, kv_dtype,
                   device="cuda", zero: bool = True):
    """Allocate a K/V cache pair [num_blocks, num_kv_heads, 16, head_size]. An INT8
    cache is a torch.int8 tensor whose bytes hold the codes in offset binary
    (byte = code + 128; :func:`int8_codes` reads them back). ``zero`` fills the
    caches with the value 0 (for INT8: code 0, byte 0x80)."""
    code = _NAMES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    dt = {KV_FP16: torch.float16, KV_BF16: torch.bfloat16, KV_E5M2: torch.uint8, KV_INT8: torch.int8}[code]
    shape = (num_blocks, num_kv_heads, BLOCK_SIZE, head_size)
    if not zero:
        return torch.empty(shape, dtype=dt, device=device), torch.empty(shape, dtype=dt, device=device)
    fill = -128 if code == KV_INT8 else 0   # int8 -128 is the byte 0x80
    return (torch.full(shape, fill, dtype=dt, device=device), torch.full(shape, fill, dtype=dt, device=device))


def alloc_kv_scales(num_blocks: int, num_kv_heads: int, device="cuda"):
    """Row scales of an INT8 cache pair: one float32 tensor [num_blocks, num_kv_heads, 2, 16],
    [..., 0, t] the K scale and [..., 1, t] the V scale of token t of a block."""
    return torch.zeros((num_blocks, num_kv_heads, 2, BLOCK_SIZE), dtype=torch.float32, device=device)


def int8_codes(cache: torch.Tensor) -> torch.Tensor:
    """The signed codes of an INT8 cache, whose bytes are stored in offset binary
    (byte = code + 128): a torch.int8 tensor of the same shape and device."""
    if cache.dtype != torch.int8:
        raise PagedKVError("int8_codes reads an INT8 cache (torch.int8)")
    return (cache.view(torch.uint8).to(torch.int16) - 128).to(torch.int8)


def kv_cache_write_int8(key, value, slot_mapping, k_cache, v_cache, scales, *,
                        device_status=None, stream=None):
    """Quantise fp16 key/value [T, Hkv, D] into INT8 caches (codes in offset binary,
    byte = code + 128) and their row scales."""
    for n, t in (("key", key), ("value", value), ("slot_mapping", slot_mapping), ("k_cache", k_cache),
                 ("v_cache", v_cache), ("scales", scales)):
        _need_cuda_contig(n, t)
    if key.dtype != torch.float16 or k_cache.dtype != torch.int8 or scales.dtype != torch.float32:
        raise PagedKVError("INT8 cache write takes fp16 key/value, int8 caches, float32 scales")
    if slot_mapping.dtype != torch.int32:
        raise PagedKVError("slot_mapping must be int32")
    d = _write_shapes(key, value, slot_mapping, k_cache, v_cache)
    _scales_shape(k_cache, scales)
    rc = load_library().pkv_kv_cache_write_int8(
        _ptr(key), _ptr(value), int(key.shape[0]), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        _ptr(scales), ctypes.byref(d), _ptr(device_status), _stream_handle(stream, key.device))
    _check(rc, "kv_cache_write_int8")


def paged_attention_decode_int8(out, q, k_cache, v_cache, scales, block_tables, context_lens,
                                q_per_seq: int, scale: float, *, workspace=None, device_status=None,
                                stream=None):
    """paged_attention_decode over an INT8 cache with its row scales (q/out fp16)."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("scales", scales),
                 ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(n, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PagedKVError("block_tables and context_lens must be int32")
    d, S = _decode_shapes(out, q, k_cache, v_cache, block_tables, context_lens,
                          rows=int(context_lens.shape[0]) * int(q_per_seq))
    _scales_shape(k_cache, scales)
    Hq = int(q.shape[1])
    lib = load_library()
    with _on_device(q.device):
        need = _ws_bytes(lib, q.device, S, Hq, int(q_per_seq), d)
        if workspace is None:
            workspace = _workspace(need, q.device)
        rc = lib.pkv_paged_attention_decode_int8(
            _ptr(out), _ptr(q), S, Hq, int(q_per_seq), _ptr(k_cache), _ptr(v_cache), _ptr(scales),
            ctypes.byref(d), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
            float(scale), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
            _ptr(device_status), _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode_int8")
    return out


def kv_cache_write(key, value, slot_mapping, k_cache, v_cache, kv_dtype=None, *,
                   device_status=None, stream=None):
    """Scatter key/value [T, Hkv, D] into their cache slots (fp16->E5M2 cast for an E5M2 cache)."""
    for n, t in (("key", key), ("value", value), ("slot_mapping", slot_mapping),
                 ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda_contig(n, t)
    if slot_mapping.dtype != torch.int32:
        raise PagedKVError("slot_mapping must be int32")
    d = _write_shapes(key, value, slot_mapping, k_cache, v_cache)
    rc = load_library().pkv_kv_cache_write(
        _ptr(key), _ptr(value), _src_code(key), int(key.shape[0]), _ptr(slot_mapping),
        _ptr(k_cache), _ptr(v_cache), _kv_code(kv_dtype, k_cache), ctypes.byref(d),
        _ptr(device_status), _stream_handle(stream, key.device))
    _check(rc, "kv_cache_write")


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, q_per_seq: int, k_cache) -> int:
    d = _desc(k_cache)
    with torch.cuda.device(k_cache.device):
        return int(load_library().pkv_decode_workspace_bytes(num_seqs, num_q_heads, q_per_seq,
                                                             ctypes.byref(d)))


def _on_device(device):
    """The device context for a call, entered only when the tensors are not on the current device."""
    if device.index is None or device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _ws_bytes(lib, device, S, Hq, n, d) -> int:
    """pkv_decode_workspace_bytes, remembered per device and problem shape."""
    key = (device.index, S, Hq, n, d.num_blocks, d.block_size, d.num_kv_heads, d.head_size)
    v = _ws_bytes_cache.get(key)
    if v is None:
        v = int(lib.pkv_decode_workspace_bytes(S, Hq, n, ctypes.byref(d)))
        _ws_bytes_cache[key] = v
    return v


def _workspace(nbytes: int, device) -> torch.Tensor:
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        # Zeroed once: the piece counters then start clear whatever the allocator
        # held there before (later calls leave them clear).
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, q_per_seq: int,
                           scale: float, kv_dtype=None, *, workspace=None, device_status=None,
                           stream=None):
    """out[s*n+j, hq] = softmax(scale * q K^T) V over sequence s's blocks (causal among its
    n = q_per_seq query tokens). q/out: [S*n, Hq, D]; caches [NB, Hkv, 16, D]."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(n, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PagedKVError("block_tables and context_lens must be int32")
    if out.dtype != q.dtype:
        raise PagedKVError("out and q must share a dtype")
    d, S = _decode_shapes(out, q, k_cache, v_cache, block_tables, context_lens,
                          rows=int(context_lens.shape[0]) * int(q_per_seq))
    Hq = int(q.shape[1])
    code = _kv_code(kv_dtype, k_cache)
    lib = load_library()
    with _on_device(q.device):
        need = _ws_bytes(lib, q.device, S, Hq, int(q_per_seq), d)
        if workspace is None:
            workspace = _workspace(need, q.device)
        rc = lib.pkv_paged_attention_decode(
            _ptr(out), _ptr(q), S, Hq, int(q_per_seq), _ptr(k_cache), _ptr(v_cache), code,
            ctypes.byref(d), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
            float(scale), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
            _ptr(device_status), _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode")
    return out


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                   q_per_seq: int, scale: float, kv_dtype=None, *,
                                   device_status=None, stream=None):
    """Same as :func:`paged_attention_decode`, but the split-KV scratch comes from a
    fixed buffer inside the library, so neither this call nor the library allocates
    device memory (for callers that cannot allocate at this point). Problems too
    large for that buffer raise PagedKVError ("workspace too small"). Calls that
    overlap on the GPU share the buffer and must be serialised."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(n, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PagedKVError("block_tables and context_lens must be int32")
    if out.dtype != q.dtype:
        raise PagedKVError("out and q must share a dtype")
    d, _ = _decode_shapes(out, q, k_cache, v_cache, block_tables, context_lens,
                          rows=int(context_lens.shape[0]) * int(q_per_seq))
    with _on_device(q.device):
        rc = load_library().pkv_paged_attention_decode_noalloc(
            _ptr(out), _ptr(q), int(context_lens.shape[0]), int(q.shape[1]), int(q_per_seq),
            _ptr(k_cache), _ptr(v_cache), _kv_code(kv_dtype, k_cache), ctypes.byref(d),
            _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(scale),
            _ptr(device_status), _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode_noalloc")
    return out


def _int8_scales(code, k_cache, scales):
    """An INT8 cache is read with its row scales; other caches take none."""
    if (code == KV_INT8) != (scales is not None):
        raise PagedKVError("an INT8 cache is read with its scales (alloc_kv_scales); other caches take none")
    if scales is not None:
        _need_cuda_contig("scales", scales)
        _scales_shape(k_cache, scales)


def paged_attention_decode_varlen(out, q, cu_q_lens, k_cache, v_cache, block_tables, context_lens,
                                  max_q_per_seq: int, scale: float, kv_dtype=None, *, scales=None,
                                  workspace=None, device_status=None, stream=None):
    """Decode attention for a batch whose sequences carry different numbers of query
    tokens, packed without padding: sequence s owns rows cu_q_lens[s]..cu_q_lens[s+1]-1
    of q/out ([total_rows, Hq, D]), 1 <= n_s <= max_q_per_seq, causal among its tokens.
    An INT8 cache takes its row scales (``scales``)."""
    for nm, t in (("out", out), ("q", q), ("cu_q_lens", cu_q_lens), ("k_cache", k_cache),
                  ("v_cache", v_cache), ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(nm, t)
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32
            or cu_q_lens.dtype != torch.int32):
        raise PagedKVError("block_tables, context_lens and cu_q_lens must be int32")
    if out.dtype != q.dtype:
        raise PagedKVError("out and q must share a dtype")
    d, S = _decode_shapes(out, q, k_cache, v_cache, block_tables, context_lens,
                          max_rows=int(context_lens.shape[0]) * int(max_q_per_seq))
    if cu_q_lens.dim() != 1 or int(cu_q_lens.shape[0]) != S + 1:
        raise PagedKVError("cu_q_lens must have num_seqs + 1 entries")
    code = _kv_code(kv_dtype, k_cache)
    _int8_scales(code, k_cache, scales)
    Hq = int(q.shape[1])
    lib = load_library()
    with _on_device(q.device):
        need = _ws_bytes(lib, q.device, S, Hq, int(max_q_per_seq), d)
        if workspace is None:
            workspace = _workspace(need, q.device)
        ws = (_ptr(workspace), int(workspace.numel() * workspace.element_size()))
        if code == KV_INT8:
            rc = lib.pkv_paged_attention_decode_int8_varlen(
                _ptr(out), _ptr(q), _ptr(cu_q_lens), int(q.shape[0]), S, Hq, int(max_q_per_seq),
                _ptr(k_cache), _ptr(v_cache), _ptr(scales), ctypes.byref(d), _ptr(block_tables),
                int(block_tables.shape[1]), _ptr(context_lens), float(scale), *ws, _ptr(device_status),
                _stream_handle(stream, q.device))
        else:
            rc = lib.pkv_paged_attention_decode_varlen(
                _ptr(out), _ptr(q), _ptr(cu_q_lens), int(q.shape[0]), S, Hq, int(max_q_per_seq),
                _ptr(k_cache), _ptr(v_cache), code, ctypes.byref(d), _ptr(block_tables),
                int(block_tables.shape[1]), _ptr(context_lens), float(scale), *ws, _ptr(device_status),
                _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode_varlen")
    return out


def _host_i32(name, x, n=None) -> np.ndarray:
    """A host int32 array (list, numpy array or CPU tensor) the library reads directly."""
    if isinstance(x, torch.Tensor):
        if x.is_cuda:
            raise PagedKVError(f"{name} must be in host memory")
        x = x.numpy()
    a = np.ascontiguousarray(np.asarray(x), dtype=np.int32)
    if a.ndim != 1 or (n is not None and a.shape[0] != n):
        raise PagedKVError(f"{name} must be 1-D" + (f" with {n} entries" if n is not None else ""))
    return a


def paged_attention_decode_chunked(out, q, q_lens, context_lens, k_cache, v_cache, block_tables, scale: float,
                                   kv_dtype=None, *, scales=None, workspace=None, device_status=None,
                                   stream=None):
    """Decode attention for a batch whose sequences carry any number of query tokens
    (prefill chunks beside decode / verify tokens), packed without padding: sequence s
    owns the next q_lens[s] rows of q/out and its token j sees positions
    <= context_lens[s] - q_lens[s] + j. q_lens and context_lens are host arrays
    (lists, numpy arrays or CPU tensors), read when the call is made (a captured CUDA
    graph replays them)."""
    for nm, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                  ("block_tables", block_tables)):
        _need_cuda_contig(nm, t)
    if block_tables.dtype != torch.int32:
        raise PagedKVError("block_tables must be int32")
    if out.dtype != q.dtype:
        raise PagedKVError("out and q must share a dtype")
    ql = _host_i32("q_lens", q_lens)
    S = int(ql.shape[0])
    cl = _host_i32("context_lens", context_lens, S)
    if S and (ql.min() < 1 or np.any(cl < ql)):
        raise PagedKVError("every sequence needs 1 <= q_lens[s] <= context_lens[s]")
    d = _pair(k_cache, v_cache)
    if q.dim() != 3 or tuple(out.shape) != tuple(q.shape) or int(q.shape[0]) != int(ql.sum()):
        raise PagedKVError(f"q and out must both be [sum(q_lens) = {int(ql.sum())}, num_q_heads, head_size]")
    if int(q.shape[2]) != int(k_cache.shape[3]):
        raise PagedKVError(f"query head size {int(q.shape[2])} != cache head size {int(k_cache.shape[3])}")
    if block_tables.dim() != 2 or int(block_tables.shape[0]) < S:
        raise PagedKVError(f"block_tables must be [num_seqs, max_blocks_per_seq], got {tuple(block_tables.shape)}")
    code = _kv_code(kv_dtype, k_cache)
    _int8_scales(code, k_cache, scales)
    Hq, mbs = int(q.shape[1]), int(block_tables.shape[1])
    lib = load_library()
    qp, cp = ql.ctypes.data_as(ctypes.c_void_p), cl.ctypes.data_as(ctypes.c_void_p)
    with _on_device(q.device):
        need = int(lib.pkv_decode_chunked_workspace_bytes(qp, S, Hq, mbs, ctypes.byref(d)))
        if S and need == 0:
            raise PagedKVError("paged_attention_decode_chunked: unsupported shape")
        if workspace is None:
            workspace = _workspace(need, q.device)
        rc = lib.pkv_paged_attention_decode_chunked(
            _ptr(out), _ptr(q), qp, cp, S, Hq, _ptr(k_cache), _ptr(v_cache), _ptr(scales), code,
            ctypes.byref(d), _ptr(block_tables), mbs, float(scale), _ptr(workspace),
            int(workspace.numel() * workspace.element_size()), _ptr(device_status),
            _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode_chunked")
    return out


def selftest_bounded_wait(limit_ns: int, device=None, stream=None):
    """Run the device self-test of the decode kernels' bounded waits (a wait on a
    barrier phase nothing completes gives up after limit_ns and flags
    PKV_DEV_TIMEOUT; a second wait leaves on the CTA's abort flag). Returns
    (status word, [duration of wait 0, duration of wait 1] in ns)."""
    device = torch.device(device or "cuda")
    status = torch.zeros(1, dtype=torch.int32, device=device)
    elapsed = torch.zeros(2, dtype=torch.int64, device=device)
    lib = load_library()
    with _on_device(status.device):
        rc = lib.pkv_selftest_bounded_wait(_ptr(status), int(limit_ns), _ptr(elapsed),
                                           _stream_handle(stream, status.device))
    _check(rc, "selftest_bounded_wait")
    torch.cuda.synchronize(status.device)
    return int(status.item()), [int(x) for x in elapsed.cpu().tolist()]


def paged_attention_decode_tree(out, q, tree_masks, k_cache, v_cache, block_tables, context_lens,
                                max_q_per_seq: int, scale: float, kv_dtype=None, *, cu_q_lens=None,
                                scales=None, workspace=None, device_status=None, stream=None):
    """Speculative verify of a token tree: tree_masks (int64/uint64, one per query row)
    bit i lets a query token attend to its sequence's draft token i; the context before
    the drafts is always visible. cu_q_lens as for paged_attention_decode_varlen, or
    None for max_q_per_seq tokens per sequence. An INT8 cache takes its row scales."""
    for nm, t in (("out", out), ("q", q), ("tree_masks", tree_masks), ("k_cache", k_cache),
                  ("v_cache", v_cache), ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(nm, t)
    if tree_masks.dtype not in (torch.int64, torch.uint64):
        raise PagedKVError("tree_masks must be 64-bit")
    if cu_q_lens is not None:
        _need_cuda_contig("cu_q_lens", cu_q_lens)
    if out.dtype != q.dtype:
        raise PagedKVError("out and q must share a dtype")
    S0, n_max = int(context_lens.shape[0]), int(max_q_per_seq)
    if cu_q_lens is None:
        d, S = _decode_shapes(out, q, k_cache, v_cache, block_tables, context_lens, rows=S0 * n_max)
    else:
        d, S = _decode_shapes(out, q, k_cache, v_cache, block_tables, context_lens, max_rows=S0 * n_max)
        if cu_q_lens.dim() != 1 or int(cu_q_lens.shape[0]) != S + 1 or cu_q_lens.dtype != torch.int32:
            raise PagedKVError("cu_q_lens must be int32 with num_seqs + 1 entries")
    if tree_masks.dim() != 1 or int(tree_masks.shape[0]) != int(q.shape[0]):
        raise PagedKVError("tree_masks must hold one mask per query row")
    code = _kv_code(kv_dtype, k_cache)
    _int8_scales(code, k_cache, scales)
    Hq = int(q.shape[1])
    lib = load_library()
    with _on_device(q.device):
        need = _ws_bytes(lib, q.device, S, Hq, int(max_q_per_seq), d)
        if workspace is None:
            workspace = _workspace(need, q.device)
        ws = (_ptr(workspace), int(workspace.numel() * workspace.element_size()))
        if code == KV_INT8:
            rc = lib.pkv_paged_attention_decode_int8_tree(
                _ptr(out), _ptr(q), _ptr(cu_q_lens), _ptr(tree_masks), int(q.shape[0]), S, Hq,
                int(max_q_per_seq), _ptr(k_cache), _ptr(v_cache), _ptr(scales), ctypes.byref(d),
                _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(scale), *ws,
                _ptr(device_status), _stream_handle(stream, q.device))
        else:
            rc = lib.pkv_paged_attention_decode_tree(
                _ptr(out), _ptr(q), _ptr(cu_q_lens), _ptr(tree_masks), int(q.shape[0]), S, Hq,
                int(max_q_per_seq), _ptr(k_cache), _ptr(v_cache), code, ctypes.byref(d),
                _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(scale), *ws,
                _ptr(device_status), _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode_tree")
    return out


# ------------------------------------------------------------------------------------
# Block pool (host) and block copy (device)
# ------------------------------------------------------------------------------------

OUT_OF_BLOCKS = -6


class BlockAllocator:
    """Host-side block pool of ``num_blocks`` 16-token blocks (the C allocator in
    libpagedkv.so): sequences, fork with copy-on-write, release, and a prefix
    cache of full blocks. Block ids index the caches' first dimension; the
    caches themselves stay with the caller."""

    def __init__(self, num_blocks: int):
        self._lib = load_library()
        self._h = self._lib.pkv_allocator_create(int(num_blocks))
        if not self._h:
            raise PagedKVError(f"pkv_allocator_create({num_blocks}) failed")
        self.num_blocks = int(num_blocks)

    def close(self):
        if self._h:
            self._lib.pkv_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def free_blocks(self) -> int:
        return int(self._lib.pkv_allocator_free_blocks(self._h))

    def evictable(self) -> int:
        return int(self._lib.pkv_allocator_evictable(self._h))

    def refcount(self, block: int) -> int:
        return int(self._lib.pkv_allocator_refcount(self._h, int(block)))

    def add(self, seq: int):
        _check(self._lib.pkv_seq_add(self._h, int(seq)), "seq_add")

    def fork(self, parent: int, child: int):
        _check(self._lib.pkv_seq_fork(self._h, int(parent), int(child)), "seq_fork")

    def release(self, seq: int):
        _check(self._lib.pkv_seq_release(self._h, int(seq)), "seq_release")

    def length(self, seq: int) -> int:
        return int(self._lib.pkv_seq_length(self._h, int(seq)))

    def block_table(self, seq: int) -> list:
        n = int(self._lib.pkv_seq_block_table(self._h, int(seq), None, 0))
        if n < 0:
            _check(n, "seq_block_table")
        buf = (ctypes.c_int32 * max(n, 1))()
        self._lib.pkv_seq_block_table(self._h, int(seq), buf, n)
        return [int(buf[i]) for i in range(n)]

    def append(self, seq: int, n: int):
        """Reserve n tokens; returns (slots, copies) with copies a list of
        (src, dst) block pairs to copy before the new tokens are written."""
        slots = (ctypes.c_int32 * max(int(n), 1))()
        src, dst, nc = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        rc = self._lib.pkv_seq_append(self._h, int(seq), int(n), slots, ctypes.byref(src),
                                      ctypes.byref(dst), ctypes.byref(nc))
        _check(rc, "seq_append")
        copies = [(int(src.value), int(dst.value))] if nc.value else []
        return [int(slots[i]) for i in range(int(n))], copies

    def prefix_insert(self, seq: int, tokens) -> int:
        arr = (ctypes.c_int32 * max(len(tokens), 1))(*[int(t) for t in tokens])
        rc = int(self._lib.pkv_prefix_insert(self._h, int(seq), arr, len(tokens)))
        if rc < 0:
            _check(rc, "prefix_insert")
        return rc

    def add_cached(self, seq: int, tokens) -> int:
        """New sequence starting from the longest cached prefix of ``tokens``
        (whole blocks); returns the number of tokens it already holds."""
        arr = (ctypes.c_int32 * max(len(tokens), 1))(*[int(t) for t in tokens])
        got = ctypes.c_int32()
        _check(self._lib.pkv_seq_add_cached(self._h, int(seq), arr, len(tokens), ctypes.byref(got)),
               "seq_add_cached")
        return int(got.value)


def copy_blocks(k_cache, v_cache, src, dst, kv_dtype=None, *, scales=None, device_status=None, stream=None):
    """Physical block dst[i] of both caches becomes a copy of block src[i]
    (int32 device tensors of equal length); an INT8 cache's row scales
    (``scales``, from alloc_kv_scales) are copied with its blocks."""
    for n_, t in (("k_cache", k_cache), ("v_cache", v_cache), ("src", src), ("dst", dst)):
        _need_cuda_contig(n_, t)
    if src.dtype != torch.int32 or dst.dtype != torch.int32 or src.numel() != dst.numel():
        raise PagedKVError("src and dst must be int32 tensors of equal length")
    d = _pair(k_cache, v_cache)
    code = _kv_code(kv_dtype, k_cache)
    if (code == KV_INT8) != (scales is not None):
        raise PagedKVError("an INT8 cache is copied with its scales; other caches take none")
    if scales is not None:
        _need_cuda_contig("scales", scales)
        _scales_shape(k_cache, scales)
    rc = load_library().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(scales), code,
                                        ctypes.byref(d), _ptr(src), _ptr(dst), int(src.numel()),
                                        _ptr(device_status), _stream_handle(stream, k_cache.device))
    _check(rc, "copy_blocks")
