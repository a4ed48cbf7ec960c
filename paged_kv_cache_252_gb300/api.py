"""Python binding of libpagedkv.so: argument marshalling only.

Every function here turns torch tensors into device pointers and sizes and
calls the C ABI declared in ``include/pagedkv.h``; the computation happens in
the library's CUDA kernels. There is no fallback: if the library is missing or
a call fails, a :class:`PagedKVError` is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

KV_FP16, KV_BF16, KV_E5M2 = 0, 1, 2
_NAMES = {"fp16": KV_FP16, "bf16": KV_BF16, "e5m2": KV_E5M2, "fp8_e5m2": KV_E5M2}
_TORCH = {torch.float16: KV_FP16, torch.bfloat16: KV_BF16, torch.uint8: KV_E5M2,
          torch.float8_e5m2: KV_E5M2}
BLOCK_SIZE = 16

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None
_workspaces: dict = {}


class PagedKVError(RuntimeError):
    pass


class _CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_size", ctypes.c_int32)]


def library_path() -> str:
    return os.path.join(_HERE, "libpagedkv.so")


def load_library():
    """Load libpagedkv.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
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
            vp, vp, vp, i32, i32, i32, vp, vp, ctypes.c_int, P(_CacheDesc), vp, i32, vp,
            ctypes.c_float, vp, ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode_varlen.restype = ctypes.c_int
        lib.pkv_paged_attention_decode_tree.argtypes = [
            vp, vp, vp, vp, i32, i32, i32, vp, vp, ctypes.c_int, P(_CacheDesc), vp, i32, vp,
            ctypes.c_float, vp, ctypes.c_size_t, vp, vp]
        lib.pkv_paged_attention_decode_tree.restype = ctypes.c_int
        lib.pkv_paged_attention_decode_noalloc.argtypes = [
            vp, vp, i32, i32, i32, vp, vp, ctypes.c_int, P(_CacheDesc), vp, i32, vp,
            ctypes.c_float, vp, vp]
        lib.pkv_paged_attention_decode_noalloc.restype = ctypes.c_int
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


def _need_cuda_contig(name, t):
    if not t.is_cuda:
        raise PagedKVError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PagedKVError(f"{name} must be contiguous")


def alloc_kv_cache(num_blocks: int, num_kv_heads: int, head_size: int, kv_dtype,
                   device="cuda", zero: bool = True):
    """Allocate a K/V cache pair [num_blocks, num_kv_heads, 16, head_size]."""
    code = _NAMES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    dt = {KV_FP16: torch.float16, KV_BF16: torch.bfloat16, KV_E5M2: torch.uint8}[code]
    mk = torch.zeros if zero else torch.empty
    shape = (num_blocks, num_kv_heads, BLOCK_SIZE, head_size)
    return mk(shape, dtype=dt, device=device), mk(shape, dtype=dt, device=device)


def kv_cache_write(key, value, slot_mapping, k_cache, v_cache, kv_dtype=None, *,
                   device_status=None, stream=None):
    """Scatter key/value [T, Hkv, D] into their cache slots (fp16->E5M2 cast for an E5M2 cache)."""
    for n, t in (("key", key), ("value", value), ("slot_mapping", slot_mapping),
                 ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda_contig(n, t)
    if slot_mapping.dtype != torch.int32:
        raise PagedKVError("slot_mapping must be int32")
    d = _desc(k_cache)
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


def _workspace(nbytes: int, device) -> torch.Tensor:
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
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
    S = int(context_lens.shape[0])
    Hq = int(q.shape[1])
    d = _desc(k_cache)
    code = _kv_code(kv_dtype, k_cache)
    lib = load_library()
    with torch.cuda.device(q.device):
        need = int(lib.pkv_decode_workspace_bytes(S, Hq, q_per_seq, ctypes.byref(d)))
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
    d = _desc(k_cache)
    with torch.cuda.device(q.device):
        rc = load_library().pkv_paged_attention_decode_noalloc(
            _ptr(out), _ptr(q), int(context_lens.shape[0]), int(q.shape[1]), int(q_per_seq),
            _ptr(k_cache), _ptr(v_cache), _kv_code(kv_dtype, k_cache), ctypes.byref(d),
            _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(scale),
            _ptr(device_status), _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode_noalloc")
    return out


def paged_attention_decode_varlen(out, q, cu_q_lens, k_cache, v_cache, block_tables, context_lens,
                                  max_q_per_seq: int, scale: float, kv_dtype=None, *,
                                  workspace=None, device_status=None, stream=None):
    """Decode attention for a batch whose sequences carry different numbers of query
    tokens, packed without padding: sequence s owns rows cu_q_lens[s]..cu_q_lens[s+1]-1
    of q/out ([total_rows, Hq, D]), 1 <= n_s <= max_q_per_seq, causal among its tokens."""
    for nm, t in (("out", out), ("q", q), ("cu_q_lens", cu_q_lens), ("k_cache", k_cache),
                  ("v_cache", v_cache), ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(nm, t)
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32
            or cu_q_lens.dtype != torch.int32):
        raise PagedKVError("block_tables, context_lens and cu_q_lens must be int32")
    if out.dtype != q.dtype:
        raise PagedKVError("out and q must share a dtype")
    S = int(context_lens.shape[0])
    if int(cu_q_lens.shape[0]) != S + 1:
        raise PagedKVError("cu_q_lens must have num_seqs + 1 entries")
    Hq = int(q.shape[1])
    d = _desc(k_cache)
    lib = load_library()
    with torch.cuda.device(q.device):
        need = int(lib.pkv_decode_workspace_bytes(S, Hq, int(max_q_per_seq), ctypes.byref(d)))
        if workspace is None:
            workspace = _workspace(need, q.device)
        rc = lib.pkv_paged_attention_decode_varlen(
            _ptr(out), _ptr(q), _ptr(cu_q_lens), S, Hq, int(max_q_per_seq), _ptr(k_cache),
            _ptr(v_cache), _kv_code(kv_dtype, k_cache), ctypes.byref(d), _ptr(block_tables),
            int(block_tables.shape[1]), _ptr(context_lens), float(scale), _ptr(workspace),
            int(workspace.numel() * workspace.element_size()), _ptr(device_status),
            _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode_varlen")
    return out


def paged_attention_decode_tree(out, q, tree_masks, k_cache, v_cache, block_tables, context_lens,
                                max_q_per_seq: int, scale: float, kv_dtype=None, *, cu_q_lens=None,
                                workspace=None, device_status=None, stream=None):
    """Speculative verify of a token tree: tree_masks (int64/uint64, one per query row)
    bit i lets a query token attend to its sequence's draft token i; the context before
    the drafts is always visible. cu_q_lens as for paged_attention_decode_varlen, or
    None for max_q_per_seq tokens per sequence."""
    for nm, t in (("out", out), ("q", q), ("tree_masks", tree_masks), ("k_cache", k_cache),
                  ("v_cache", v_cache), ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(nm, t)
    if tree_masks.dtype not in (torch.int64, torch.uint64):
        raise PagedKVError("tree_masks must be 64-bit")
    if cu_q_lens is not None:
        _need_cuda_contig("cu_q_lens", cu_q_lens)
    if out.dtype != q.dtype:
        raise PagedKVError("out and q must share a dtype")
    S = int(context_lens.shape[0])
    Hq = int(q.shape[1])
    d = _desc(k_cache)
    lib = load_library()
    with torch.cuda.device(q.device):
        need = int(lib.pkv_decode_workspace_bytes(S, Hq, int(max_q_per_seq), ctypes.byref(d)))
        if workspace is None:
            workspace = _workspace(need, q.device)
        rc = lib.pkv_paged_attention_decode_tree(
            _ptr(out), _ptr(q), _ptr(cu_q_lens), _ptr(tree_masks), S, Hq, int(max_q_per_seq),
            _ptr(k_cache), _ptr(v_cache), _kv_code(kv_dtype, k_cache), ctypes.byref(d),
            _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(scale),
            _ptr(workspace), int(workspace.numel() * workspace.element_size()),
            _ptr(device_status), _stream_handle(stream, q.device))
    _check(rc, "paged_attention_decode_tree")
    return out
