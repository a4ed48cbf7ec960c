"""ctypes wrapper around the C++ oracle (``pagedkv_oracle.cpp``).

Test infrastructure only: the tests, the smoke check and the bench's CPU
baseline use it; nothing on the product path imports it.

All arrays are numpy arrays on the host. fp16/bf16 data travel as their raw
16-bit patterns (``np.uint16``), E5M2 as bytes (``np.uint8``); results are fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FP16, BF16, E5M2, INT8 = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (plain g++)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype)) if a is not None else None


def load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        P = ctypes.POINTER
        lib.orc_version.restype = ctypes.c_int
        lib.orc_fp16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_fp16_to_f64.restype = dbl
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = dbl
        lib.orc_e5m2_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_e5m2_to_f64.restype = dbl
        lib.orc_e5m2_from_fp16.argtypes = [ctypes.c_uint16]
        lib.orc_e5m2_from_fp16.restype = ctypes.c_uint8
        lib.orc_fp16_from_e5m2.argtypes = [ctypes.c_uint8]
        lib.orc_fp16_from_e5m2.restype = ctypes.c_uint16
        lib.orc_e5m2_from_fp16_array.argtypes = [P(ctypes.c_uint16), P(ctypes.c_uint8), i64]
        lib.orc_e5m2_from_fp16_array.restype = None
        lib.orc_round_from_f64.argtypes = [P(dbl), P(ctypes.c_uint16), i64, ctypes.c_int]
        lib.orc_round_from_f64.restype = None
        lib.orc_decode_to_f64.argtypes = [vp, P(dbl), i64, ctypes.c_int]
        lib.orc_decode_to_f64.restype = None
        lib.orc_kv_cache_write.argtypes = [
            P(ctypes.c_uint16), P(ctypes.c_uint16), ctypes.c_int, ctypes.c_int, P(i32),
            vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.orc_kv_cache_write.restype = ctypes.c_int
        lib.orc_paged_attention.argtypes = [
            P(dbl), P(dbl), i64, P(ctypes.c_uint16), ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, P(i32), ctypes.c_int, P(i32), dbl, P(i32), ctypes.c_int, ctypes.c_int,
            P(i32), P(ctypes.c_uint64), P(ctypes.c_float), P(ctypes.c_float)]
        lib.orc_paged_attention.restype = ctypes.c_int
        lib.orc_kv_cache_write_int8.argtypes = [
            P(ctypes.c_uint16), P(ctypes.c_uint16), ctypes.c_int, P(i32), P(ctypes.c_int8),
            P(ctypes.c_int8), P(ctypes.c_float), P(ctypes.c_float), ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int]
        lib.orc_kv_cache_write_int8.restype = ctypes.c_int
        lib.orc_hardware_threads.restype = ctypes.c_int
        assert lib.orc_version() == 1
        _lib = lib
        return lib


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        a = a.view(np.uint16)
    return a


def fp16_to_f64(bits: int) -> float:
    return load().orc_fp16_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return load().orc_bf16_to_f64(int(bits))


def e5m2_to_f64(b: int) -> float:
    return load().orc_e5m2_to_f64(int(b))


def fp16_from_e5m2(b: int) -> int:
    return load().orc_fp16_from_e5m2(int(b))


def e5m2_from_fp16(bits) -> np.ndarray:
    """fp16 bit patterns (any shape) -> E5M2 bytes (same shape)."""
    src = _u16(np.asarray(bits))
    dst = np.empty(src.shape, dtype=np.uint8)
    load().orc_e5m2_from_fp16_array(_p(src.reshape(-1), ctypes.c_uint16),
                                    _p(dst.reshape(-1), ctypes.c_uint8), src.size)
    return dst


def round_from_f64(x, dtype: int) -> np.ndarray:
    """fp64 -> fp16/bf16 bit patterns, round to nearest even."""
    src = np.ascontiguousarray(x, dtype=np.float64)
    dst = np.empty(src.shape, dtype=np.uint16)
    load().orc_round_from_f64(_p(src.reshape(-1), ctypes.c_double),
                              _p(dst.reshape(-1), ctypes.c_uint16), src.size, dtype)
    return dst


def decode_to_f64(raw, dtype: int) -> np.ndarray:
    """fp16/bf16 (uint16 patterns) or E5M2 (uint8) -> fp64."""
    raw = np.ascontiguousarray(raw)
    if dtype == E5M2:
        assert raw.dtype == np.uint8
    else:
        raw = _u16(raw)
    out = np.empty(raw.shape, dtype=np.float64)
    load().orc_decode_to_f64(raw.ctypes.data_as(ctypes.c_void_p),
                             _p(out.reshape(-1), ctypes.c_double), raw.size, dtype)
    return out


def kv_cache_write(key, value, src_dtype: int, slot_mapping, k_cache, v_cache,
                   kv_dtype: int, block_size: int = 16) -> int:
    """Scatter key/value [T, Hkv, D] into caches [NB, Hkv, block_size, D] in place."""
    key, value = _u16(key), _u16(value)
    T, Hkv, D = key.shape
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    NB = k_cache.shape[0]
    return load().orc_kv_cache_write(
        _p(key, ctypes.c_uint16), _p(value, ctypes.c_uint16), src_dtype, T,
        _p(slot_mapping, ctypes.c_int32), k_cache.ctypes.data_as(ctypes.c_void_p),
        v_cache.ctypes.data_as(ctypes.c_void_p), kv_dtype, NB, block_size, Hkv, D)


def kv_cache_write_int8(key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                        block_size: int = 16) -> int:
    """INT8 cache write: fp16 key/value [T, Hkv, D] -> int8 caches [NB, Hkv, block_size, D]
    and float32 scales [NB, Hkv, block_size], in place."""
    key, value = _u16(key), _u16(value)
    T, Hkv, D = key.shape
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    for a in (k_cache, v_cache, k_scale, v_scale):
        assert a.flags.c_contiguous
    assert k_cache.dtype == np.int8 and k_scale.dtype == np.float32
    return load().orc_kv_cache_write_int8(
        _p(key, ctypes.c_uint16), _p(value, ctypes.c_uint16), T, _p(slot_mapping, ctypes.c_int32),
        _p(k_cache, ctypes.c_int8), _p(v_cache, ctypes.c_int8), _p(k_scale, ctypes.c_float),
        _p(v_scale, ctypes.c_float), k_cache.shape[0], block_size, Hkv, D)


def paged_attention(q, q_dtype: int, q_per_seq: int, k_cache, v_cache, kv_dtype: int,
                    block_tables, context_lens, scale: float, *, block_size: int = 16,
                    seqs=None, num_threads: int = 1, want_weights: bool = False,
                    out=None, cu_q_lens=None, tree_masks=None, k_scale=None, v_scale=None):
    """fp64 paged decode attention.

    q: [rows, Hq, D] uint16 patterns: S*q_per_seq rows, or cu_q_lens[S] rows when
    cu_q_lens (int32 [S+1]) gives each sequence its own number of query tokens.
    Caches: [NB, Hkv, block_size, D]. Returns (out_f64 [rows, Hq, D], weights or
    None, rc). Only the rows of ``seqs`` are computed when given. tree_masks (uint64,
    one per query row) replaces the causal rule: bit i lets a token see draft token i.
    An INT8 cache (kv_dtype 3) needs its float32 scales k_scale / v_scale [NB, Hkv, block_size].
    """
    q = _u16(q)
    SN, Hq, D = q.shape
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    S = context_lens.shape[0] if cu_q_lens is not None else SN // q_per_seq
    cu = None if cu_q_lens is None else np.ascontiguousarray(cu_q_lens, dtype=np.int32)
    tm = None if tree_masks is None else np.ascontiguousarray(tree_masks, dtype=np.uint64)
    NB, Hkv = k_cache.shape[0], k_cache.shape[1]
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    mbs = block_tables.shape[1]
    if out is None:
        out = np.full((SN, Hq, D), np.nan, dtype=np.float64)
    weights = None
    wstride = 0
    if want_weights:
        wstride = mbs * block_size
        weights = np.zeros((SN, Hq, wstride), dtype=np.float64)
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
    subset = None
    nsub = 0
    if seqs is not None:
        subset = np.ascontiguousarray(seqs, dtype=np.int32)
        nsub = subset.size
    rc = load().orc_paged_attention(
        _p(out, ctypes.c_double), _p(weights, ctypes.c_double), wstride,
        _p(q, ctypes.c_uint16), q_dtype, S, Hq, q_per_seq,
        k_cache.ctypes.data_as(ctypes.c_void_p), v_cache.ctypes.data_as(ctypes.c_void_p),
        kv_dtype, NB, block_size, Hkv, D, _p(block_tables, ctypes.c_int32), mbs,
        _p(context_lens, ctypes.c_int32), float(scale), _p(subset, ctypes.c_int32), nsub,
        int(num_threads), _p(cu, ctypes.c_int32), _p(tm, ctypes.c_uint64),
        _p(ks, ctypes.c_float), _p(vs, ctypes.c_float))
    return out, weights, rc


def hardware_threads() -> int:
    return load().orc_hardware_threads()
