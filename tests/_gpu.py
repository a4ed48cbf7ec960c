"""GPU-side test helpers: run the CUDA path through the Python binding, run the
oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_252_gb300 as pkv
from paged_kv_cache_252_gb300 import workloads as wl
from _helpers import bits16, oracle_caches, oracle_attention, query_rows

ATOL, RTOL = 2e-3, 1e-2


def cuda_path(w, vals, dev, *, split_write=True, status=None):
    """Cache write (prefill tokens, then the step's new tokens) and decode on the GPU."""
    kc, vc = pkv.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, w.kv_dtype, dev)
    k_all, v_all = vals["k_all"].to(dev), vals["v_all"].to(dev)
    slots = vals["slot_all"].to(dev)
    if split_write:
        pre = torch.from_numpy(wl.prefill_mask(w)).to(dev)
        new = ~pre
        if bool(pre.any()):
            pkv.kv_cache_write(k_all[pre].contiguous(), v_all[pre].contiguous(),
                               slots[pre].contiguous(), kc, vc, device_status=status)
        pkv.kv_cache_write(k_all[new].contiguous(), v_all[new].contiguous(), slots[new].contiguous(),
                           kc, vc, device_status=status)
    else:
        pkv.kv_cache_write(k_all, v_all, slots, kc, vc, device_status=status)
    q = vals["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    if w.q_lens is not None:
        cu = torch.from_numpy(w.cu_q_lens()).to(dev)
        pkv.paged_attention_decode_varlen(out, q, cu, kc, vc, bt, cl, w.q_per_seq, w.scale,
                                          device_status=status)
    else:
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, w.q_per_seq, w.scale, device_status=status)
    torch.cuda.synchronize(dev)
    return kc, vc, out


def cache_bytes(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


def compare(got: torch.Tensor, ref: np.ndarray, rows=None, atol=ATOL, rtol=RTOL):
    """Element-wise |got - ref| <= atol + rtol*|ref| (ref in fp64). Returns max abs error."""
    g = got.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g = g[rows]
        ref = ref[rows]
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outputs out of tolerance; max abs err "
                             f"{err.max():.3e}; first bad {idx.tolist()} got "
                             f"{[g[tuple(i)] for i in idx]} ref {[ref[tuple(i)] for i in idx]}")
    return float(err.max())


def full_check(orc, w, dev, *, seqs=None, values_device="cpu", check_cache=True, threads=None):
    """CUDA path vs oracle on workload w. Cache images must match bit for bit; outputs
    within tolerance (all sequences, or the sampled ones in `seqs`)."""
    vals = wl.token_values(w, device=values_device)
    return check_values(orc, w, vals, dev, seqs=seqs, check_cache=check_cache, threads=threads)


def check_values(orc, w, vals, dev, *, seqs=None, check_cache=True, threads=None):
    """full_check on given token values (q, k_all, v_all, slot_all)."""
    kc, vc, out = cuda_path(w, vals, dev)
    vals = {k: v.cpu() for k, v in vals.items()}
    okc, ovc = oracle_caches(orc, w, vals)
    if check_cache:
        assert np.array_equal(cache_bytes(kc), okc), "K cache bytes differ from the oracle's"
        assert np.array_equal(cache_bytes(vc), ovc), "V cache bytes differ from the oracle's"
    nthreads = threads or orc.hardware_threads()
    ref, _, rc = oracle_attention(orc, w, vals, okc, ovc, seqs=seqs, num_threads=nthreads)
    assert rc == 0
    rows = None
    if seqs is not None:
        rows = query_rows(w, seqs)
    return compare(out, ref, rows)
