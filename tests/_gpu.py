"""GPU-side test helpers: run the CUDA path through the Python binding, run the
oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_252_gb300 as pkv
from paged_kv_cache_252_gb300 import workloads as wl
from _helpers import bits16, oracle_caches, oracle_attention, query_rows

# Parity gate for attention outputs against the fp64 oracle:
#   max |gpu - oracle| <= ABS_GATE over every element, and
#   max |gpu - oracle| / |oracle| <= REL_GATE over elements with |oracle| >= REL_FLOOR
# (below REL_FLOOR a 1e-2 relative bound is tighter than the fp16 output's own
# rounding). An E5M2 or INT8 cache is read by the oracle from the same bytes the GPU
# wrote (the cache comparison proves them identical), so the gate is the same.
# A bf16 output cannot meet a 2e-3 absolute bound once |o| >= 0.5 by rounding
# alone (8 significant bits: its half-ulp is 9.8e-4 on [0.25, 0.5), 1.95e-3 on
# [0.5, 1) and 3.9e-3 on [1, 2)), so for bf16 outputs the absolute gate covers
# |oracle| < BF16_ABS_CEIL and the relative gate the rest.
ABS_GATE, REL_GATE, REL_FLOOR = 2e-3, 1e-2, 0.2
BF16_ABS_CEIL = 0.5


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


def parity_errors(got: torch.Tensor, ref: np.ndarray, rows=None):
    """(max abs error over the gated elements, max relative error over |ref| >=
    REL_FLOOR, element count) of got against the fp64 oracle output ref."""
    g = got.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g = g[rows]
        ref = ref[rows]
    assert np.all(np.isfinite(g)), "non-finite output"
    assert np.all(np.isfinite(ref)), "non-finite oracle output"
    err = np.abs(g - ref)
    mag = np.abs(ref)
    abs_region = mag < BF16_ABS_CEIL if got.dtype == torch.bfloat16 else np.ones(err.shape, bool)
    max_abs = float(err[abs_region].max()) if abs_region.any() else 0.0
    big = mag >= REL_FLOOR
    max_rel = float((err[big] / mag[big]).max()) if big.any() else 0.0
    return max_abs, max_rel, err, g, ref


def compare(got: torch.Tensor, ref: np.ndarray, rows=None, label: str = ""):
    """Gate got (the GPU output) against ref (the oracle's, fp64): max-abs and
    max-rel as above. Prints and returns (max_abs, max_rel)."""
    max_abs, max_rel, err, g, ref = parity_errors(got, ref, rows)
    print(f"parity {label or '-'} [{str(got.dtype).replace('torch.', '')} out, {err.size} elements]: "
          f"max-abs {max_abs:.3e} (gate {ABS_GATE:g}), max-rel {max_rel:.3e} (gate {REL_GATE:g})")
    if max_abs > ABS_GATE or max_rel > REL_GATE:
        mag = np.abs(ref)
        abs_region = mag < BF16_ABS_CEIL if got.dtype == torch.bfloat16 else np.ones(err.shape, bool)
        bad = (abs_region & (err > ABS_GATE)) | ((mag >= REL_FLOOR) & (err > REL_GATE * mag))
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outputs out of the gate: max-abs "
                             f"{max_abs:.3e}, max-rel {max_rel:.3e}; first bad {idx.tolist()} got "
                             f"{[g[tuple(k)] for k in idx]} ref {[ref[tuple(k)] for k in idx]}")
    return max_abs, max_rel


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
    label = f"{w.name} {w.kv_dtype} D{w.head_size} G{w.group} n{w.q_per_seq} S{w.num_seqs}"
    return compare(out, ref, rows, label=label)
