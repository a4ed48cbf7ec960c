"""Shared test utilities: raw-bit views and oracle-side cache construction."""
from __future__ import annotations

import numpy as np
import torch

KV_CODE = {"fp16": 0, "bf16": 1, "e5m2": 2}
Q_CODE = {"fp16": 0, "bf16": 1}


def bits16(t: torch.Tensor) -> np.ndarray:
    """fp16/bf16 torch tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits16(a: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)


def cache_shape(w):
    return (w.num_blocks, w.num_kv_heads, 16, w.head_size)


def oracle_caches(orc, w, vals, *, token_mask=None):
    """Build K/V cache images with the oracle's own cache write from the packed tokens."""
    dt = np.uint8 if w.kv_dtype == "e5m2" else np.uint16
    kc = np.zeros(cache_shape(w), dtype=dt)
    vc = np.zeros(cache_shape(w), dtype=dt)
    k_all, v_all = bits16(vals["k_all"]), bits16(vals["v_all"])
    slots = vals["slot_all"].cpu().numpy().astype(np.int32)
    if token_mask is not None:
        k_all, v_all, slots = k_all[token_mask], v_all[token_mask], slots[token_mask]
    src = KV_CODE["bf16"] if w.kv_dtype == "bf16" else KV_CODE["fp16"]
    rc = orc.kv_cache_write(k_all, v_all, src, slots, kc, vc, KV_CODE[w.kv_dtype])
    assert rc == 0
    return kc, vc


def oracle_attention(orc, w, vals, kc, vc, **kw):
    q = bits16(vals["q"])
    if w.q_lens is not None:
        kw.setdefault("cu_q_lens", w.cu_q_lens())
    return orc.paged_attention(q, Q_CODE[w.q_dtype], w.q_per_seq, kc, vc, KV_CODE[w.kv_dtype],
                               w.block_tables, w.context_lens, w.scale, **kw)


def query_rows(w, seqs):
    """Rows of q/out that belong to the given sequences."""
    cu = w.cu_q_lens()
    return np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])


def dense_kv_f64(w, vals, s):
    """Contiguous K/V of sequence s as fp64 [ctx, Hkv, D], decoded by torch (no block table)."""
    starts = w.seq_starts()
    k = vals["k_all"][starts[s]:starts[s + 1]].cpu()
    v = vals["v_all"][starts[s]:starts[s + 1]].cpu()
    if w.kv_dtype == "e5m2":
        k = k.to(torch.float8_e5m2)
        v = v.to(torch.float8_e5m2)
    return k.to(torch.float64), v.to(torch.float64)


def sdpa_reference(w, vals, s, tree_masks=None):
    """Library reference for sequence s: torch SDPA in fp64 on contiguous K/V, GQA by
    repeating each KV head over its G query heads, causal among the n query tokens."""
    G = w.group
    cu = w.cu_q_lens()
    n = int(cu[s + 1] - cu[s])
    ctx = int(w.context_lens[s])
    k, v = dense_kv_f64(w, vals, s)                          # [ctx, Hkv, D]
    q = vals["q"][cu[s]:cu[s + 1]].cpu().to(torch.float64)   # [n, Hq, D]
    k = k.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]  # [1, Hq, ctx, D]
    v = v.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    qq = q.permute(1, 0, 2)[None]                              # [1, Hq, n, D]
    pos = torch.arange(ctx)[None, :]
    if tree_masks is None:
        lim = (ctx - n + torch.arange(n))[:, None]
        mask = pos <= lim                                      # [n, ctx]
    else:
        base = ctx - n
        mask = torch.zeros(n, ctx, dtype=torch.bool)
        mask[:, :base] = True
        for j in range(n):
            m = int(tree_masks[cu[s] + j])
            for i in range(n):
                mask[j, base + i] = bool((m >> i) & 1)
    o = torch.nn.functional.scaled_dot_product_attention(qq, k, v, attn_mask=mask, scale=w.scale)
    return o[0].permute(1, 0, 2).numpy()                       # [n, Hq, D]
