"""Seeded synthetic workloads for paged decode attention.

This module only draws inputs: sequence lengths, a shuffled physical block
pool with its block table and slot mapping, and N(0,1) keys, values and
queries. It holds none of the attention or cast arithmetic, so both the CUDA
path and the CPU oracle can take their inputs from it.

Shapes follow the serving workloads the pages talk about (Llama-3-8B and
Llama-3-70B decode layers, a long-context decode and a speculative verify
step): "AI大模型推理速度翻倍，Colossal-Inference开源发布" (性能对比, 投机采样) and
"TACO-LLM 如何实现降本增效?" (长序列推理优化中的 TurboAttention). The block
size is 16 ("AI 大模型推理优化技术详解", 2.1.2 Paged Attention).

Structure (lengths, pool permutation) comes from numpy's PCG64 seeded with
the workload's seed; values come from a torch generator with the same seed,
on the device the caller asks for.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

BLOCK_SIZE = 16

KV_DTYPES = ("fp16", "bf16", "e5m2", "int8")


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    q_per_seq: int
    kv_dtype: str
    scale: float
    seed: int
    context_lens: np.ndarray            # int32 [S]
    num_blocks: int                     # physical blocks in the pool
    block_tables: np.ndarray            # int32 [S, max_blocks]; -1 past a sequence's blocks
    notes: str = ""
    extra: dict = field(default_factory=dict)
    q_lens: np.ndarray | None = None    # int32 [S] query tokens per sequence (None: q_per_seq each)

    # ---- derived --------------------------------------------------------------
    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def q_dtype(self) -> str:
        return "bf16" if self.kv_dtype == "bf16" else "fp16"

    @property
    def torch_q_dtype(self):
        return torch.bfloat16 if self.q_dtype == "bf16" else torch.float16

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype in ("e5m2", "int8") else 2

    @property
    def kv_row_extra_bytes(self) -> int:
        """Bytes stored per (token, KV head) row besides the elements: the INT8
        cache's float32 row scale."""
        return 4 if self.kv_dtype == "int8" else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_tokens_total(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())

    @property
    def num_new_tokens(self) -> int:
        return int(self.query_lens().sum())

    def query_lens(self) -> np.ndarray:
        """Query tokens of every sequence (q_per_seq each unless q_lens is set)."""
        if self.q_lens is not None:
            return self.q_lens.astype(np.int32)
        return np.full(self.num_seqs, self.q_per_seq, dtype=np.int32)

    def cu_q_lens(self) -> np.ndarray:
        """Row offsets of each sequence's query tokens in the packed q/out ([S+1])."""
        c = np.zeros(self.num_seqs + 1, dtype=np.int32)
        np.cumsum(self.query_lens(), out=c[1:])
        return c

    def seq_starts(self) -> np.ndarray:
        """Start of each sequence in the packed all-token arrays."""
        c = np.zeros(self.num_seqs + 1, dtype=np.int64)
        np.cumsum(self.context_lens.astype(np.int64), out=c[1:])
        return c

    def slot_mapping_all(self) -> np.ndarray:
        """Physical slot of every cached token, sequences packed in order.

        The slot of position p of sequence s is block_tables[s][p // 16] * 16 + p % 16,
        the logical-to-physical map of the blocked cache.
        """
        out = np.empty(self.num_tokens_total, dtype=np.int32)
        starts = self.seq_starts()
        for s in range(self.num_seqs):
            ctx = int(self.context_lens[s])
            p = np.arange(ctx, dtype=np.int64)
            blocks = self.block_tables[s, p // BLOCK_SIZE].astype(np.int64)
            out[starts[s]:starts[s + 1]] = (blocks * BLOCK_SIZE + p % BLOCK_SIZE).astype(np.int32)
        return out

    def new_token_index(self) -> np.ndarray:
        """Indices (into the packed all-token arrays) of each sequence's newest tokens
        (its query tokens, which the step writes into the cache)."""
        starts = self.seq_starts()
        ql = self.query_lens()
        idx = [np.arange(starts[s + 1] - ql[s], starts[s + 1]) for s in range(self.num_seqs)]
        return np.concatenate(idx).astype(np.int64)

    def kv_bytes_read(self) -> int:
        """Algorithmic KV bytes one decode call must read (K and V of every visible token,
        and an INT8 cache's row scales)."""
        row = self.head_size * self.kv_elem_bytes + self.kv_row_extra_bytes
        return int(self.num_tokens_total * self.num_kv_heads * row * 2)

    def q_out_bytes(self) -> int:
        return int(2 * self.num_new_tokens * self.num_q_heads * self.head_size * 2)

    def write_bytes(self) -> int:
        """Algorithmic bytes of the per-step cache write (read new K/V, write cache slots)."""
        t = self.num_new_tokens
        src = t * self.num_kv_heads * self.head_size * 2 * 2
        dst = t * self.num_kv_heads * (self.head_size * self.kv_elem_bytes + self.kv_row_extra_bytes) * 2
        return int(src + dst + 4 * t)

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "num_seqs": self.num_seqs,
            "num_q_heads": self.num_q_heads,
            "num_kv_heads": self.num_kv_heads,
            "head_size": self.head_size,
            "block_size": BLOCK_SIZE,
            "q_per_seq": self.q_per_seq,
            "kv_dtype": self.kv_dtype,
            "q_dtype": self.q_dtype,
            "context_len_mean": float(self.context_lens.mean()),
            "context_len_min": int(self.context_lens.min()),
            "context_len_max": int(self.context_lens.max()),
            "query_tokens": int(self.num_new_tokens),
            "num_blocks": self.num_blocks,
            "seed": self.seed,
        }


def _pool_and_tables(rng: np.random.Generator, context_lens: np.ndarray, pool_factor: float,
                     min_pool: int = 0):
    nb = (context_lens.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE
    need = int(nb.sum())
    num_blocks = max(int(math.ceil(pool_factor * need)), min_pool, need)
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_nb = int(nb.max())
    tables = np.full((len(context_lens), max_nb), -1, dtype=np.int32)
    pos = 0
    for s, k in enumerate(nb):
        tables[s, :k] = perm[pos:pos + k]
        pos += k
    return num_blocks, tables


def make_workload(name: str, *, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                  head_size: int, q_per_seq: int, kv_dtype: str, scale: float, seed: int,
                  context_lens, pool_factor: float = 1.25, min_pool: int = 0,
                  notes: str = "", q_lens=None) -> Workload:
    assert kv_dtype in KV_DTYPES
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    context_lens = np.asarray(context_lens, dtype=np.int32)
    num_blocks, tables = _pool_and_tables(rng, context_lens, pool_factor, min_pool)
    if q_lens is not None:
        q_lens = np.asarray(q_lens, dtype=np.int32)
        assert q_lens.shape == (num_seqs,) and q_lens.min() >= 1
        assert np.all(q_lens <= context_lens)
        q_per_seq = int(q_lens.max())
    return Workload(name, num_seqs, num_q_heads, num_kv_heads, head_size, q_per_seq, kv_dtype,
                    float(scale), seed, context_lens, num_blocks, tables, notes, q_lens=q_lens)


def _uniform_lens(seed, n, lo, hi):
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(lo, hi + 1, size=n).astype(np.int32)


def _lognormal_lens(seed, n, median, sigma, lo, hi):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = np.rint(np.exp(np.log(median) + sigma * rng.standard_normal(n)))
    return np.clip(x, lo, hi).astype(np.int32)


# ---- the five named workloads ------------------------------------------------------

def tiny() -> Workload:
    """4 sequences, lengths {1,17,33,64}, 4 q heads / 2 KV heads, head 64, fp16,
    scale 1/8, block table drawn from a shuffled 32-block pool, 1 new token each."""
    return make_workload("tiny_paged_decode", num_seqs=4, num_q_heads=4, num_kv_heads=2,
                         head_size=64, q_per_seq=1, kv_dtype="fp16", scale=1.0 / 8.0, seed=253,
                         context_lens=[1, 17, 33, 64], pool_factor=1.0, min_pool=32,
                         notes="pool of 32 physical blocks, 10 used")


def llama3_8b_bs64_fp16(num_seqs: int = 64) -> Workload:
    """Llama-3-8B-shaped decode layer: 32 q / 8 KV heads, head 128, fp16 KV,
    lengths uniform in [512, 2048], pool 1.25x the blocks needed, shuffled."""
    seed = 254
    return make_workload("llama3_8b_decode_bs64_fp16", num_seqs=num_seqs, num_q_heads=32,
                         num_kv_heads=8, head_size=128, q_per_seq=1, kv_dtype="fp16",
                         scale=1.0 / math.sqrt(128), seed=seed,
                         context_lens=_uniform_lens(seed, num_seqs, 512, 2048))


def llama3_8b_bs256_e5m2(num_seqs: int = 256) -> Workload:
    """Same 8B heads with an FP8 E5M2 KV cache: 256 sequences, lengths uniform in
    [1024, 4096], fp16 queries and output."""
    seed = 255
    return make_workload("llama3_8b_decode_bs256_e5m2", num_seqs=num_seqs, num_q_heads=32,
                         num_kv_heads=8, head_size=128, q_per_seq=1, kv_dtype="e5m2",
                         scale=1.0 / math.sqrt(128), seed=seed,
                         context_lens=_uniform_lens(seed, num_seqs, 1024, 4096))


def llama3_8b_bs256_int8(num_seqs: int = 256) -> Workload:
    """The 8B fp8 workload with an INT8 KV cache (per-row float32 scales): 256
    sequences, lengths uniform in [1024, 4096], fp16 queries and output."""
    seed = 259
    return make_workload("llama3_8b_decode_bs256_int8", num_seqs=num_seqs, num_q_heads=32,
                         num_kv_heads=8, head_size=128, q_per_seq=1, kv_dtype="int8",
                         scale=1.0 / math.sqrt(128), seed=seed,
                         context_lens=_uniform_lens(seed, num_seqs, 1024, 4096))


def long_bs8_bf16(num_seqs: int = 8, lo: int = 32768, hi: int = 131072) -> Workload:
    """Long-context split-KV decode: 8 sequences, 32 q / 8 KV heads, head 128,
    bf16 KV, lengths uniform in [32768, 131072], fully shuffled blocks."""
    seed = 256
    return make_workload("long_context_bs8_bf16", num_seqs=num_seqs, num_q_heads=32,
                         num_kv_heads=8, head_size=128, q_per_seq=1, kv_dtype="bf16",
                         scale=1.0 / math.sqrt(128), seed=seed,
                         context_lens=_uniform_lens(seed, num_seqs, lo, hi))


def llama3_70b_spec4_e5m2(num_seqs: int = 128) -> Workload:
    """Llama-3-70B-shaped speculative verify: 128 sequences, 64 q / 8 KV heads,
    head 128, E5M2 KV, 4 query tokens per sequence (causal among themselves),
    lengths lognormal (median 1024, sigma 1) clipped to [4, 16384]."""
    seed = 257
    return make_workload("llama3_70b_spec_verify4_e5m2", num_seqs=num_seqs, num_q_heads=64,
                         num_kv_heads=8, head_size=128, q_per_seq=4, kv_dtype="e5m2",
                         scale=1.0 / math.sqrt(128), seed=seed,
                         context_lens=_lognormal_lens(seed, num_seqs, 1024.0, 1.0, 4, 16384))


def mixed_8b_decode_verify(num_seqs: int = 64) -> Workload:
    """Continuous-batching mix on the 8B decode layer: each sequence carries 1 query
    token (plain decode) or 4 (speculative verify), 3:1, packed without padding;
    lengths uniform in [512, 2048], fp16 KV."""
    seed = 258
    rng = np.random.Generator(np.random.PCG64(seed))
    q_lens = rng.choice(np.array([1, 1, 1, 4], dtype=np.int32), size=num_seqs)
    return make_workload("mixed_8b_decode_verify_fp16", num_seqs=num_seqs, num_q_heads=32,
                         num_kv_heads=8, head_size=128, q_per_seq=4, kv_dtype="fp16",
                         scale=1.0 / math.sqrt(128), seed=seed,
                         context_lens=_uniform_lens(seed, num_seqs, 512, 2048), q_lens=q_lens)


NAMED = {
    "tiny": tiny,
    "8b": llama3_8b_bs64_fp16,
    "8b_fp8": llama3_8b_bs256_e5m2,
    "8b_int8": llama3_8b_bs256_int8,
    "long": long_bs8_bf16,
    "70b_spec": llama3_70b_spec4_e5m2,
    "mixed": mixed_8b_decode_verify,
}


def by_name(key: str, **kw) -> Workload:
    return NAMED[key](**kw)


def reduced(w: Workload, *, num_seqs: int | None = None, ctx_scale: float = 1.0,
            ctx_cap: int | None = None, name_suffix: str = "_small") -> Workload:
    """Same heads/dtypes/distribution family with fewer sequences and/or shorter lengths,
    for oracle-sized parity runs. Lengths are rescaled, then clipped to [q_per_seq, cap]."""
    S = num_seqs or w.num_seqs
    lens = w.context_lens[:S].astype(np.float64) * ctx_scale
    lens = np.rint(lens)
    if ctx_cap is not None:
        lens = np.minimum(lens, ctx_cap)
    lens = np.maximum(lens, w.q_per_seq).astype(np.int32)
    q_lens = None if w.q_lens is None else w.q_lens[:S]
    return make_workload(w.name + name_suffix, num_seqs=S, num_q_heads=w.num_q_heads,
                         num_kv_heads=w.num_kv_heads, head_size=w.head_size,
                         q_per_seq=w.q_per_seq, kv_dtype=w.kv_dtype, scale=w.scale,
                         seed=w.seed, context_lens=lens, q_lens=q_lens)


def custom(*, num_seqs, num_q_heads, num_kv_heads, head_size, q_per_seq, kv_dtype,
           context_lens, seed=1000, scale=None, pool_factor=1.25, min_pool=0,
           name="custom", q_lens=None) -> Workload:
    if scale is None:
        scale = 1.0 / math.sqrt(head_size)
    return make_workload(name, num_seqs=num_seqs, num_q_heads=num_q_heads,
                         num_kv_heads=num_kv_heads, head_size=head_size, q_per_seq=q_per_seq,
                         kv_dtype=kv_dtype, scale=scale, seed=seed, context_lens=context_lens,
                         pool_factor=pool_factor, min_pool=min_pool, q_lens=q_lens)


# ---- values ---------------------------------------------------------------------------

def _randn(gen, shape, device, dtype):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def token_values(w: Workload, device="cpu", *, chunk_tokens: int = 1 << 20):
    """N(0,1) keys/values for every cached token and queries for the new tokens.

    Returns a dict of torch tensors on ``device``:
      k_all, v_all : [T_total, Hkv, D]  source dtype (fp16, or bf16 for a bf16 cache)
      q            : [rows, Hq, D]       query dtype (S*n rows, or sum(q_lens))
      slot_all     : [T_total] int32     physical slots (sequences packed in order)
      new_idx      : [rows] int64        which of the packed tokens are the step's new ones
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    src = torch.bfloat16 if w.kv_dtype == "bf16" else torch.float16
    T = w.num_tokens_total
    Hkv, D = w.num_kv_heads, w.head_size
    k_all = torch.empty((T, Hkv, D), dtype=src, device=device)
    v_all = torch.empty((T, Hkv, D), dtype=src, device=device)
    for t0 in range(0, T, chunk_tokens):
        t1 = min(T, t0 + chunk_tokens)
        k_all[t0:t1] = _randn(gen, (t1 - t0, Hkv, D), device, src)
        v_all[t0:t1] = _randn(gen, (t1 - t0, Hkv, D), device, src)
    q = _randn(gen, (w.num_new_tokens, w.num_q_heads, D), device, w.torch_q_dtype)
    slot_all = torch.from_numpy(w.slot_mapping_all()).to(device)
    new_idx = torch.from_numpy(w.new_token_index()).to(device)
    return {"k_all": k_all, "v_all": v_all, "q": q, "slot_all": slot_all, "new_idx": new_idx}


def prefill_mask(w: Workload) -> np.ndarray:
    """Boolean mask over the packed tokens: True for tokens already cached before the step."""
    m = np.ones(w.num_tokens_total, dtype=bool)
    m[w.new_token_index()] = False
    return m


def random_tree_masks(q_lens, seed: int) -> np.ndarray:
    """Seeded token trees for speculative verify: in each sequence, draft token i
    (i = 0..n_s-1) has a parent drawn uniformly from {context, draft 0..i-1}; its
    mask holds its ancestors' bits and its own. Returns uint64 [sum(q_lens)]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for n in np.asarray(q_lens, dtype=np.int64):
        masks = []
        for i in range(int(n)):
            parent = int(rng.integers(-1, i)) if i > 0 else -1
            m = (masks[parent] if parent >= 0 else 0) | (1 << i)
            masks.append(m)
        out.extend(masks)
    return np.array(out, dtype=np.uint64)
