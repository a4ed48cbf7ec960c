"""GB300-native paged decode attention over a blocked KV cache.

Two calls, both hand-written CUDA for sm_103a behind a C ABI (``libpagedkv.so``):

* :func:`kv_cache_write` scatters new key/value tokens into their physical
  cache slots (fp16/bf16 copy, or fp16 -> FP8 E5M2 cast).
* :func:`paged_attention_decode` computes softmax(q K^T * scale) V for every
  sequence over its blocks, one CTA stream per KV head serving the whole GQA
  group, causal among a sequence's query tokens (speculative verify).

:class:`BlockAllocator` (host, C++) hands out the blocks: sequences, fork with
copy-on-write (:func:`copy_blocks` performs the copies), and a prefix cache.

The Python layer only marshals torch tensors into pointers and sizes; every
step of the computation runs in the CUDA library. Importing this package does
not load the library; the first call does, and fails loudly if it is missing.
"""
from . import workloads  # noqa: F401
from .api import (  # noqa: F401
    KV_FP16, KV_BF16, KV_E5M2, KV_INT8,
    kv_cache_write, paged_attention_decode, paged_attention_decode_varlen,
    paged_attention_decode_tree, paged_attention_decode_chunked, selftest_bounded_wait,
    paged_attention_decode_noalloc, decode_workspace_bytes,
    library_path, load_library, alloc_kv_cache, PagedKVError,
    BlockAllocator, copy_blocks,
    alloc_kv_scales, kv_cache_write_int8, paged_attention_decode_int8, int8_codes,
)
