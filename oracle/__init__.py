"""CPU oracle for paged decode attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package. The product path (the CUDA library and
its Python binding) never imports it.
"""
from .oracle import (  # noqa: F401
    FP16, BF16, E5M2, INT8,
    build, load,
    e5m2_from_fp16, fp16_from_e5m2, e5m2_to_f64, fp16_to_f64, bf16_to_f64,
    round_from_f64, decode_to_f64,
    kv_cache_write, kv_cache_write_int8, paged_attention, hardware_threads,
)
