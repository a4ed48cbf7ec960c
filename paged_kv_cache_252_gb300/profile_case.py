"""Run one decode workload a few times, for profilers (ncu) and quick timing.

    python -m paged_kv_cache_252_gb300.profile_case --config 8b [--num-seqs N] [--iters 3]

Builds the cache with the library's own cache write (the INT8 one for an INT8
workload), then calls the matching decode --iters times on the same stream and prints the device
status word. --num-seqs N keeps the workload's shapes and length distribution
but only its first N sequences (a smaller case that still exceeds the L2).
"""
from __future__ import annotations

import argparse

import torch

from . import api
from . import workloads as wl


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="8b", choices=list(wl.NAMED))
    ap.add_argument("--num-seqs", type=int, default=0)
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    dev = torch.device("cuda:0")
    w = wl.by_name(args.config)
    if args.num_seqs:
        w = wl.reduced(w, num_seqs=args.num_seqs)
    vals = wl.token_values(w, device=dev)
    kc, vc = api.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, w.kv_dtype, dev)
    int8 = w.kv_dtype == "int8"
    if int8:
        sc = api.alloc_kv_scales(w.num_blocks, w.num_kv_heads, dev)
        api.kv_cache_write_int8(vals["k_all"], vals["v_all"], vals["slot_all"], kc, vc, sc)
    else:
        api.kv_cache_write(vals["k_all"], vals["v_all"], vals["slot_all"], kc, vc)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    out = torch.empty_like(vals["q"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cu = torch.from_numpy(w.cu_q_lens()).to(dev) if w.q_lens is not None else None
    for _ in range(args.iters):
        if int8:
            api.paged_attention_decode_int8(out, vals["q"], kc, vc, sc, bt, cl, w.q_per_seq, w.scale,
                                            device_status=status)
        elif cu is not None:
            api.paged_attention_decode_varlen(out, vals["q"], cu, kc, vc, bt, cl, w.q_per_seq,
                                              w.scale, device_status=status)
        else:
            api.paged_attention_decode(out, vals["q"], kc, vc, bt, cl, w.q_per_seq, w.scale,
                                       device_status=status)
    torch.cuda.synchronize()
    print(f"{w.name}: {w.num_seqs} seqs, {w.kv_bytes_read() / 1e6:.1f} MB KV per call, "
          f"status {int(status.item())}")


if __name__ == "__main__":
    main()
