"""Decode captured in a CUDA graph and replayed: every replay must give exactly
the direct call's output. Replays reuse the launch's arguments (including the
epoch that tags the split-KV piece counters), so this holds only because each
launch leaves the counters clear; the workloads are chosen so that most units
are split across CTAs (mma.sync and tcgen05 kernels)."""
import math

import pytest
import torch

from paged_kv_cache_252_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


CASES = {
    "long_fp16_split": lambda: wl.reduced(wl.by_name("long"), num_seqs=2, ctx_scale=0.25),
    "spec_e5m2_tcgen05": lambda: wl.reduced(wl.by_name("70b_spec"), num_seqs=16),
    "mixed_varlen": lambda: wl.reduced(wl.by_name("mixed"), num_seqs=24),
}


@pytest.mark.parametrize("name", list(CASES))
def test_graph_replays_match_the_direct_call(dev, name):
    import paged_kv_cache_252_gb300 as pkv
    w = CASES[name]()
    vals = wl.token_values(w, device=dev)
    kc, vc = pkv.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, w.kv_dtype, dev)
    pkv.kv_cache_write(vals["k_all"], vals["v_all"], vals["slot_all"], kc, vc)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    cu = torch.from_numpy(w.cu_q_lens()).to(dev) if w.q_lens is not None else None
    q = vals["q"]

    def call(out):
        if cu is not None:
            pkv.paged_attention_decode_varlen(out, q, cu, kc, vc, bt, cl, w.q_per_seq, w.scale)
        else:
            pkv.paged_attention_decode(out, q, kc, vc, bt, cl, w.q_per_seq, w.scale)

    ref = torch.empty_like(q)
    call(ref)
    out = torch.empty_like(q)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(2):
            call(out)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(out)
    for _ in range(4):
        out.fill_(math.nan)
        g.replay()
        torch.cuda.synchronize(dev)
        assert torch.equal(out, ref), "a graph replay differs from the direct call"
