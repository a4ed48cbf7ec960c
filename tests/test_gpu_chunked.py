"""Decode attention over batches that mix prefill chunks of any length with decode
and verify tokens (the chunked entry point, host-side query counts) against the
oracle, and bit for bit against the varlen entry point where both apply."""
import numpy as np
import pytest
import torch

from paged_kv_cache_252_gb300 import workloads as wl
from _helpers import bits16, cache_shape, oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def gpu(dev):
    import _gpu
    return _gpu


def _caches(w, vals, dev):
    """Prefill tokens, then the step's new tokens, through the library's cache write.
    Returns (k_cache, v_cache, INT8 scales or None)."""
    import paged_kv_cache_252_gb300 as pkv
    kc, vc = pkv.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, w.kv_dtype, dev)
    sc = pkv.alloc_kv_scales(w.num_blocks, w.num_kv_heads, dev) if w.kv_dtype == "int8" else None
    k_all, v_all, slots = vals["k_all"].to(dev), vals["v_all"].to(dev), vals["slot_all"].to(dev)
    pre = torch.from_numpy(wl.prefill_mask(w)).to(dev)
    for m in (pre, ~pre):
        if bool(m.any()):
            args = (k_all[m].contiguous(), v_all[m].contiguous(), slots[m].contiguous(), kc, vc)
            if sc is None:
                pkv.kv_cache_write(*args)
            else:
                pkv.kv_cache_write_int8(*args, sc)
    return kc, vc, sc


def _oracle_ref(orc, w, vals):
    vals = {k: v.cpu() for k, v in vals.items()}
    if w.kv_dtype != "int8":
        okc, ovc = oracle_caches(orc, w, vals)
        ref, _, rc = oracle_attention(orc, w, vals, okc, ovc, num_threads=orc.hardware_threads())
        assert rc == 0
        return ref
    okc = np.zeros(cache_shape(w), np.int8)
    ovc = np.zeros_like(okc)
    oks = np.zeros(cache_shape(w)[:3], np.float32)
    ovs = np.zeros_like(oks)
    assert orc.kv_cache_write_int8(bits16(vals["k_all"]), bits16(vals["v_all"]),
                                   vals["slot_all"].numpy().astype(np.int32), okc, ovc, oks, ovs) == 0
    ref, _, rc = orc.paged_attention(bits16(vals["q"]), 0, w.q_per_seq, okc, ovc, 3, w.block_tables,
                                     w.context_lens, w.scale, num_threads=orc.hardware_threads(),
                                     cu_q_lens=w.cu_q_lens(), k_scale=oks, v_scale=ovs)
    assert rc == 0
    return ref


CHUNKED = [
    # (kv, D, Hq, Hkv, q_lens, context_lens): prefill chunks of 33..150 tokens beside
    # decode (1) and verify (2..9) tokens; row tiles hold 64 / G tokens
    ("fp16", 128, 32, 8, [1, 150, 4, 1, 37], [300, 410, 64, 1, 37]),   # G 4: 16-token tiles
    ("bf16", 64, 8, 4, [70, 1, 2, 33], [90, 500, 40, 33]),              # G 2: 32-token tiles
    ("e5m2", 128, 64, 8, [1, 100, 9, 4], [200, 180, 9, 50]),            # G 8: 64-row tiles (tcgen05)
    ("e5m2", 64, 16, 4, [130, 1, 5], [260, 77, 20]),
    ("int8", 128, 32, 8, [1, 120, 3], [250, 300, 40]),
]


@pytest.mark.parametrize("case", CHUNKED, ids=[f"{c[0]}-D{c[1]}-G{c[2] // c[3]}" for c in CHUNKED])
def test_chunked_batches_match_the_oracle(orc, dev, gpu, case):
    import paged_kv_cache_252_gb300 as pkv
    kv, D, Hq, Hkv, q_lens, ctx = case
    w = wl.custom(num_seqs=len(q_lens), num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, q_per_seq=max(q_lens),
                  kv_dtype=kv, context_lens=ctx, seed=700 + D + Hq, q_lens=q_lens)
    vals = wl.token_values(w)
    kc, vc, sc = _caches(w, vals, dev)
    q = vals["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    bt = torch.from_numpy(w.block_tables).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode_chunked(out, q, q_lens, w.context_lens, kc, vc, bt, w.scale, scales=sc,
                                       device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gpu.compare(out, _oracle_ref(orc, w, vals), label=f"chunked {kv} D{D} G{Hq // Hkv} q_lens {q_lens}")


def test_chunked_equals_varlen_when_every_sequence_fits_one_tile(dev, gpu):
    """With at most 64 / G tokens per sequence every sequence is one tile: the same
    units, shares and block ids as the varlen call, so the same output bits."""
    import paged_kv_cache_252_gb300 as pkv
    q_lens = [1, 4, 2, 16, 1, 9]
    w = wl.custom(num_seqs=6, num_q_heads=32, num_kv_heads=8, head_size=128, q_per_seq=16, kv_dtype="fp16",
                  context_lens=[30, 700, 64, 200, 1, 333], seed=77, q_lens=q_lens)
    vals = wl.token_values(w)
    kc, vc, _ = _caches(w, vals, dev)
    q = vals["q"].to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    a = torch.full_like(q, float("nan"))
    b = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode_chunked(a, q, q_lens, w.context_lens, kc, vc, bt, w.scale)
    pkv.paged_attention_decode_varlen(b, q, torch.from_numpy(w.cu_q_lens()).to(dev), kc, vc, bt,
                                      torch.from_numpy(w.context_lens).to(dev), 16, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_chunked_rows_of_one_chunk_equal_the_single_token_decodes(dev, gpu):
    """Query token j of a chunk is a decode of context ctx - n + j + 1: the chunk's
    rows must equal those decodes (different tiles, shares and splits; the same
    attention up to fp32 summation order)."""
    import paged_kv_cache_252_gb300 as pkv
    n, ctx = 90, 200
    w = wl.custom(num_seqs=1, num_q_heads=16, num_kv_heads=4, head_size=128, q_per_seq=n, kv_dtype="fp16",
                  context_lens=[ctx], seed=91, q_lens=[n])
    vals = wl.token_values(w)
    kc, vc, _ = _caches(w, vals, dev)
    q = vals["q"].to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode_chunked(out, q, [n], [ctx], kc, vc, bt, w.scale)
    # n sequences of one token each over the same block-table row
    one = torch.full_like(q, float("nan"))
    lens = torch.arange(ctx - n + 1, ctx + 1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode(one, q, kc, vc, bt.expand(n, -1).contiguous(), lens, 1, w.scale)
    torch.cuda.synchronize()
    gpu.compare(out, one.float().cpu().numpy().astype(np.float64), label="chunk rows vs single-token decodes")


def test_chunked_call_replays_from_a_cuda_graph(dev, gpu):
    """The tiles' metadata travels as launch parameters: a captured call replays to
    the same output bits."""
    import paged_kv_cache_252_gb300 as pkv
    q_lens, ctx = [1, 70, 3], [100, 300, 20]
    w = wl.custom(num_seqs=3, num_q_heads=16, num_kv_heads=4, head_size=128, q_per_seq=70, kv_dtype="fp16",
                  context_lens=ctx, seed=19, q_lens=q_lens)
    vals = wl.token_values(w)
    kc, vc, _ = _caches(w, vals, dev)
    q = vals["q"].to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    ref = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode_chunked(ref, q, q_lens, ctx, kc, vc, bt, w.scale)
    torch.cuda.synchronize()
    out = torch.full_like(q, float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # the binding's workspace for this stream, outside the capture
        pkv.paged_attention_decode_chunked(out, q, q_lens, ctx, kc, vc, bt, w.scale)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        pkv.paged_attention_decode_chunked(out, q, q_lens, ctx, kc, vc, bt, w.scale)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
