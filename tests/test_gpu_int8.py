"""INT8 KV cache on the GPU against the oracle: the cache write's codes and
row scales bit for bit, decode attention within the parity gate of tests/_gpu.py
(the oracle reads the same codes and scales)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_252_gb300 import workloads as wl
from _helpers import bits16, cache_shape, query_rows

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


def _gpu_caches(w, vals, dev, status=None):
    """Prefill tokens, then the step's new tokens, through the INT8 cache write.
    Returns the caches and the one scales tensor [nb, Hkv, 2, 16] (K, then V)."""
    import paged_kv_cache_252_gb300 as pkv
    kc, vc = pkv.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, "int8", dev)
    sc = pkv.alloc_kv_scales(w.num_blocks, w.num_kv_heads, dev)
    k_all, v_all, slots = vals["k_all"].to(dev), vals["v_all"].to(dev), vals["slot_all"].to(dev)
    pre = torch.from_numpy(wl.prefill_mask(w)).to(dev)
    for m in (pre, ~pre):
        if bool(m.any()):
            pkv.kv_cache_write_int8(k_all[m].contiguous(), v_all[m].contiguous(), slots[m].contiguous(),
                                    kc, vc, sc, device_status=status)
    return kc, vc, sc


def _split_scales(sc):
    """The GPU's scales tensor as the oracle's separate K and V arrays [nb, Hkv, 16]."""
    a = sc.cpu().numpy()
    return a[:, :, 0, :], a[:, :, 1, :]


def _oracle_caches(orc, w, vals):
    kc = np.zeros(cache_shape(w), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros(cache_shape(w)[:3], np.float32)
    vs = np.zeros_like(ks)
    rc = orc.kv_cache_write_int8(bits16(vals["k_all"]), bits16(vals["v_all"]),
                                 vals["slot_all"].cpu().numpy().astype(np.int32), kc, vc, ks, vs)
    assert rc == 0
    return kc, vc, ks, vs


def _check(orc, gpu, w, dev, *, seqs=None, values_device="cpu"):
    import paged_kv_cache_252_gb300 as pkv
    vals = wl.token_values(w, device=values_device)
    kc, vc, sc = _gpu_caches(w, vals, dev)
    q = vals["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode_int8(out, q, kc, vc, sc, bt, cl, w.q_per_seq, w.scale, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ks, vs = _split_scales(sc)
    vals = {k: v.cpu() for k, v in vals.items()}
    okc, ovc, oks, ovs = _oracle_caches(orc, w, vals)
    assert np.array_equal(pkv.int8_codes(kc).cpu().numpy(), okc) and np.array_equal(pkv.int8_codes(vc).cpu().numpy(), ovc)
    assert np.array_equal(ks, oks) and np.array_equal(vs, ovs)
    ref, _, rc = orc.paged_attention(bits16(vals["q"]), 0, w.q_per_seq, okc, ovc, 3, w.block_tables,
                                     w.context_lens, w.scale, seqs=seqs, num_threads=orc.hardware_threads(),
                                     k_scale=oks, v_scale=ovs)
    assert rc == 0
    return gpu.compare(out, ref, None if seqs is None else query_rows(w, seqs), label=f"{w.name} int8 D{w.head_size} G{w.group} n{w.q_per_seq} S{w.num_seqs}")


def test_int8_cache_write_bit_exact_on_hard_rows(orc, dev):
    import paged_kv_cache_252_gb300 as pkv
    for D in (64, 128):
        T, Hkv = 48, 3
        rng = np.random.default_rng(D)
        x = (rng.standard_normal((T, Hkv, D)) * rng.choice([1e-4, 1.0, 1e3], size=(T, Hkv, 1))).astype(np.float16)
        x[3] = 0.0
        x[4, 0, 5] = np.float16(65504.0)
        x[5, 1, :] = np.float16(-2.5)              # every element at the row maximum
        slots = np.arange(T, dtype=np.int32)[rng.permutation(T)]
        slots[7] = -1                              # skipped
        nb = (T + 15) // 16 + 1
        key = torch.from_numpy(x).to(dev)
        val = torch.from_numpy(x[::-1].copy()).to(dev)
        kc, vc = pkv.alloc_kv_cache(nb, Hkv, D, "int8", dev)
        sc = pkv.alloc_kv_scales(nb, Hkv, dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        pkv.kv_cache_write_int8(key, val, torch.from_numpy(slots).to(dev), kc, vc, sc, device_status=status)
        torch.cuda.synchronize()
        okc = np.zeros((nb, Hkv, 16, D), np.int8)
        ovc = np.zeros_like(okc)
        oks = np.zeros((nb, Hkv, 16), np.float32)
        ovs = np.zeros_like(oks)
        assert orc.kv_cache_write_int8(x.view(np.uint16), x[::-1].copy().view(np.uint16), slots,
                                       okc, ovc, oks, ovs) == 0
        assert np.array_equal(pkv.int8_codes(kc).cpu().numpy(), okc) and np.array_equal(pkv.int8_codes(vc).cpu().numpy(), ovc)
        ks, vs = _split_scales(sc)
        assert np.array_equal(ks, oks) and np.array_equal(vs, ovs)
        assert int(status.item()) == 0
        bad = torch.tensor([nb * 16 + 2], dtype=torch.int32, device=dev)
        pkv.kv_cache_write_int8(key[:1].contiguous(), val[:1].contiguous(), bad, kc, vc, sc,
                                device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & 0x1


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 48, 49, 64, 65, 127, 200]
SHAPES = [(4, 4, 1), (8, 2, 1), (8, 1, 1), (16, 2, 2), (12, 4, 5), (64, 8, 4), (16, 1, 4)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"Hq{a}-Hkv{b}-n{c}" for a, b, c in SHAPES])
def test_int8_decode_small_parity(orc, dev, gpu, D, shape):
    Hq, Hkv, n = shape
    lens = [max(x, n) for x in EDGE_LENS]
    w = wl.custom(num_seqs=len(lens), num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, q_per_seq=n,
                  kv_dtype="int8", context_lens=lens, seed=2000 + D + Hq * 7 + n)
    _check(orc, gpu, w, dev)


def test_int8_workload_reduced(orc, dev, gpu):
    _check(orc, gpu, wl.reduced(wl.by_name("8b_int8"), num_seqs=6), dev)


def test_int8_workload_full_size(orc, dev, gpu):
    """The full-size INT8 workload: every code, scale and output element."""
    _check(orc, gpu, wl.by_name("8b_int8"), dev, values_device=dev)


def test_int8_single_token_contexts_are_exact_up_to_the_output_rounding(orc, dev, gpu):
    """Contexts of one or two tokens put a single token's dequantised V row (code *
    scale) in the output with weight ~1: the fp16 rounding of P * scale must not
    reach the output. Many rows of N(0,1) values give row maxima near 4, where the
    scale's fp16 rounding and the output's are each worth up to ~1.95e-3."""
    S = 256
    w = wl.custom(num_seqs=S, num_q_heads=8, num_kv_heads=8, head_size=128, q_per_seq=1, kv_dtype="int8",
                  context_lens=[1 + (s % 2) for s in range(S)], seed=4242)
    _check(orc, gpu, w, dev)


def test_int8_bad_block_is_flagged_not_faulted(orc, dev, gpu):
    import paged_kv_cache_252_gb300 as pkv
    w = wl.custom(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=128, q_per_seq=1, kv_dtype="int8",
                  context_lens=[40, 70, 9], seed=6)
    vals = wl.token_values(w)
    kc, vc, sc = _gpu_caches(w, vals, dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    bt[0, 1] = w.num_blocks + 3
    cl = torch.from_numpy(w.context_lens).to(dev)
    q = vals["q"].to(dev)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode_int8(out, q, kc, vc, sc, bt, cl, 1, w.scale, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x2
    okc, ovc, oks, ovs = _oracle_caches(orc, w, vals)
    ref, _, _ = orc.paged_attention(bits16(vals["q"]), 0, 1, okc, ovc, 3, w.block_tables, w.context_lens,
                                    w.scale, seqs=[1, 2], k_scale=oks, v_scale=ovs)
    gpu.compare(out, ref, rows=[1, 2])


# ------------------------------------------------------------------------------------
# INT8 cache under the mixed-batch (per-sequence query counts) and token-tree calls
# ------------------------------------------------------------------------------------

def _check_packed(orc, gpu, w, dev, *, tree_masks=None, values_device="cpu"):
    """Varlen (w.q_lens set) or token-tree decode over an INT8 cache against the oracle
    on the same codes and scales."""
    import paged_kv_cache_252_gb300 as pkv
    vals = wl.token_values(w, device=values_device)
    kc, vc, sc = _gpu_caches(w, vals, dev)
    q = vals["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    cu = torch.from_numpy(w.cu_q_lens()).to(dev) if w.q_lens is not None else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if tree_masks is None:
        pkv.paged_attention_decode_varlen(out, q, cu, kc, vc, bt, cl, w.q_per_seq, w.scale, scales=sc,
                                          device_status=status)
    else:
        tm = torch.from_numpy(tree_masks.view(np.int64)).to(dev)
        pkv.paged_attention_decode_tree(out, q, tm, kc, vc, bt, cl, w.q_per_seq, w.scale, cu_q_lens=cu,
                                        scales=sc, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ks, vs = _split_scales(sc)
    vals = {k: v.cpu() for k, v in vals.items()}
    okc, ovc, oks, ovs = _oracle_caches(orc, w, vals)
    assert np.array_equal(pkv.int8_codes(kc).cpu().numpy(), okc) and np.array_equal(pkv.int8_codes(vc).cpu().numpy(), ovc)
    assert np.array_equal(ks, oks) and np.array_equal(vs, ovs)
    ref, _, rc = orc.paged_attention(bits16(vals["q"]), 0, w.q_per_seq, okc, ovc, 3, w.block_tables,
                                     w.context_lens, w.scale, num_threads=orc.hardware_threads(),
                                     cu_q_lens=w.cu_q_lens(), tree_masks=tree_masks, k_scale=oks, v_scale=ovs)
    assert rc == 0
    kind = "varlen" if tree_masks is None else "tree"
    return gpu.compare(out, ref, label=f"{w.name} int8 {kind} D{w.head_size} G{w.group} n<={w.q_per_seq}")


INT8_VARLEN = [
    # (D, Hq, Hkv, q_lens)
    (128, 32, 8, [1, 4, 1, 1, 4, 2, 1, 3]),
    (64, 16, 4, [2, 1, 4, 1, 1, 3]),
    (128, 64, 8, [4, 1, 2, 4, 1]),
    (64, 8, 1, [1, 8, 3, 1, 5, 2]),
]


@pytest.mark.parametrize("case", INT8_VARLEN, ids=[f"D{c[0]}-G{c[1] // c[2]}" for c in INT8_VARLEN])
def test_int8_varlen_parity(orc, dev, gpu, case):
    D, Hq, Hkv, q_lens = case
    lens = [max(l, ql) for l, ql in zip([1, 17, 300, 16, 64, 1000, 33, 129], q_lens)]
    w = wl.custom(num_seqs=len(q_lens), num_q_heads=Hq, num_kv_heads=Hkv, head_size=D,
                  q_per_seq=max(q_lens), kv_dtype="int8", context_lens=lens, seed=3300 + D + Hq,
                  q_lens=q_lens)
    _check_packed(orc, gpu, w, dev)


INT8_TREES = [
    # (D, Hq, Hkv, q_lens or uniform n)
    (128, 64, 8, 4),
    (128, 32, 8, [5, 1, 8, 3, 2]),
    (64, 8, 4, [16, 3, 9]),
    # two row groups, with sequences whose rows fit one group
    (128, 32, 8, [4, 1, 2, 1, 3]),
]


def _int8_tree_id(c):
    n = c[3] if isinstance(c[3], int) else max(c[3])
    return f"D{c[0]}-G{c[1] // c[2]}-n{n}"


@pytest.mark.parametrize("case", INT8_TREES, ids=[_int8_tree_id(c) for c in INT8_TREES])
def test_int8_tree_verify_parity(orc, dev, gpu, case):
    D, Hq, Hkv, ql = case
    S = 5 if isinstance(ql, int) else len(ql)
    q_lens = [ql] * S if isinstance(ql, int) else ql
    lens = [max(l, n) for l, n in zip([20, 1, 300, 33, 1200], q_lens)]
    w = wl.custom(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, q_per_seq=max(q_lens),
                  kv_dtype="int8", context_lens=lens, seed=3500 + D,
                  q_lens=None if isinstance(ql, int) else q_lens)
    _check_packed(orc, gpu, w, dev, tree_masks=wl.random_tree_masks(q_lens, seed=13 + D))


def test_int8_mixed_workload_full_size(orc, dev, gpu):
    """The mixed decode/verify batch of the 8B layer (1 or 4 query tokens per
    sequence) over an INT8 cache, every output element."""
    m = wl.by_name("mixed")
    w = wl.make_workload("mixed_8b_decode_verify_int8", num_seqs=m.num_seqs, num_q_heads=m.num_q_heads,
                         num_kv_heads=m.num_kv_heads, head_size=m.head_size, q_per_seq=m.q_per_seq,
                         kv_dtype="int8", scale=m.scale, seed=m.seed, context_lens=m.context_lens,
                         q_lens=m.q_lens)
    _check_packed(orc, gpu, w, dev, values_device=dev)
