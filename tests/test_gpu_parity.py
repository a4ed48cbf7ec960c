"""CUDA path vs the CPU oracle, through the C ABI (Python binding = marshalling only).

Cache writes must match the oracle's cache image bit for bit; attention outputs
must meet the parity gate of tests/_gpu.py: max |gpu - oracle| <= 2e-3 over every
element and max relative error <= 1e-2 over elements with |oracle| >= 0.2 (fp64
oracle; an E5M2 cache is read by the oracle from the same bytes, which the cache
check proves identical; bf16 outputs take the absolute gate below |oracle| 0.5).
"""
import numpy as np
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


@pytest.fixture(scope="module")
def gpu(dev):
    import _gpu
    return _gpu


# ------------------------------------------------------------------------------------
# cache write
# ------------------------------------------------------------------------------------

def test_e5m2_cast_exhaustive_through_cache_write(orc, dev, gpu):
    """All 65,536 fp16 patterns written through kv_cache_write into an E5M2 cache
    equal the oracle's cast byte for byte (NaN, inf, saturation, subnormals, ties)."""
    import paged_kv_cache_252_gb300 as pkv
    T, Hkv, D = 512, 1, 128
    pat = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(T, Hkv, D)
    key = torch.from_numpy(pat.view(np.int16)).view(torch.float16).to(dev)
    val = torch.from_numpy(pat[::-1].copy().view(np.int16)).view(torch.float16).to(dev)
    slots = torch.from_numpy(np.random.default_rng(0).permutation(T).astype(np.int32)).to(dev)
    kc, vc = pkv.alloc_kv_cache(T // 16, Hkv, D, "e5m2", dev)
    pkv.kv_cache_write(key, val, slots, kc, vc)
    torch.cuda.synchronize()
    okc = np.zeros(kc.shape, np.uint8)
    ovc = np.zeros(vc.shape, np.uint8)
    assert orc.kv_cache_write(pat, pat[::-1].copy(), orc.FP16, slots.cpu().numpy(), okc, ovc, orc.E5M2) == 0
    assert np.array_equal(gpu.cache_bytes(kc), okc)
    assert np.array_equal(gpu.cache_bytes(vc), ovc)


@pytest.mark.parametrize("kv", ["fp16", "bf16", "e5m2"])
@pytest.mark.parametrize("D", [64, 128])
def test_cache_write_bit_exact(orc, dev, gpu, kv, D):
    w = wl.custom(num_seqs=5, num_q_heads=8, num_kv_heads=4, head_size=D, q_per_seq=1,
                  kv_dtype=kv, context_lens=[1, 16, 17, 100, 333], seed=70 + D)
    vals = wl.token_values(w)
    kc, vc, _ = gpu.cuda_path(w, vals, dev)
    okc, ovc = gpu.oracle_caches(orc, w, vals)
    assert np.array_equal(gpu.cache_bytes(kc), okc)
    assert np.array_equal(gpu.cache_bytes(vc), ovc)


def test_cache_write_skips_minus_one_and_flags_bad_slots(orc, dev, gpu):
    import paged_kv_cache_252_gb300 as pkv
    key = torch.randn(4, 2, 64, device=dev).half()
    slots = torch.tensor([-1, 5, 1 << 20, -7], dtype=torch.int32, device=dev)
    kc, vc = pkv.alloc_kv_cache(4, 2, 64, "fp16", dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.kv_cache_write(key, key, slots, kc, vc, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x1
    flat = kc.permute(0, 2, 1, 3).reshape(64, 2, 64)   # slot-major view
    assert torch.equal(flat[5], key[1])
    nz = (kc != 0).any(dim=-1).sum().item()
    assert nz == 2                                      # only slot 5 (two heads) written


# ------------------------------------------------------------------------------------
# decode attention: small shapes, all dtypes, block edges, GQA groups, spec tokens
# ------------------------------------------------------------------------------------

EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 48, 49, 64, 65, 127, 200]

SHAPES = [
    # (Hq, Hkv, n)   rows = Hq/Hkv * n
    (4, 4, 1),     # GQA-H (MHA), rows 1
    (8, 4, 1),     # rows 2
    (8, 2, 1),     # rows 4
    (8, 1, 1),     # GQA-1 (MQA), rows 8
    (16, 2, 2),    # rows 16
    (12, 4, 5),    # rows 15 (ragged tile)
    (64, 8, 4),    # 70B verify, rows 32
    (24, 1, 1),    # rows 24 (padded to 32 on the tensor-core path)
    (8, 1, 5),     # rows 40 (padded to 64)
    (16, 1, 4),    # rows 64
]


@pytest.mark.parametrize("kv", ["fp16", "bf16", "e5m2"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"Hq{a}-Hkv{b}-n{c}" for a, b, c in SHAPES])
def test_decode_small_parity(orc, dev, gpu, kv, D, shape):
    Hq, Hkv, n = shape
    lens = [max(x, n) for x in EDGE_LENS]
    w = wl.custom(num_seqs=len(lens), num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, q_per_seq=n,
                  kv_dtype=kv, context_lens=lens, seed=1000 + D + Hq * 7 + n)
    gpu.full_check(orc, w, dev)


def test_tiny_workload(orc, dev, gpu):
    gpu.full_check(orc, wl.tiny(), dev)


def test_decode_is_deterministic(orc, dev, gpu):
    w = wl.custom(num_seqs=6, num_q_heads=32, num_kv_heads=8, head_size=128, q_per_seq=1,
                  kv_dtype="fp16", context_lens=[700, 1, 64, 3000, 17, 999], seed=5)
    vals = wl.token_values(w)
    _, _, o1 = gpu.cuda_path(w, vals, dev)
    _, _, o2 = gpu.cuda_path(w, vals, dev)
    assert torch.equal(o1, o2)


def test_scale_zero_gives_mean_of_v(orc, dev, gpu):
    w = wl.custom(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=128, q_per_seq=1,
                  kv_dtype="bf16", context_lens=[5, 40, 300], seed=8, scale=0.0)
    gpu.full_check(orc, w, dev)


def test_bad_block_and_context_are_flagged_not_faulted(orc, dev, gpu):
    import paged_kv_cache_252_gb300 as pkv
    w = wl.custom(num_seqs=3, num_q_heads=4, num_kv_heads=2, head_size=64, q_per_seq=2,
                  kv_dtype="fp16", context_lens=[20, 40, 9], seed=3)
    vals = wl.token_values(w)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kc, vc, _ = gpu.cuda_path(w, vals, dev, status=status)
    assert int(status.item()) == 0
    bt = torch.from_numpy(w.block_tables).to(dev)
    bt[0, 1] = w.num_blocks + 5          # out-of-range physical block
    cl = torch.from_numpy(w.context_lens).to(dev)
    cl[2] = 1                            # shorter than q_per_seq
    q = vals["q"].to(dev)
    out = torch.empty_like(q)
    pkv.paged_attention_decode(out, q, kc, vc, bt, cl, 2, w.scale, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x2 and int(status.item()) & 0x4
    assert torch.isfinite(out[2:4]).all()   # sequence 1 untouched by the bad inputs
    okc, ovc = gpu.oracle_caches(orc, w, vals)
    ref, _, _ = gpu.oracle_attention(orc, w, vals, okc, ovc, seqs=[1])
    gpu.compare(out, ref, rows=[2, 3])


def test_bad_block_and_context_flagged_on_wide_units(orc, dev, gpu):
    """The same checks on a unit of 32 rows over an E5M2 cache (tensor-core kernel)."""
    import paged_kv_cache_252_gb300 as pkv
    w = wl.custom(num_seqs=3, num_q_heads=64, num_kv_heads=8, head_size=128, q_per_seq=4,
                  kv_dtype="e5m2", context_lens=[200, 400, 9], seed=4)
    vals = wl.token_values(w)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kc, vc, _ = gpu.cuda_path(w, vals, dev, status=status)
    assert int(status.item()) == 0
    bt = torch.from_numpy(w.block_tables).to(dev)
    bt[0, 1] = w.num_blocks + 5          # out-of-range physical block
    cl = torch.from_numpy(w.context_lens).to(dev)
    cl[2] = 1                            # shorter than q_per_seq
    q = vals["q"].to(dev)
    out = torch.empty_like(q)
    pkv.paged_attention_decode(out, q, kc, vc, bt, cl, 4, w.scale, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x2 and int(status.item()) & 0x4
    assert not int(status.item()) & 0x8
    okc, ovc = gpu.oracle_caches(orc, w, vals)
    ref, _, _ = gpu.oracle_attention(orc, w, vals, okc, ovc, seqs=[1])
    gpu.compare(out, ref, rows=[4, 5, 6, 7])


def _ramp_keys(w, vals, slope):
    """Scale each sequence's keys by 1 + slope*position: later tokens score far
    higher, so the running max of every row keeps moving after the first chunk."""
    starts = w.seq_starts()
    k = vals["k_all"].float()
    for s in range(w.num_seqs):
        n = int(starts[s + 1] - starts[s])
        f = 1.0 + slope * torch.arange(n, dtype=torch.float32)
        k[starts[s]:starts[s + 1]] *= f[:, None, None]
    vals["k_all"] = k.to(vals["k_all"].dtype)
    return vals


@pytest.mark.parametrize("kv,Hq,Hkv,n", [("e5m2", 64, 8, 4), ("e5m2", 8, 1, 5), ("fp16", 32, 8, 1),
                                         ("bf16", 64, 8, 4)])
def test_rising_scores_move_the_running_max(orc, dev, gpu, kv, Hq, Hkv, n):
    w = wl.custom(num_seqs=4, num_q_heads=Hq, num_kv_heads=Hkv, head_size=128, q_per_seq=n,
                  kv_dtype=kv, context_lens=[900, 300, 129, 2000], seed=77)
    vals = _ramp_keys(w, wl.token_values(w), 1.0 / 32)
    gpu.check_values(orc, w, vals, dev)


def test_empty_batch_is_a_no_op(dev):
    import paged_kv_cache_252_gb300 as pkv
    kc, vc = pkv.alloc_kv_cache(4, 2, 64, "fp16", dev)
    q = torch.empty(0, 4, 64, dtype=torch.float16, device=dev)
    bt = torch.empty(0, 1, dtype=torch.int32, device=dev)
    cl = torch.empty(0, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode(q, q, kc, vc, bt, cl, 1, 0.125)
    pkv.kv_cache_write(q.view(0, 2, 128)[:, :, :64].contiguous(), q.view(0, 2, 128)[:, :, :64].contiguous(),
                       cl, kc, vc)
    torch.cuda.synchronize()


# ------------------------------------------------------------------------------------
# the five workloads: reduced sizes, and full sizes over every sequence
# ------------------------------------------------------------------------------------

REDUCED = {
    "8b": dict(num_seqs=6),
    "8b_fp8": dict(num_seqs=6),
    "long": dict(num_seqs=2, ctx_scale=0.06),
    "70b_spec": dict(num_seqs=10),
}


@pytest.mark.parametrize("key", list(REDUCED))
def test_workload_reduced_full_parity(orc, dev, gpu, key):
    w = wl.reduced(wl.by_name(key), **REDUCED[key])
    gpu.full_check(orc, w, dev)


@pytest.mark.parametrize("key", ["8b", "8b_fp8", "long", "70b_spec"])
def test_workload_full_size_parity(orc, dev, gpu, key):
    """Full-size workload in the bench's launch configuration: every cache byte and
    every output element of every sequence against the oracle."""
    w = wl.by_name(key)
    gpu.full_check(orc, w, dev, values_device=dev)


# ------------------------------------------------------------------------------------
# mixed batches (per-sequence query-token counts)
# ------------------------------------------------------------------------------------

VARLEN = [
    # (kv, D, Hq, Hkv, q_lens)
    ("fp16", 128, 32, 8, [1, 4, 1, 1, 4, 2, 1, 3]),
    ("bf16", 64, 16, 4, [2, 1, 4, 1, 1, 3]),
    ("e5m2", 128, 64, 8, [4, 1, 2, 4, 1]),
    ("fp16", 64, 8, 1, [1, 8, 3, 1, 5, 2]),
    # units of 9..16 rows run two row groups; a sequence whose rows fit one group
    # spreads its blocks over every consumer warp (12 rows: 6 per group)
    ("fp16", 128, 12, 4, [1, 2, 3, 4, 1, 2, 3, 1]),
    ("e5m2", 128, 32, 8, [1, 4, 2, 1, 3, 1]),
    ("e5m2", 64, 32, 8, [2, 1, 1, 4, 1, 3]),
]


@pytest.mark.parametrize("case", VARLEN, ids=[f"{c[0]}-D{c[1]}-G{c[2] // c[3]}-n{max(c[4])}" for c in VARLEN])
def test_varlen_parity(orc, dev, gpu, case):
    kv, D, Hq, Hkv, q_lens = case
    lens = [max(l, ql) for l, ql in zip([1, 17, 300, 16, 64, 1000, 33, 129], q_lens)]
    w = wl.custom(num_seqs=len(q_lens), num_q_heads=Hq, num_kv_heads=Hkv, head_size=D,
                  q_per_seq=max(q_lens), kv_dtype=kv, context_lens=lens, seed=300 + D + Hq,
                  q_lens=q_lens)
    gpu.full_check(orc, w, dev)


def test_mixed_workload_reduced(orc, dev, gpu):
    gpu.full_check(orc, wl.reduced(wl.by_name("mixed"), num_seqs=12), dev)


def test_mixed_workload_full_size(orc, dev, gpu):
    gpu.full_check(orc, wl.by_name("mixed"), dev, values_device=dev)


def test_varlen_rejects_bad_counts_without_faulting(orc, dev, gpu):
    import paged_kv_cache_252_gb300 as pkv
    w = wl.custom(num_seqs=3, num_q_heads=4, num_kv_heads=2, head_size=64, q_per_seq=2,
                  kv_dtype="fp16", context_lens=[20, 40, 9], seed=3, q_lens=[1, 2, 2])
    vals = wl.token_values(w)
    kc, vc, out = gpu.cuda_path(w, vals, dev)
    cu = torch.tensor([0, 1, 4, 5], dtype=torch.int32, device=dev)   # sequence 1 claims 3 > max 2
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    q = vals["q"].to(dev)
    out2 = torch.full_like(q, float("nan"))
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    pkv.paged_attention_decode_varlen(out2, q, cu, kc, vc, bt, cl, 2, w.scale, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4
    assert torch.equal(out2[0], out[0])           # sequence 0 unaffected
    assert torch.isnan(out2[1:4]).all()           # sequence 1 got no output rows


@pytest.mark.parametrize("kv,Hq,Hkv", [("fp16", 8, 2), ("e5m2", 64, 8)], ids=["mma", "tcgen05"])
def test_varlen_rows_past_q_are_flagged_not_read(orc, dev, gpu, kv, Hq, Hkv):
    """cu_q_lens that send a sequence's rows past the end of q: the sequence is
    flagged and gets no output, the others are unaffected. q and out are the first
    rows of larger buffers, so even a missed check would stay inside memory; the
    rows past the view must come back untouched."""
    import paged_kv_cache_252_gb300 as pkv
    q_lens = [2, 4, 3]
    w = wl.custom(num_seqs=3, num_q_heads=Hq, num_kv_heads=Hkv, head_size=128, q_per_seq=4,
                  kv_dtype=kv, context_lens=[40, 70, 33], seed=12, q_lens=q_lens)
    vals = wl.token_values(w)
    kc, vc, out = gpu.cuda_path(w, vals, dev)        # all 9 rows, the reference for rows 0..5
    qbuf = torch.zeros(12, Hq, 128, dtype=torch.float16, device=dev)
    qbuf[:9] = vals["q"].to(dev)
    obuf = torch.full_like(qbuf, float("nan"))
    q7, o7 = qbuf[:7], obuf[:7]                      # sequence 2 owns rows 6..8: past row 7
    cu = torch.from_numpy(w.cu_q_lens()).to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode_varlen(o7, q7, cu, kc, vc, bt, cl, 4, w.scale, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4
    assert torch.equal(obuf[:6], out[:6])            # sequences 0 and 1 as in the full call
    assert torch.isnan(obuf[6:]).all()               # nothing written for sequence 2 or past the view


# ------------------------------------------------------------------------------------
# token-tree verify
# ------------------------------------------------------------------------------------

TREES = [
    # (kv, D, Hq, Hkv, q_lens or uniform n)
    ("e5m2", 128, 64, 8, 4),
    ("fp16", 128, 32, 8, [5, 1, 8, 3, 2]),
    ("bf16", 64, 8, 4, [16, 3, 9]),
    ("fp16", 64, 4, 4, 16),
    # two row groups, with sequences whose rows fit one group
    ("fp16", 128, 32, 8, [4, 1, 2, 1, 3]),
    ("bf16", 64, 12, 4, [1, 2, 4, 3, 1]),
]


def _tree_id(c):
    n = c[4] if isinstance(c[4], int) else max(c[4])
    return f"{c[0]}-D{c[1]}-G{c[2] // c[3]}-n{n}"


@pytest.mark.parametrize("case", TREES, ids=[_tree_id(c) for c in TREES])
def test_tree_verify_parity(orc, dev, gpu, case):
    import paged_kv_cache_252_gb300 as pkv
    kv, D, Hq, Hkv, ql = case
    S = 5 if isinstance(ql, int) else len(ql)
    q_lens = [ql] * S if isinstance(ql, int) else ql
    lens = [max(l, n) for l, n in zip([20, 1, 300, 33, 1200], q_lens)]
    w = wl.custom(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, q_per_seq=max(q_lens),
                  kv_dtype=kv, context_lens=lens, seed=500 + D, q_lens=None if isinstance(ql, int) else q_lens)
    masks = wl.random_tree_masks(q_lens, seed=11 + D)
    vals = wl.token_values(w)
    kc, vc, _ = gpu.cuda_path(w, vals, dev)
    q = vals["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    tm = torch.from_numpy(masks.view(np.int64)).to(dev)
    cu = torch.from_numpy(w.cu_q_lens()).to(dev) if w.q_lens is not None else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode_tree(out, q, tm, kc, vc, bt, cl, w.q_per_seq, w.scale, cu_q_lens=cu,
                                    device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    okc, ovc = gpu.oracle_caches(orc, w, vals)
    kw = {"tree_masks": masks}
    if w.q_lens is None:
        kw["cu_q_lens"] = w.cu_q_lens()
    ref, _, rc = gpu.oracle_attention(orc, w, vals, okc, ovc, **kw)
    assert rc == 0
    gpu.compare(out, ref, label=f"tree {kv} D{D} G{Hq // Hkv} q_lens {q_lens}")


def test_workspace_left_holding_small_integers_gives_the_same_output(dev, gpu):
    """A workspace reused after holding other data (here every int32 value 0..4095,
    as block ids or lengths would leave it) decodes exactly as a zeroed one: the
    piece counters' per-call tags do not look like small integers."""
    import paged_kv_cache_252_gb300 as pkv
    w = wl.custom(num_seqs=8, num_q_heads=32, num_kv_heads=8, head_size=128, q_per_seq=1, kv_dtype="fp16",
                  context_lens=[3000, 17, 2500, 900, 1, 4000, 64, 1200], seed=31)
    vals = wl.token_values(w)
    kc, vc, ref = gpu.cuda_path(w, vals, dev)
    q = vals["q"].to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    need = pkv.decode_workspace_bytes(w.num_seqs, w.num_q_heads, 1, kc)
    for _ in range(3):
        ws = (torch.arange(need // 4 + 1, dtype=torch.int32, device=dev) % 4096).view(torch.uint8)
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, 1, w.scale, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
