"""Pins for the CPU oracle: checks against what the formats, the mathematics and
library routines fix, never against the oracle itself.

Pages followed: "AI大模型推理速度翻倍，Colossal-Inference开源发布" (分块式KV缓存,
KV缓存量化, 分页注意力算法, 投机采样) and "AI 大模型推理优化技术详解" (2.1.2 Paged
Attention, 2.2.2 GQA).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from paged_kv_cache_252_gb300 import workloads as wl
from _helpers import (bits16, oracle_caches, oracle_attention, sdpa_reference, KV_CODE,
                      cache_shape)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


# ---------------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------------

def _e5m2_code_values():
    """The 256 E5M2 codes decoded from the format definition (numpy, independent)."""
    b = np.arange(256)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 2) & 0x1F
    m = b & 0x3
    mag = np.where(e == 0, m * 2.0 ** -16, (1 + m / 4.0) * 2.0 ** (e.astype(np.float64) - 15))
    mag = np.where(e == 31, np.where(m == 0, np.inf, np.nan), mag)
    return sign * mag


def _nearest_e5m2(x: np.ndarray) -> np.ndarray:
    """Nearest finite E5M2 code by exhaustive search; ties to the even code; beyond the
    largest finite magnitude (and +-inf) saturate; NaN -> 0x7E with the sign bit."""
    vals = _e5m2_code_values()
    finite = np.isfinite(vals)
    codes = np.arange(256)[finite]
    cv = vals[finite]
    out = np.zeros(x.shape, dtype=np.uint8)
    sign = np.signbit(x)
    nan = np.isnan(x)
    xs = np.where(nan, 0.0, np.clip(x, -57344.0, 57344.0))  # saturate (covers inf)
    dist = np.abs(xs[:, None] - cv[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among tied candidates prefer an even mantissa code; for +-0 prefer the input's sign
    score = cand * (2 + (codes[None, :] % 2 == 0) * 2 + (np.signbit(cv)[None, :] == sign[:, None]))
    out = codes[np.argmax(score, axis=1)].astype(np.uint8)
    out = np.where(nan, np.where(sign, 0xFE, 0x7E), out).astype(np.uint8)
    return out


def test_e5m2_exhaustive_vs_nearest_code_search(orc):
    x = ALL16.view(np.float16).astype(np.float64)
    got = orc.e5m2_from_fp16(ALL16)
    want = _nearest_e5m2(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(int(ALL16[i])), hex(int(got[i])), hex(int(want[i]))) for i in bad[:8]]


def test_e5m2_matches_torch_cast_in_range(orc):
    """torch's float8_e5m2 cast (round-to-nearest-even, no saturation) agrees on every
    finite fp16 value below the overflow threshold 61440."""
    x16 = torch.from_numpy(ALL16.view(np.int16)).view(torch.float16)
    finite = torch.isfinite(x16) & (x16.abs() < 61440)
    t = x16[finite].to(torch.float8_e5m2).view(torch.uint8).numpy()
    got = orc.e5m2_from_fp16(ALL16[finite.numpy()])
    assert np.array_equal(got, t)


def test_e5m2_roundtrip_and_bit_identity(orc):
    vals = _e5m2_code_values()
    for b in range(256):
        h = orc.fp16_from_e5m2(b)
        if np.isnan(vals[b]):
            continue
        # the fp16 pattern of an E5M2 value is the byte followed by 8 zero bits
        assert h == (b << 8), (b, h)
        assert orc.e5m2_to_f64(b) == vals[b]
        back = int(orc.e5m2_from_fp16(np.array([h], np.uint16))[0])
        if np.isinf(vals[b]):
            assert back == (b & 0x80) | 0x7B   # infinities saturate (satfinite reading)
        else:
            assert back == b


def test_e5m2_golden_cases(orc):
    """Hand-worked cases (tests/golden/e5m2_cases.json): ties, subnormals, saturation, NaN."""
    with open(os.path.join(GOLDEN, "e5m2_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        h = int(c["fp16"], 16)
        got = int(orc.e5m2_from_fp16(np.array([h], np.uint16))[0])
        assert got == int(c["e5m2"], 16), (c, hex(got))


def test_fp16_bf16_decode_exhaustive(orc):
    got16 = orc.decode_to_f64(ALL16, orc.FP16)
    ref16 = ALL16.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got16), np.isnan(ref16))
    ok = ~np.isnan(ref16)
    assert np.array_equal(got16[ok], ref16[ok])
    assert np.array_equal(np.signbit(got16[ok]), np.signbit(ref16[ok]))
    gotb = orc.decode_to_f64(ALL16, orc.BF16)
    refb = torch.from_numpy(ALL16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(gotb), np.isnan(refb))
    ok = ~np.isnan(refb)
    assert np.array_equal(gotb[ok], refb[ok])


def test_round_from_f64_fp16_matches_numpy(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 5, 20000),
        # exact halfway points between adjacent fp16 values (ties)
        (ALL16[:0x7BFF].view(np.float16).astype(np.float64)
         + ALL16[1:0x7C00].view(np.float16).astype(np.float64)) / 2.0,
        [65504.0, 65519.99, 65520.0, 1e6, -1e6, 5.96e-8, 2.98e-8, 0.0, -0.0],
    ])
    got = orc.round_from_f64(x, orc.FP16)
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_round_from_f64_bf16_matches_torch(orc):
    rng = np.random.default_rng(1)
    # fp32-representable inputs, so torch's fp32 -> bf16 rounding is a single rounding
    x = (rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000)).astype(np.float32)
    ties = (np.arange(1, 40000, dtype=np.uint32) << 15).view(np.float32)  # bit 15 set: halfway cases
    x = np.concatenate([x, ties, -ties]).astype(np.float64)
    got = orc.round_from_f64(x, orc.BF16)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------------
# cache write
# ---------------------------------------------------------------------------------

@pytest.mark.parametrize("kv", ["fp16", "bf16", "e5m2"])
def test_cache_write_roundtrip_through_block_table(orc, kv):
    """Writing every token through the slot mapping and reading position p back through
    block_tables[s][p // 16] returns the token (cast for E5M2), for every sequence."""
    w = wl.custom(num_seqs=3, num_q_heads=4, num_kv_heads=2, head_size=64, q_per_seq=1,
                  kv_dtype=kv, context_lens=[5, 16, 40], seed=11)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    starts = w.seq_starts()
    kb = bits16(vals["k_all"])
    for s in range(w.num_seqs):
        for p in range(int(w.context_lens[s])):
            blk = w.block_tables[s, p // 16]
            row = kc[blk, :, p % 16, :]
            src = kb[starts[s] + p]
            if kv == "e5m2":
                src = orc.e5m2_from_fp16(src)
            assert np.array_equal(row, src)


def test_cache_write_skips_minus_one_and_flags_out_of_range(orc):
    kc = np.zeros((2, 1, 16, 8), np.uint16)
    vc = np.zeros_like(kc)
    key = np.full((3, 1, 8), 0x3C00, np.uint16)
    rc = orc.kv_cache_write(key, key, orc.FP16, np.array([-1, 3, 31], np.int32), kc, vc, orc.FP16)
    assert rc == 0
    assert kc.reshape(-1, 8)[3].tolist() == [0x3C00] * 8
    assert kc.reshape(-1, 8)[31].tolist() == [0x3C00] * 8
    assert int((kc != 0).sum()) == 16
    rc = orc.kv_cache_write(key, key, orc.FP16, np.array([0, 32, 1], np.int32), kc, vc, orc.FP16)
    assert rc == -1


def test_cache_write_golden_fixture(orc):
    """Two tokens, one KV head, head size 8, written into a 2-block pool as E5M2
    (tests/golden/cache_write_e5m2.json, worked by hand from the format)."""
    with open(os.path.join(GOLDEN, "cache_write_e5m2.json")) as f:
        g = json.load(f)
    key = np.array([[int(x, 16) for x in row] for row in g["key_fp16"]], np.uint16)[:, None, :]
    kc = np.zeros((2, 1, 16, 8), np.uint8)
    vc = np.zeros_like(kc)
    rc = orc.kv_cache_write(key, key, orc.FP16, np.array(g["slot_mapping"], np.int32), kc, vc,
                            orc.E5M2)
    assert rc == 0
    for slot, row in zip(g["slot_mapping"], g["expect_e5m2"]):
        assert kc.reshape(-1, 8)[slot].tolist() == [int(x, 16) for x in row]


# ---------------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------------

CASES = [
    # (kv, S, Hq, Hkv, D, n, lens)
    ("fp16", 4, 4, 2, 64, 1, [1, 17, 33, 64]),
    ("bf16", 3, 8, 2, 64, 1, [15, 16, 47]),
    ("e5m2", 3, 8, 8, 128, 1, [2, 31, 70]),
    ("fp16", 2, 8, 1, 64, 1, [20, 50]),
    ("e5m2", 3, 8, 2, 64, 4, [4, 19, 40]),
    ("fp16", 2, 4, 4, 64, 3, [3, 33]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-G{c[2] // c[3]}-n{c[5]}" for c in CASES])
def test_attention_matches_torch_sdpa_dense(orc, case):
    kv, S, Hq, Hkv, D, n, lens = case
    w = wl.custom(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, q_per_seq=n,
                  kv_dtype=kv, context_lens=lens, seed=31 + S + n)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, rc = oracle_attention(orc, w, vals, kc, vc)
    assert rc == 0
    for s in range(S):
        ref = sdpa_reference(w, vals, s)
        got = out[s * n:(s + 1) * n]
        np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_tiny_workload_matches_sdpa(orc):
    w = wl.tiny()
    assert w.num_blocks == 32 and int(((w.context_lens + 15) // 16).sum()) == 10
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, rc = oracle_attention(orc, w, vals, kc, vc)
    assert rc == 0
    for s in range(w.num_seqs):
        np.testing.assert_allclose(out[s:s + 1], sdpa_reference(w, vals, s), rtol=1e-10, atol=1e-12)


def test_block_permutation_invariance(orc):
    """Moving every physical block elsewhere in the pool (and re-pointing the block table)
    leaves the output bit-for-bit unchanged."""
    w = wl.custom(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=64, q_per_seq=2,
                  kv_dtype="e5m2", context_lens=[9, 40, 77], seed=5)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    out1, _, _ = oracle_attention(orc, w, vals, kc, vc)
    perm = np.random.default_rng(3).permutation(w.num_blocks)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt = w.block_tables.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    q = bits16(vals["q"])
    out2, _, rc = orc.paged_attention(q, 0, w.q_per_seq, kc2, vc2, KV_CODE["e5m2"], bt,
                                      w.context_lens, w.scale)
    assert rc == 0
    assert np.array_equal(out1, out2)


def test_weights_sum_to_one_and_respect_causality(orc):
    w = wl.custom(num_seqs=3, num_q_heads=4, num_kv_heads=2, head_size=64, q_per_seq=4,
                  kv_dtype="fp16", context_lens=[4, 21, 64], seed=9)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    _, wts, rc = oracle_attention(orc, w, vals, kc, vc, want_weights=True)
    assert rc == 0
    sums = wts.sum(axis=-1)
    assert np.max(np.abs(sums - 1.0)) <= 1e-12
    for s in range(w.num_seqs):
        ctx = int(w.context_lens[s])
        for j in range(w.q_per_seq):
            row = wts[s * w.q_per_seq + j]
            assert np.all(row[:, ctx - w.q_per_seq + j + 1:] == 0.0)
            assert np.all(row[:, :ctx - w.q_per_seq + j + 1] > 0.0)


@pytest.mark.parametrize("kv", ["fp16", "bf16", "e5m2"])
def test_single_token_context_returns_v(orc, kv):
    """ctx = 1: the only weight is exactly 1, so the output is V itself (dequantised)."""
    w = wl.custom(num_seqs=2, num_q_heads=4, num_kv_heads=2, head_size=64, q_per_seq=1,
                  kv_dtype=kv, context_lens=[1, 1], seed=4)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, rc = oracle_attention(orc, w, vals, kc, vc)
    assert rc == 0
    for s in range(2):
        blk = w.block_tables[s, 0]
        v = orc.decode_to_f64(vc[blk, :, 0, :], KV_CODE[kv])   # [Hkv, D]
        want = np.repeat(v, w.group, axis=0)
        assert np.array_equal(out[s], want)


def test_gqa_group_equals_replicated_mha(orc):
    """GQA-G equals MHA on a cache where KV head hq // G is copied to every query head
    (the grouping reading: contiguous query heads share a KV head)."""
    G, Hkv, D = 4, 2, 64
    w = wl.custom(num_seqs=2, num_q_heads=G * Hkv, num_kv_heads=Hkv, head_size=D, q_per_seq=2,
                  kv_dtype="bf16", context_lens=[18, 50], seed=21)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, _ = oracle_attention(orc, w, vals, kc, vc)
    kc_m = np.repeat(kc, G, axis=1)
    vc_m = np.repeat(vc, G, axis=1)
    out_m, _, rc = orc.paged_attention(bits16(vals["q"]), 1, 2, kc_m, vc_m, KV_CODE["bf16"],
                                       w.block_tables, w.context_lens, w.scale)
    assert rc == 0
    assert np.array_equal(out, out_m)


def test_gqa_one_is_mqa_and_gqa_h_is_mha(orc):
    """GQA-1 (one KV head) = MQA: every query head attends to the same K/V, so its output
    equals a one-head run of that head's query. GQA-H (G = 1) = MHA: head h equals a
    one-head run on KV head h alone."""
    for Hkv in (1, 4):
        w = wl.custom(num_seqs=2, num_q_heads=4, num_kv_heads=Hkv, head_size=64, q_per_seq=1,
                      kv_dtype="fp16", context_lens=[7, 35], seed=40 + Hkv)
        vals = wl.token_values(w)
        kc, vc = oracle_caches(orc, w, vals)
        out, _, _ = oracle_attention(orc, w, vals, kc, vc)
        q = bits16(vals["q"])
        for hq in range(4):
            h = hq // w.group
            o1, _, rc = orc.paged_attention(np.ascontiguousarray(q[:, hq:hq + 1]), 0, 1,
                                            np.ascontiguousarray(kc[:, h:h + 1]),
                                            np.ascontiguousarray(vc[:, h:h + 1]), 0,
                                            w.block_tables, w.context_lens, w.scale)
            assert rc == 0
            assert np.array_equal(out[:, hq:hq + 1], o1)


def test_spec_verify_row_equals_shorter_single_token_decode(orc):
    """Query token j of an n-token verify equals a one-token decode whose context ends at
    position ctx - n + j."""
    n = 4
    w = wl.custom(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=64, q_per_seq=n,
                  kv_dtype="e5m2", context_lens=[4, 20, 63], seed=12)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, _ = oracle_attention(orc, w, vals, kc, vc)
    q = bits16(vals["q"])
    for j in range(n):
        qj = np.ascontiguousarray(q.reshape(w.num_seqs, n, 8, 64)[:, j])
        lens = (w.context_lens - n + j + 1).astype(np.int32)
        o1, _, rc = orc.paged_attention(qj, 0, 1, kc, vc, 2, w.block_tables, lens, w.scale)
        assert rc == 0
        assert np.array_equal(out.reshape(w.num_seqs, n, 8, 64)[:, j], o1)


def test_zero_scale_gives_mean_of_v(orc):
    w = wl.custom(num_seqs=2, num_q_heads=4, num_kv_heads=2, head_size=64, q_per_seq=2,
                  kv_dtype="fp16", context_lens=[5, 30], seed=2, scale=0.0)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, _ = oracle_attention(orc, w, vals, kc, vc)
    starts = w.seq_starts()
    v = vals["v_all"].to(torch.float64).numpy()
    for s in range(2):
        ctx = int(w.context_lens[s])
        for j in range(2):
            lim = ctx - 2 + j + 1
            mean = v[starts[s]:starts[s] + lim].mean(axis=0)   # [Hkv, D]
            want = np.repeat(mean, w.group, axis=0)
            np.testing.assert_allclose(out[s * 2 + j], want, rtol=1e-13, atol=1e-15)


def test_bad_block_id_is_reported(orc):
    w = wl.custom(num_seqs=1, num_q_heads=2, num_kv_heads=1, head_size=64, q_per_seq=1,
                  kv_dtype="fp16", context_lens=[20], seed=2)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    bt = w.block_tables.copy()
    bt[0, 1] = w.num_blocks  # out of range
    _, _, rc = orc.paged_attention(bits16(vals["q"]), 0, 1, kc, vc, 0, bt, w.context_lens, w.scale)
    assert rc == -1


def test_threads_do_not_change_results(orc):
    w = wl.custom(num_seqs=5, num_q_heads=8, num_kv_heads=2, head_size=64, q_per_seq=2,
                  kv_dtype="bf16", context_lens=[3, 17, 33, 64, 90], seed=8)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    o1, _, _ = oracle_attention(orc, w, vals, kc, vc, num_threads=1)
    o4, _, _ = oracle_attention(orc, w, vals, kc, vc, num_threads=4)
    assert np.array_equal(o1, o4)


# ---------------------------------------------------------------------------------
# mixed batches: per-sequence query-token counts, packed without padding
# ---------------------------------------------------------------------------------

def test_varlen_matches_sdpa_and_per_sequence_runs(orc):
    """A packed mixed batch (1..5 query tokens per sequence) equals torch SDPA per
    sequence, and each sequence's rows equal a uniform run with its own token count."""
    q_lens = [1, 5, 2, 1, 3]
    w = wl.custom(num_seqs=5, num_q_heads=8, num_kv_heads=2, head_size=64, q_per_seq=5,
                  kv_dtype="e5m2", context_lens=[7, 40, 16, 1, 90], seed=17, q_lens=q_lens)
    vals = wl.token_values(w)
    assert vals["q"].shape[0] == sum(q_lens)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, rc = oracle_attention(orc, w, vals, kc, vc)
    assert rc == 0
    cu = w.cu_q_lens()
    q = bits16(vals["q"])
    for s in range(w.num_seqs):
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], sdpa_reference(w, vals, s), rtol=1e-10, atol=1e-12)
        one, _, rc = orc.paged_attention(np.ascontiguousarray(q[cu[s]:cu[s + 1]]), 0, q_lens[s], kc, vc,
                                         KV_CODE["e5m2"], w.block_tables[s:s + 1], w.context_lens[s:s + 1],
                                         w.scale)
        assert rc == 0
        assert np.array_equal(out[cu[s]:cu[s + 1]], one)


def test_long_query_chunks_are_causal_past_64_tokens(orc):
    """Prefill chunks longer than 64 tokens mixed with decodes: every query token j
    sees positions <= ctx - n + j, however far past the 64th draft position (SDPA with
    the explicit causal mask is the reference)."""
    q_lens = [1, 150, 3, 70]
    w = wl.custom(num_seqs=4, num_q_heads=4, num_kv_heads=2, head_size=64, q_per_seq=150,
                  kv_dtype="fp16", context_lens=[9, 230, 40, 70], seed=61, q_lens=q_lens)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, rc = oracle_attention(orc, w, vals, kc, vc)
    assert rc == 0
    cu = w.cu_q_lens()
    for s in range(w.num_seqs):
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], sdpa_reference(w, vals, s), rtol=1e-10, atol=1e-12)


def test_varlen_with_equal_counts_is_the_uniform_batch(orc):
    w = wl.custom(num_seqs=3, num_q_heads=4, num_kv_heads=2, head_size=64, q_per_seq=2,
                  kv_dtype="fp16", context_lens=[5, 33, 18], seed=23)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    uni, _, _ = oracle_attention(orc, w, vals, kc, vc)
    var, _, rc = oracle_attention(orc, w, vals, kc, vc, cu_q_lens=np.array([0, 2, 4, 6], np.int32))
    assert rc == 0
    assert np.array_equal(uni, var)


# ---------------------------------------------------------------------------------
# token-tree verify (FlexFlow Serve, token-tree verification)
# ---------------------------------------------------------------------------------

def test_tree_masks_match_sdpa_with_the_tree_mask(orc):
    q_lens = [4, 6, 1, 3]
    w = wl.custom(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_size=64, q_per_seq=6,
                  kv_dtype="fp16", context_lens=[10, 40, 5, 17], seed=44, q_lens=q_lens)
    vals = wl.token_values(w)
    masks = wl.random_tree_masks(q_lens, seed=7)
    kc, vc = oracle_caches(orc, w, vals)
    out, _, rc = oracle_attention(orc, w, vals, kc, vc, tree_masks=masks)
    assert rc == 0
    cu = w.cu_q_lens()
    for s in range(w.num_seqs):
        ref = sdpa_reference(w, vals, s, tree_masks=masks)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], ref, rtol=1e-10, atol=1e-12)


def test_chain_tree_is_the_causal_verify(orc):
    w = wl.custom(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=64, q_per_seq=4,
                  kv_dtype="bf16", context_lens=[4, 33, 70], seed=45)
    vals = wl.token_values(w)
    kc, vc = oracle_caches(orc, w, vals)
    causal, _, _ = oracle_attention(orc, w, vals, kc, vc)
    chain = np.array([(2 << j) - 1 for _ in range(3) for j in range(4)], dtype=np.uint64)
    tree, _, rc = oracle_attention(orc, w, vals, kc, vc, tree_masks=chain)
    assert rc == 0
    assert np.array_equal(causal, tree)


def test_random_tree_masks_are_ancestor_closed():
    masks = wl.random_tree_masks([7, 1, 5], seed=3)
    off = 0
    for n in (7, 1, 5):
        m = [int(x) for x in masks[off:off + n]]
        for i in range(n):
            assert (m[i] >> i) & 1 and m[i] < (1 << (i + 1))
            for a in range(i):
                if (m[i] >> a) & 1:
                    assert m[a] & m[i] == m[a]     # every ancestor's ancestors are visible too
        off += n


# ---------------------------------------------------------------------------------
# INT8 KV cache (symmetric codes per (token, KV head) row, float32 row scales)
# ---------------------------------------------------------------------------------

def _int8_rows(orc, x16):
    """Quantise fp16 rows x16 [T, Hkv, D] with the oracle's INT8 cache write into
    slots 0..T-1; returns codes [T, Hkv, D] and scales [T, Hkv]."""
    T, Hkv, D = x16.shape
    nb = (T + 15) // 16
    kc = np.zeros((nb, Hkv, 16, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nb, Hkv, 16), np.float32)
    vs = np.zeros_like(ks)
    assert orc.kv_cache_write_int8(x16.view(np.uint16), x16.view(np.uint16), np.arange(T, dtype=np.int32),
                                   kc, vc, ks, vs) == 0
    codes = kc.transpose(0, 2, 1, 3).reshape(nb * 16, Hkv, D)[:T]
    scales = ks.transpose(0, 2, 1).reshape(nb * 16, Hkv)[:T]
    assert np.array_equal(codes, vc.transpose(0, 2, 1, 3).reshape(nb * 16, Hkv, D)[:T])
    return codes, scales


def test_int8_codes_are_nearest_and_span_the_row(orc):
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((40, 3, 64)) * rng.choice([1e-3, 1.0, 300.0], size=(40, 3, 1))).astype(np.float16)
    x[5, 1] = 0.0                                          # an all-zero row
    x[7, 2, 3] = np.float16(-60000.0)                      # one element dominates its row
    codes, scales = _int8_rows(orc, x)
    xf = x.astype(np.float64)
    amax = np.abs(xf).max(axis=2)
    # the scale is max|x| / 127 (a float32 division) rounded up to the nearest fp16 value
    s32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(scales.astype(np.float16).astype(np.float32), scales)   # fp16 values
    assert np.all(scales >= s32)
    below = np.nextafter(scales.astype(np.float16), np.float16(0)).astype(np.float32)
    assert np.all((below < s32) | (scales == 0))                                   # the smallest such
    nz = scales > 0
    ratio = xf / np.where(nz, scales, 1.0)[..., None]
    # each code is the integer nearest x / scale (within the float32 rounding of the ratio)
    assert np.all(np.abs(ratio - codes)[nz] <= 0.5 + 1e-5)
    assert np.all(np.abs(codes) <= 127)
    # the row's largest magnitude maps to +-127, with the element's sign
    i = np.abs(xf).argmax(axis=2)
    top = np.take_along_axis(codes, i[..., None], axis=2)[..., 0]
    sgn = np.sign(np.take_along_axis(xf, i[..., None], axis=2)[..., 0])
    assert np.array_equal(top[nz], (127 * sgn[nz]).astype(np.int8))
    # zero rows: scale 0 and codes 0
    assert scales[5, 1] == 0 and not codes[5, 1].any()
    # reconstruction error is at most half a step
    assert np.all(np.abs(xf - codes * scales[..., None].astype(np.float64)) <= 0.5 * scales[..., None] * (1 + 1e-5))


def test_int8_golden_ties(orc):
    """Hand-worked rows (tests/golden/int8_ties.json) whose x / scale values are exact
    ties: the codes pin round-half-to-even (half away from zero or truncation fail)."""
    with open(os.path.join(GOLDEN, "int8_ties.json")) as f:
        g = json.load(f)
    D = g["head_size"]
    rows = g["rows"]
    x = np.zeros((len(rows), 1, D), np.float16)
    for i, r in enumerate(rows):
        for idx, val, _, _ in r["elements"]:
            x[i, 0, idx] = np.float16(val)
    codes, scales = _int8_rows(orc, x)
    for i, r in enumerate(rows):
        assert scales[i, 0] == np.float32(r["scale"])
        want = np.zeros(D, np.int8)
        for idx, _, code, why in r["elements"]:
            want[idx] = code
            assert codes[i, 0, idx] == code, f"row {i} element {idx}: {why}"
        assert np.array_equal(codes[i, 0], want)


def test_int8_attention_matches_sdpa_on_the_dequantised_cache(orc):
    w = wl.custom(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_size=64, q_per_seq=2, kv_dtype="int8",
                  context_lens=[2, 17, 40, 77], seed=42)
    vals = wl.token_values(w)
    k_all, v_all = bits16(vals["k_all"]), bits16(vals["v_all"])
    slots = vals["slot_all"].numpy().astype(np.int32)
    kc = np.zeros(cache_shape(w), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros(cache_shape(w)[:3], np.float32)
    vs = np.zeros_like(ks)
    assert orc.kv_cache_write_int8(k_all, v_all, slots, kc, vc, ks, vs) == 0
    out, _, rc = orc.paged_attention(bits16(vals["q"]), 0, w.q_per_seq, kc, vc, 3, w.block_tables,
                                     w.context_lens, w.scale, k_scale=ks, v_scale=vs)
    assert rc == 0
    n, G = w.q_per_seq, w.group
    for s in range(w.num_seqs):
        ctx = int(w.context_lens[s])
        p = np.arange(ctx)
        blk = w.block_tables[s][p // 16]
        off = p % 16
        k = torch.from_numpy(kc[blk, :, off, :].astype(np.float64) * ks[blk, :, off][..., None])  # [ctx, Hkv, D]
        v = torch.from_numpy(vc[blk, :, off, :].astype(np.float64) * vs[blk, :, off][..., None])
        q = vals["q"][s * n:(s + 1) * n].to(torch.float64)
        kk = k.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
        vv = v.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
        mask = torch.arange(ctx)[None, :] <= (ctx - n + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(q.permute(1, 0, 2)[None], kk, vv,
                                                               attn_mask=mask, scale=w.scale)
        np.testing.assert_allclose(out[s * n:(s + 1) * n], ref[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
