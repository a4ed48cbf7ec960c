"""The seeded input generator: deterministic, and the block pool is a valid
logical-to-physical map (each used physical block owned by exactly one sequence)."""
import numpy as np
import pytest

from paged_kv_cache_252_gb300 import workloads as wl


@pytest.mark.parametrize("key", list(wl.NAMED))
def test_named_workloads_are_deterministic_and_valid(key):
    a, b = wl.by_name(key), wl.by_name(key)
    assert np.array_equal(a.context_lens, b.context_lens)
    assert np.array_equal(a.block_tables, b.block_tables)
    nb = (a.context_lens.astype(np.int64) + 15) // 16
    used = np.concatenate([a.block_tables[s, :k] for s, k in enumerate(nb)])
    assert used.size == len(np.unique(used))           # no physical block shared
    assert used.min() >= 0 and used.max() < a.num_blocks
    for s, k in enumerate(nb):
        assert np.all(a.block_tables[s, k:] == -1)
    assert a.context_lens.min() >= a.q_per_seq


def test_shapes_of_the_five_workloads():
    t = wl.tiny()
    assert list(t.context_lens) == [1, 17, 33, 64] and t.num_blocks == 32 and t.head_size == 64
    e = wl.llama3_8b_bs64_fp16()
    assert e.num_seqs == 64 and e.group == 4 and 512 <= e.context_lens.min() and e.context_lens.max() <= 2048
    assert abs(e.num_blocks - 1.25 * ((e.context_lens + 15) // 16).sum()) <= 1
    f = wl.llama3_8b_bs256_e5m2()
    assert f.num_seqs == 256 and f.kv_dtype == "e5m2" and 1024 <= f.context_lens.min()
    g = wl.long_bs8_bf16()
    assert g.num_seqs == 8 and g.kv_dtype == "bf16" and g.context_lens.min() >= 32768
    h = wl.llama3_70b_spec4_e5m2()
    assert h.group == 8 and h.q_per_seq == 4 and h.context_lens.min() >= 4 and h.context_lens.max() <= 16384
    assert 700 < np.median(h.context_lens) < 1400


def test_slot_mapping_follows_block_table():
    w = wl.custom(num_seqs=3, num_q_heads=2, num_kv_heads=1, head_size=64, q_per_seq=2,
                  kv_dtype="fp16", context_lens=[2, 16, 35], seed=3)
    slots = w.slot_mapping_all()
    starts = w.seq_starts()
    for s in range(3):
        for p in range(int(w.context_lens[s])):
            assert slots[starts[s] + p] == w.block_tables[s, p // 16] * 16 + p % 16
    assert len(np.unique(slots)) == slots.size
    assert list(w.new_token_index()) == [0, 1, 16, 17, 51, 52]


def test_values_are_seeded():
    w = wl.tiny()
    a, b = wl.token_values(w), wl.token_values(w)
    assert (a["k_all"] == b["k_all"]).all() and (a["q"] == b["q"]).all()
    assert a["k_all"].shape == (115, 2, 64) and a["q"].shape == (4, 4, 64)
