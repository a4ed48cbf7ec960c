"""Host block pool: the C++ allocator in libpagedkv.so against the plain model
in oracle/block_pool.py (every block id, slot, copy pair and reference count
after every operation), the model against hand-worked cases, and invariants.
No GPU needed."""
import numpy as np
import pytest

from oracle.block_pool import B, BlockPoolModel, INVALID, OK, OUT_OF_BLOCKS


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_252_gb300 as pkv
    return pkv


# ---- the model against hand-worked cases ------------------------------------------

def test_model_append_fork_copy_on_write_by_hand():
    m = BlockPoolModel(6)
    assert m.add(1) == OK
    st, slots, copies = m.append(1, 20)            # blocks 0 (full) and 1 (4 tokens)
    assert (st, copies) == (OK, []) and slots == list(range(20))
    assert m.block_table(1) == [0, 1] and m.ref[:3] == [1, 1, 0]
    assert m.fork(1, 2) == OK                      # both blocks shared
    assert m.ref[:2] == [2, 2]
    st, slots, copies = m.append(2, 3)             # last block shared, partly filled: copy it
    assert copies == [(1, 2)] and slots == [2 * B + 4, 2 * B + 5, 2 * B + 6]
    assert m.block_table(2) == [0, 2] and m.ref[:3] == [2, 1, 1]
    st, slots, copies = m.append(1, 12)            # block 1 now exclusive to seq 1: no copy
    assert copies == [] and slots[:12] == [B + 4 + i for i in range(12)]
    st, slots, copies = m.append(1, 1)             # position 32 opens block 3
    assert slots == [3 * B] and m.block_table(1) == [0, 1, 3]
    assert m.release(1) == OK                      # blocks 1, 3 free; 0 still held by seq 2
    assert m.ref[:4] == [1, 0, 1, 0] and sorted(m.free) == [1, 3, 4, 5]


def test_model_prefix_tree_and_eviction_order_by_hand():
    m = BlockPoolModel(3)
    toks = list(range(100, 140))                   # 40 tokens: 2 full blocks + 8
    m.add(1)
    m.append(1, 40)                                # blocks 0, 1, 2
    assert m.prefix_insert(1, toks) == 2           # blocks 0 and 1 cached (1 is 0's child)
    assert m.ref == [2, 2, 1]
    m.release(1)                                   # 0 and 1 held by the tree only, 2 free
    assert m.ref == [1, 1, 0] and m.free == {2} and m.lru == [1]   # only the leaf is evictable
    assert m.available() == 3
    st, cached = m.add_cached(2, toks[:35])        # both cached blocks match
    assert (st, cached) == (OK, 32) and m.block_table(2) == [0, 1] and m.lru == []
    m.release(2)
    assert m.lru == [1]
    m.add(3)
    st, slots, _ = m.append(3, 33)                 # needs 3 blocks: free 2, then evict 1, then 0
    assert st == OK and m.block_table(3) == [2, 1, 0] and m.cache == {}
    assert slots[0] == 2 * B and slots[16] == 1 * B and slots[32] == 0


def test_model_out_of_blocks_changes_nothing():
    m = BlockPoolModel(2)
    m.add(1)
    m.append(1, 20)
    before = (list(m.ref), set(m.free), m.block_table(1), m.length(1))
    assert m.append(1, 13)[0] == OUT_OF_BLOCKS     # 33 tokens need 3 blocks
    assert (list(m.ref), set(m.free), m.block_table(1), m.length(1)) == before
    assert m.add(1) == INVALID and m.fork(7, 8) == INVALID and m.release(9) == INVALID


# ---- the C++ allocator against the model ---------------------------------------------

def _state(a, m, ids):
    assert a.free_blocks() == len(m.free)
    assert a.evictable() == m.evictable()
    assert [a.refcount(b) for b in range(m.n)] == m.ref
    for s in ids:
        assert a.length(s) == m.length(s)
        if s in m.seqs:
            assert a.block_table(s) == m.block_table(s)


def _random_ops(pkv, seed, num_blocks, steps):
    rng = np.random.default_rng(seed)
    a = pkv.BlockAllocator(num_blocks)
    m = BlockPoolModel(num_blocks)
    prompts = {}                                   # seq -> token ids written so far
    vocab = 2                                      # tiny vocabulary: prefixes repeat
    next_id = 1
    for _ in range(steps):
        live = sorted(m.seqs)
        op = rng.choice(["add", "add_cached", "fork", "append", "release", "insert"],
                        p=[0.08, 0.16, 0.12, 0.34, 0.16, 0.14])
        if op in ("add", "add_cached") or not live:
            s = next_id
            next_id += 1
            if op == "add_cached" and live:
                base = prompts[live[int(rng.integers(len(live)))]]
                toks = base[:int(rng.integers(0, len(base) + 1))]
                st, got = m.add_cached(s, toks)
                assert a.add_cached(s, toks) == got and st == OK
                prompts[s] = list(toks[:got])
            else:
                assert m.add(s) == OK
                a.add(s)
                prompts[s] = []
        elif op == "fork":
            p = live[int(rng.integers(len(live)))]
            c = next_id
            next_id += 1
            assert m.fork(p, c) == OK
            a.fork(p, c)
            prompts[c] = list(prompts[p])
        elif op == "append":
            s = live[int(rng.integers(len(live)))]
            n = int(rng.integers(0, 24))
            st, slots, copies = m.append(s, n)
            if st == OUT_OF_BLOCKS:
                with pytest.raises(pkv.PagedKVError):
                    a.append(s, n)
            else:
                got_slots, got_copies = a.append(s, n)
                assert got_slots == slots and got_copies == copies
                prompts[s] += [int(x) for x in rng.integers(0, vocab, size=n)]
        elif op == "release":
            s = live[int(rng.integers(len(live)))]
            assert m.release(s) == OK
            a.release(s)
            prompts.pop(s)
        else:
            s = live[int(rng.integers(len(live)))]
            toks = prompts[s][:int(rng.integers(0, len(prompts[s]) + 1))]
            assert a.prefix_insert(s, toks) == m.prefix_insert(s, toks)
        _state(a, m, list(range(1, next_id)))
        # invariants of the model itself
        held = [0] * num_blocks
        for blocks, length in m.seqs.values():
            assert len(blocks) == (length + B - 1) // B
            for b in blocks:
                held[b] += 1
        for b in m.key_of:
            held[b] += 1
        assert held == m.ref
        assert all((m.ref[b] == 0) == (b in m.free) for b in range(num_blocks))
    a.close()


@pytest.mark.parametrize("seed", range(6))
def test_allocator_matches_model_on_random_operations(pkv, seed):
    _random_ops(pkv, seed, num_blocks=[8, 24, 64][seed % 3], steps=500)


def test_allocator_rejects_bad_calls_without_changes(pkv):
    a = pkv.BlockAllocator(2)
    a.add(1)
    a.append(1, 20)
    before = (a.free_blocks(), a.block_table(1), a.length(1), [a.refcount(b) for b in range(2)])
    with pytest.raises(pkv.PagedKVError, match="block pool exhausted"):
        a.append(1, 13)
    with pytest.raises(pkv.PagedKVError):
        a.add(1)
    with pytest.raises(pkv.PagedKVError):
        a.fork(5, 6)
    with pytest.raises(pkv.PagedKVError):
        a.release(5)
    with pytest.raises(pkv.PagedKVError):
        a.prefix_insert(1, list(range(21)))     # more tokens than the sequence holds
    assert (a.free_blocks(), a.block_table(1), a.length(1), [a.refcount(b) for b in range(2)]) == before
    assert a.refcount(-1) == -1 and a.refcount(2) == -1 and a.length(99) == -1
