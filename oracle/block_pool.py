"""Plain Python model of the host block pool — test infrastructure only.

Only tests (and nothing on the product path) import this module. It restates
the rules of the block pool in the plainest data structures, so that every
block id, slot, copy pair and reference count of the C++ allocator in
libpagedkv.so can be checked against it after each operation.

Rules ("AI 大模型推理优化技术详解", 2.1.2 Paged Attention: a table maps each
sequence's logical blocks to physical blocks of a pool allocated up front;
several logical blocks may share a physical block, counted by a reference
count; a block whose count drops to 0 returns to the pool. "TACO-LLM
如何实现降本增效?", 2、使用 Prefix Cache 技术降低 TTFT: earlier prompts' KV kept in
a prefix tree and looked up for a new prompt's matching prefix):
  - a block holds 16 tokens; token p of a sequence is in its block p // 16 at
    offset p % 16; slot = block * 16 + offset;
  - a new block is the lowest-numbered free block; if none is free, the cached
    block that became evictable longest ago is taken out of the tree and used;
  - fork: the child gets the parent's blocks and length (each block +1 ref);
  - append n tokens: if the last block is partly filled, shared (ref > 1) and
    n > 0, it is first replaced by a new block (copy-on-write, reported as a
    (src, dst) pair); then a new block starts at every position p % 16 == 0;
    it fails with nothing changed if the pool cannot supply the blocks;
  - release: every block of the sequence loses one reference;
  - prefix tree: full blocks keyed by (parent cached block or -1, 16 token ids);
    the tree holds one reference per cached block; a cached block is evictable
    when only the tree references it and it has no cached children.
"""
from __future__ import annotations

B = 16
OK, INVALID, OUT_OF_BLOCKS = 0, -1, -6


class BlockPoolModel:
    def __init__(self, num_blocks: int):
        self.n = num_blocks
        self.ref = [0] * num_blocks
        self.free = set(range(num_blocks))
        self.seqs = {}            # id -> [blocks list, length]
        self.cache = {}           # (parent, tokens tuple) -> block
        self.key_of = {}          # cached block -> key
        self.kids = {}            # cached block -> list of cached children
        self.lru = []             # evictable blocks, the longest evictable first

    # ---- reference bookkeeping ------------------------------------------------
    def _evictable(self, b):
        return b in self.key_of and self.ref[b] == 1 and not self.kids.get(b)

    def _update(self, b):
        if self._evictable(b):
            if b not in self.lru:
                self.lru.append(b)
        elif b in self.lru:
            self.lru.remove(b)

    def _inc(self, b):
        self.ref[b] += 1
        self._update(b)

    def _dec(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.add(b)
        else:
            self._update(b)

    def _evict(self, b):
        key = self.key_of.pop(b)
        del self.cache[key]
        if b in self.lru:
            self.lru.remove(b)
        self.kids.pop(b, None)
        parent = key[0]
        if parent >= 0:
            self.kids[parent].remove(b)
            self._update(parent)
        self.ref[b] = 0

    def _take(self):
        if self.free:
            b = min(self.free)
            self.free.remove(b)
        else:
            b = self.lru[0]
            self._evict(b)
        self.ref[b] = 1
        return b

    def _descendants(self, b):
        out, todo = [], list(self.kids.get(b, []))
        while todo:
            x = todo.pop()
            out.append(x)
            todo.extend(self.kids.get(x, []))
        return out

    def available(self):
        """Free blocks plus cached blocks that leaf-by-leaf eviction can free."""
        n = len(self.free)
        for b in self.key_of:
            if self.ref[b] == 1 and all(self.ref[d] == 1 for d in self._descendants(b)):
                n += 1
        return n

    def evictable(self):
        return self.available() - len(self.free)

    # ---- sequences ---------------------------------------------------------------
    def add(self, seq):
        if seq in self.seqs:
            return INVALID
        self.seqs[seq] = [[], 0]
        return OK

    def fork(self, parent, child):
        if parent == child or child in self.seqs or parent not in self.seqs:
            return INVALID
        blocks, length = self.seqs[parent]
        self.seqs[child] = [list(blocks), length]
        for b in blocks:
            self._inc(b)
        return OK

    def release(self, seq):
        if seq not in self.seqs:
            return INVALID
        for b in self.seqs[seq][0]:
            self._dec(b)
        del self.seqs[seq]
        return OK

    def length(self, seq):
        return self.seqs[seq][1] if seq in self.seqs else -1

    def block_table(self, seq):
        return list(self.seqs[seq][0])

    def append(self, seq, n):
        """Returns (status, slots, copies)."""
        if seq not in self.seqs or n < 0:
            return INVALID, [], []
        blocks, length = self.seqs[seq]
        new_len = length + n
        cow = n > 0 and length % B != 0 and self.ref[blocks[-1]] > 1
        need = (new_len + B - 1) // B - (length + B - 1) // B + (1 if cow else 0)
        if need > self.available():
            return OUT_OF_BLOCKS, [], []
        copies = []
        if cow:
            src = blocks[-1]
            dst = self._take()
            self._dec(src)
            blocks[-1] = dst
            copies.append((src, dst))
        slots = []
        for p in range(length, new_len):
            if p % B == 0:
                blocks.append(self._take())
            slots.append(blocks[p // B] * B + p % B)
        self.seqs[seq][1] = new_len
        return OK, slots, copies

    # ---- prefix tree -------------------------------------------------------------
    def prefix_insert(self, seq, tokens):
        if seq not in self.seqs or len(tokens) > self.seqs[seq][1]:
            return INVALID
        blocks = self.seqs[seq][0]
        parent, added = -1, 0
        for k in range(len(tokens) // B):
            key = (parent, tuple(int(t) for t in tokens[k * B:(k + 1) * B]))
            if key in self.cache:
                parent = self.cache[key]
                continue
            b = blocks[k]
            if b in self.key_of:
                break
            self.cache[key] = b
            self.key_of[b] = key
            if parent >= 0:
                self.kids.setdefault(parent, []).append(b)
            self.ref[b] += 1
            self._update(b)
            if parent >= 0:
                self._update(parent)
            parent = b
            added += 1
        return added

    def add_cached(self, seq, tokens):
        """Returns (status, cached tokens)."""
        if seq in self.seqs:
            return INVALID, 0
        hit, parent = [], -1
        for k in range(len(tokens) // B):
            key = (parent, tuple(int(t) for t in tokens[k * B:(k + 1) * B]))
            if key not in self.cache:
                break
            hit.append(self.cache[key])
            parent = self.cache[key]
        self.seqs[seq] = [list(hit), B * len(hit)]
        for b in hit:
            self._inc(b)
        return OK, B * len(hit)
