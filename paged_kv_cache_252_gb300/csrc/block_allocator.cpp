// Host-side block pool for the paged KV cache (declared in include/pagedkv.h).
//
// "AI 大模型推理优化技术详解", 2.1.2 Paged Attention: a sequence's KV cache is a
// list of fixed-size blocks taken from a pool allocated up front; a table maps
// its logical blocks to physical ones; several logical blocks may share one
// physical block, counted by a reference count, and a block whose count drops to
// 0 returns to the pool. "TACO-LLM 如何实现降本增效?", 2、使用 Prefix Cache 技术降低
// TTFT: the KV of earlier prompts is kept in a prefix tree, so a new prompt's
// matching prefix is looked up instead of recomputed.
//
// Here: reference counts per block; fork (sharing) with copy-on-write of a
// shared last block on append; and a prefix tree of full blocks keyed by
// (parent block, the block's 16 token ids). The tree holds one reference to
// each cached block. A cached block that only the tree references and that has
// no cached children is evictable; when the pool has no free block the least
// recently evictable one is reused. Choices are deterministic (lowest free block
// first) so that a plain model of the same rules reproduces every block id.
#include <array>
#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

constexpr int32_t kTokensPerBlock = 16;

struct PrefixKey {
  int32_t parent;                            // cached parent block, -1 at the root
  std::array<int32_t, kTokensPerBlock> tok;  // the block's token ids
  bool operator==(const PrefixKey& o) const { return parent == o.parent && tok == o.tok; }
};

struct PrefixKeyHash {
  size_t operator()(const PrefixKey& k) const {
    uint64_t h = 1469598103934665603ull;     // FNV-1a over the key's 17 words
    auto mix = [&h](uint32_t w) {
      for (int i = 0; i < 4; ++i) {
        h ^= (w >> (8 * i)) & 0xffu;
        h *= 1099511628211ull;
      }
    };
    mix(static_cast<uint32_t>(k.parent));
    for (int32_t t : k.tok) mix(static_cast<uint32_t>(t));
    return static_cast<size_t>(h);
  }
};

struct Seq {
  std::vector<int32_t> blocks;
  int32_t len = 0;
};

int32_t blocks_for(int64_t tokens) {
  return static_cast<int32_t>((tokens + kTokensPerBlock - 1) / kTokensPerBlock);
}

}  // namespace

struct pkv_allocator {
  int32_t n = 0;
  std::vector<int32_t> ref;
  std::set<int32_t> free;
  std::unordered_map<int64_t, Seq> seqs;

  std::unordered_map<PrefixKey, int32_t, PrefixKeyHash> cache;
  std::vector<char> cached;
  std::vector<PrefixKey> key_of;
  std::vector<std::vector<int32_t>> kids;    // cached children of a cached block
  std::list<int32_t> lru;                    // evictable blocks, least recent first
  std::vector<std::list<int32_t>::iterator> lru_pos;
  std::vector<char> in_lru;

  bool evictable(int32_t b) const { return cached[b] && ref[b] == 1 && kids[b].empty(); }

  void update_lru(int32_t b) {
    const bool want = evictable(b);
    if (want && !in_lru[b]) {
      lru_pos[b] = lru.insert(lru.end(), b);
      in_lru[b] = 1;
    } else if (!want && in_lru[b]) {
      lru.erase(lru_pos[b]);
      in_lru[b] = 0;
    }
  }

  void inc_ref(int32_t b) {
    ++ref[b];
    update_lru(b);
  }

  void dec_ref(int32_t b) {
    if (--ref[b] == 0) {
      free.insert(b);
    } else {
      update_lru(b);
    }
  }

  // Removes an evictable block from the tree; it is then unreferenced.
  void evict(int32_t b) {
    const PrefixKey key = key_of[b];
    cache.erase(key);
    cached[b] = 0;
    if (in_lru[b]) {
      lru.erase(lru_pos[b]);
      in_lru[b] = 0;
    }
    if (key.parent >= 0) {
      std::vector<int32_t>& k = kids[key.parent];
      for (size_t i = 0; i < k.size(); ++i) {
        if (k[i] == b) {
          k.erase(k.begin() + static_cast<std::ptrdiff_t>(i));
          break;
        }
      }
      update_lru(key.parent);
    }
    ref[b] = 0;
  }

  // A block for a new use (reference count 1); -1 if none is free or evictable.
  int32_t take_block() {
    int32_t b;
    if (!free.empty()) {
      b = *free.begin();
      free.erase(free.begin());
    } else if (!lru.empty()) {
      b = lru.front();
      evict(b);
    } else {
      return -1;
    }
    ref[b] = 1;
    return b;
  }

  // Blocks the pool can supply: the free ones, plus every cached block that only
  // the tree references and none of whose cached descendants anything else
  // references (evicting leaves one after another frees exactly these).
  int64_t available() const {
    int64_t avail = static_cast<int64_t>(free.size());
    if (cache.empty()) return avail;
    std::vector<char> pinned_below(static_cast<size_t>(n), 0);
    for (const auto& kv : cache) {
      const int32_t b = kv.second;
      if (ref[b] == 1) continue;
      // b is held by a sequence: it and its ancestors cannot be evicted.
      for (int32_t x = key_of[b].parent; x >= 0 && !pinned_below[x]; x = key_of[x].parent) pinned_below[x] = 1;
    }
    for (const auto& kv : cache) {
      const int32_t b = kv.second;
      if (ref[b] == 1 && !pinned_below[b]) ++avail;
    }
    return avail;
  }
};

extern "C" {

pkv_allocator* pkv_allocator_create(int32_t num_blocks) {
  if (num_blocks < 1 || num_blocks > (1 << 26)) return nullptr;
  pkv_allocator* a = new (std::nothrow) pkv_allocator();
  if (!a) return nullptr;
  try {
    a->n = num_blocks;
    a->ref.assign(num_blocks, 0);
    for (int32_t b = 0; b < num_blocks; ++b) a->free.insert(a->free.end(), b);
    a->cached.assign(num_blocks, 0);
    a->key_of.resize(num_blocks);
    a->kids.resize(num_blocks);
    a->lru_pos.resize(num_blocks);
    a->in_lru.assign(num_blocks, 0);
  } catch (...) {
    delete a;
    return nullptr;
  }
  return a;
}

void pkv_allocator_destroy(pkv_allocator* a) { delete a; }

int32_t pkv_allocator_free_blocks(const pkv_allocator* a) {
  return a ? static_cast<int32_t>(a->free.size()) : 0;
}

int32_t pkv_allocator_evictable(const pkv_allocator* a) {
  return a ? static_cast<int32_t>(a->available() - static_cast<int64_t>(a->free.size())) : 0;
}

int32_t pkv_allocator_refcount(const pkv_allocator* a, int32_t block) {
  if (!a || block < 0 || block >= a->n) return -1;
  return a->ref[block];
}

int pkv_seq_add(pkv_allocator* a, int64_t seq) {
  if (!a || a->seqs.count(seq)) return PKV_ERR_INVALID_ARGUMENT;
  try {
    a->seqs.emplace(seq, Seq{});
  } catch (...) {
    return PKV_ERR_CUDA;   // host out of memory; nothing changed
  }
  return PKV_OK;
}

int pkv_seq_fork(pkv_allocator* a, int64_t parent, int64_t child) {
  if (!a || parent == child || a->seqs.count(child)) return PKV_ERR_INVALID_ARGUMENT;
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end()) return PKV_ERR_INVALID_ARGUMENT;
  std::vector<int32_t> shared;
  try {
    Seq copy = it->second;
    shared = copy.blocks;
    a->seqs.emplace(child, std::move(copy));   // may rehash: `it` is not used after this
  } catch (...) {
    return PKV_ERR_CUDA;
  }
  for (int32_t b : shared) a->inc_ref(b);
  return PKV_OK;
}

int pkv_seq_release(pkv_allocator* a, int64_t seq) {
  if (!a) return PKV_ERR_INVALID_ARGUMENT;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PKV_ERR_INVALID_ARGUMENT;
  for (int32_t b : it->second.blocks) a->dec_ref(b);
  a->seqs.erase(it);
  return PKV_OK;
}

int32_t pkv_seq_length(const pkv_allocator* a, int64_t seq) {
  if (!a) return -1;
  auto it = a->seqs.find(seq);
  return it == a->seqs.end() ? -1 : it->second.len;
}

int32_t pkv_seq_block_table(const pkv_allocator* a, int64_t seq, int32_t* out, int32_t capacity) {
  if (!a || capacity < 0 || (capacity > 0 && !out)) return PKV_ERR_INVALID_ARGUMENT;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PKV_ERR_INVALID_ARGUMENT;
  const std::vector<int32_t>& bl = it->second.blocks;
  const size_t m = bl.size() < static_cast<size_t>(capacity) ? bl.size() : static_cast<size_t>(capacity);
  if (m) std::memcpy(out, bl.data(), m * sizeof(int32_t));
  return static_cast<int32_t>(bl.size());
}

int pkv_seq_append(pkv_allocator* a, int64_t seq, int32_t n, int32_t* slots, int32_t* copy_src,
                   int32_t* copy_dst, int32_t* num_copies) {
  if (!a || n < 0 || (n > 0 && !slots) || !copy_src || !copy_dst || !num_copies)
    return PKV_ERR_INVALID_ARGUMENT;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PKV_ERR_INVALID_ARGUMENT;
  Seq& s = it->second;
  const int64_t new_len = static_cast<int64_t>(s.len) + n;
  if (new_len > (1ll << 30)) return PKV_ERR_INVALID_ARGUMENT;
  const bool cow = n > 0 && (s.len % kTokensPerBlock) != 0 && a->ref[s.blocks.back()] > 1;
  const int64_t need = blocks_for(new_len) - blocks_for(s.len) + (cow ? 1 : 0);
  if (need > static_cast<int64_t>(a->free.size()) && need > a->available()) return PKV_ERR_OUT_OF_BLOCKS;
  try {
    s.blocks.reserve(static_cast<size_t>(blocks_for(new_len)));
  } catch (...) {
    return PKV_ERR_CUDA;
  }
  *num_copies = 0;
  if (cow) {
    const int32_t src = s.blocks.back();
    const int32_t dst = a->take_block();
    a->dec_ref(src);
    s.blocks.back() = dst;
    copy_src[0] = src;
    copy_dst[0] = dst;
    *num_copies = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int64_t p = static_cast<int64_t>(s.len) + i;
    if (p % kTokensPerBlock == 0) s.blocks.push_back(a->take_block());
    slots[i] = s.blocks[static_cast<size_t>(p / kTokensPerBlock)] * kTokensPerBlock +
               static_cast<int32_t>(p % kTokensPerBlock);
  }
  s.len = static_cast<int32_t>(new_len);
  return PKV_OK;
}

int32_t pkv_prefix_insert(pkv_allocator* a, int64_t seq, const int32_t* tokens, int32_t n) {
  if (!a || n < 0 || (n > 0 && !tokens)) return PKV_ERR_INVALID_ARGUMENT;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end() || n > it->second.len) return PKV_ERR_INVALID_ARGUMENT;
  const Seq& s = it->second;
  int32_t parent = -1, added = 0;
  for (int32_t k = 0; k < n / kTokensPerBlock; ++k) {
    PrefixKey key;
    key.parent = parent;
    std::memcpy(key.tok.data(), tokens + k * kTokensPerBlock, sizeof(int32_t) * kTokensPerBlock);
    auto c = a->cache.find(key);
    if (c != a->cache.end()) {
      parent = c->second;   // this prefix is cached (possibly in another block): follow it
      continue;
    }
    const int32_t b = s.blocks[static_cast<size_t>(k)];
    if (a->cached[b]) break;   // the block already caches other contents: stop here
    try {
      a->cache.emplace(key, b);
      if (parent >= 0) a->kids[parent].push_back(b);
    } catch (...) {
      a->cache.erase(key);
      return PKV_ERR_CUDA;
    }
    a->cached[b] = 1;
    a->key_of[b] = key;
    ++a->ref[b];                  // the tree's reference
    a->update_lru(b);
    if (parent >= 0) a->update_lru(parent);
    parent = b;
    ++added;
  }
  return added;
}

int pkv_seq_add_cached(pkv_allocator* a, int64_t seq, const int32_t* tokens, int32_t n,
                       int32_t* cached_tokens) {
  if (!a || n < 0 || (n > 0 && !tokens) || !cached_tokens || a->seqs.count(seq))
    return PKV_ERR_INVALID_ARGUMENT;
  std::vector<int32_t> hit;
  int32_t parent = -1;
  try {
    for (int32_t k = 0; k < n / kTokensPerBlock; ++k) {
      PrefixKey key;
      key.parent = parent;
      std::memcpy(key.tok.data(), tokens + k * kTokensPerBlock, sizeof(int32_t) * kTokensPerBlock);
      auto c = a->cache.find(key);
      if (c == a->cache.end()) break;
      hit.push_back(c->second);
      parent = c->second;
    }
    Seq s;
    s.blocks = hit;
    s.len = static_cast<int32_t>(hit.size()) * kTokensPerBlock;
    a->seqs.emplace(seq, std::move(s));
  } catch (...) {
    return PKV_ERR_CUDA;
  }
  for (int32_t b : hit) a->inc_ref(b);
  *cached_tokens = static_cast<int32_t>(hit.size()) * kTokensPerBlock;
  return PKV_OK;
}

}  // extern "C"
