// block_manager.cpp -- host allocator of the paged KV cache's blocks.
//
// The cache is a pool of fixed 256-token blocks whose allocation and release
// are managed by reference counts (nano-vllm hub page, "core tech 4: KV Cache
// block manager"); a sequence's block table maps its logical blocks to
// physical ones, a new block being taken when the length reaches a multiple
// of the block size plus one (CSDN essay "from nanoVLLM to vLLM", Mountain 1).
// Prefix sharing: a full block is keyed by a hash chained over the keys of
// the blocks before it and its own tokens, so a new sequence whose prompt
// starts with the same full blocks reuses them (reference count + 1) instead
// of storing and attending over fresh copies; freed blocks keep their content
// and key until they are handed out again.
//
// Single-threaded: one manager per host thread (or external locking).
#include <stdint.h>
#include <string.h>

#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace {

// FNV-1a, 64-bit (offset basis 0xcbf29ce484222325, prime 0x100000001b3),
// fed the parent key and then the block's token ids, byte by byte.
uint64_t fnv1a(uint64_t h, const void *data, size_t n) {
  const unsigned char *p = static_cast<const unsigned char *>(data);
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

uint64_t block_key(uint64_t parent, const int32_t *tokens, int n) {
  uint64_t h = fnv1a(0xcbf29ce484222325ull, &parent, sizeof(parent));
  h = fnv1a(h, tokens, sizeof(int32_t) * (size_t)n);
  return h == 0 ? 1 : h;  // 0 marks "no key"
}

struct Seq {
  std::vector<int32_t> table;   // physical block of each logical block
  std::vector<int32_t> tokens;  // all tokens so far (keys of blocks that fill up)
};

}  // namespace

struct pkv_block_manager {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> ref;               // reference count per block
  std::vector<uint64_t> key;              // content key of a full block, 0 = none
  std::vector<int32_t> content;           // [num_blocks][block_size] token ids of keyed blocks
  std::vector<int32_t> prev, next;        // free list (doubly linked, FIFO: oldest freed first)
  std::vector<uint8_t> is_free;
  int free_head = -1, free_tail = -1, num_free = 0;
  std::unordered_map<uint64_t, int32_t> by_key;
  std::unordered_map<int64_t, Seq> seqs;

  void push_free(int b) {
    prev[b] = free_tail;
    next[b] = -1;
    if (free_tail >= 0) next[free_tail] = b;
    else free_head = b;
    free_tail = b;
    is_free[b] = 1;
    ++num_free;
  }
  void unlink_free(int b) {
    if (prev[b] >= 0) next[prev[b]] = next[b];
    else free_head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b];
    else free_tail = prev[b];
    is_free[b] = 0;
    --num_free;
  }
  // A fresh block: the oldest free one, forgetting any content it held.
  int take_fresh() {
    if (free_head < 0) return -1;
    const int b = free_head;
    unlink_free(b);
    if (key[b] != 0) {
      auto it = by_key.find(key[b]);
      if (it != by_key.end() && it->second == b) by_key.erase(it);
      key[b] = 0;
    }
    ref[b] = 1;
    return b;
  }
  // The keyed block holding exactly these tokens after `parent`, or -1.
  int lookup(uint64_t k, const int32_t *tokens) const {
    auto it = by_key.find(k);
    if (it == by_key.end()) return -1;
    const int b = it->second;
    if (memcmp(&content[(size_t)b * block_size], tokens, sizeof(int32_t) * block_size) != 0)
      return -1;  // hash collision: treat as a miss
    return b;
  }
  void set_key(int b, uint64_t k, const int32_t *tokens) {
    key[b] = k;
    memcpy(&content[(size_t)b * block_size], tokens, sizeof(int32_t) * block_size);
    by_key[k] = b;
  }
  void release(int b) {
    if (--ref[b] == 0) push_free(b);
  }
  uint64_t key_of_block(const Seq &s, int i) const {
    return i < 0 ? 0 : key[s.table[i]];
  }
};

extern "C" pkv_block_manager *pkv_bm_create(int num_blocks, int block_size) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pkv_block_manager *m = new (std::nothrow) pkv_block_manager();
  if (m == nullptr) return nullptr;
  try {
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->ref.assign(num_blocks, 0);
    m->key.assign(num_blocks, 0);
    m->content.assign((size_t)num_blocks * block_size, 0);
    m->prev.assign(num_blocks, -1);
    m->next.assign(num_blocks, -1);
    m->is_free.assign(num_blocks, 0);
    for (int b = 0; b < num_blocks; ++b) m->push_free(b);
  } catch (...) {
    delete m;
    return nullptr;
  }
  return m;
}

extern "C" void pkv_bm_destroy(pkv_block_manager *m) { delete m; }

extern "C" int pkv_bm_num_free_blocks(const pkv_block_manager *m) {
  return m == nullptr ? -1 : m->num_free;
}

extern "C" pkv_status pkv_bm_allocate(pkv_block_manager *m, int64_t seq_id, const int32_t *tokens,
                                      int num_tokens, int *num_cached_tokens) {
  if (m == nullptr || num_tokens <= 0 || tokens == nullptr || num_cached_tokens == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (m->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
  const int bs = m->block_size;
  const int nblocks = (num_tokens + bs - 1) / bs;
  const int full = num_tokens / bs;
  // Leading full blocks already in the cache (content keys chained from the start).
  std::vector<int32_t> hits;
  uint64_t parent = 0;
  for (int i = 0; i < full; ++i) {
    const uint64_t k = block_key(parent, tokens + (size_t)i * bs, bs);
    const int b = m->lookup(k, tokens + (size_t)i * bs);
    if (b < 0) break;
    hits.push_back(b);
    parent = k;
  }
  // Fresh blocks needed beyond the hits: all must be available up front.
  const int fresh = nblocks - (int)hits.size();
  int hits_free = 0;
  for (int b : hits) hits_free += m->is_free[b] ? 1 : 0;
  if (m->num_free - hits_free < fresh) return PKV_ERR_OUT_OF_BLOCKS;
  Seq s;
  s.tokens.assign(tokens, tokens + num_tokens);
  for (int b : hits) {
    if (m->is_free[b]) m->unlink_free(b);
    ++m->ref[b];
    s.table.push_back(b);
  }
  for (int i = (int)hits.size(); i < nblocks; ++i) {
    const int b = m->take_fresh();
    s.table.push_back(b);
    if (i < full) {  // a full block gets its key now, for later sequences
      const uint64_t k = block_key(m->key_of_block(s, i - 1), tokens + (size_t)i * bs, bs);
      m->set_key(b, k, tokens + (size_t)i * bs);
    }
  }
  // At least the last prompt token is computed even when every block was found.
  int cached = (int)hits.size() * bs;
  if (cached >= num_tokens) cached = num_tokens - 1;
  *num_cached_tokens = cached;
  m->seqs.emplace(seq_id, std::move(s));
  return PKV_OK;
}

extern "C" pkv_status pkv_bm_append(pkv_block_manager *m, int64_t seq_id, int32_t token) {
  if (m == nullptr) return PKV_ERR_INVALID_ARG;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
  Seq &s = it->second;
  const int bs = m->block_size;
  const int len = (int)s.tokens.size();
  if (len % bs == 0) {  // the new token starts block len / bs (length reaches k*bs + 1)
    if (m->num_free == 0) return PKV_ERR_OUT_OF_BLOCKS;
    s.table.push_back(m->take_fresh());
  }
  s.tokens.push_back(token);
  if ((len + 1) % bs == 0) {  // a block just filled up: key it for later sequences
    const int i = (len + 1) / bs - 1;
    const int b = s.table[i];
    if (m->key[b] == 0) {
      const uint64_t k = block_key(m->key_of_block(s, i - 1), &s.tokens[(size_t)i * bs], bs);
      if (m->lookup(k, &s.tokens[(size_t)i * bs]) < 0) m->set_key(b, k, &s.tokens[(size_t)i * bs]);
    }
  }
  return PKV_OK;
}

extern "C" pkv_status pkv_bm_free(pkv_block_manager *m, int64_t seq_id) {
  if (m == nullptr) return PKV_ERR_INVALID_ARG;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
  // Last block first, so that a sequence's tail is reused before its prefix.
  for (int i = (int)it->second.table.size() - 1; i >= 0; --i) m->release(it->second.table[i]);
  m->seqs.erase(it);
  return PKV_OK;
}

extern "C" int pkv_bm_num_tokens(const pkv_block_manager *m, int64_t seq_id) {
  if (m == nullptr) return -1;
  auto it = m->seqs.find(seq_id);
  return it == m->seqs.end() ? -1 : (int)it->second.tokens.size();
}

extern "C" int pkv_bm_block_table(const pkv_block_manager *m, int64_t seq_id, int32_t *out,
                                  int max_blocks) {
  if (m == nullptr) return -1;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return -1;
  const auto &t = it->second.table;
  if (out != nullptr)
    for (int i = 0; i < max_blocks; ++i) out[i] = i < (int)t.size() ? t[i] : -1;
  return (int)t.size();
}

extern "C" pkv_status pkv_bm_slots(const pkv_block_manager *m, int64_t seq_id, int first,
                                   int count, int32_t *slots) {
  if (m == nullptr || first < 0 || count < 0 || (count > 0 && slots == nullptr))
    return PKV_ERR_INVALID_ARG;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
  const Seq &s = it->second;
  if ((int64_t)first + count > (int64_t)s.tokens.size()) return PKV_ERR_INVALID_ARG;
  const int bs = m->block_size;
  for (int i = 0; i < count; ++i) {
    const int p = first + i;
    slots[i] = s.table[p / bs] * bs + p % bs;
  }
  return PKV_OK;
}

extern "C" int pkv_bm_ref_count(const pkv_block_manager *m, int block) {
  if (m == nullptr || block < 0 || block >= m->num_blocks) return -1;
  return m->ref[block];
}
