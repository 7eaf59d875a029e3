// pkv_pool.cpp -- the host block pool of include/pkv_pool.h.
//
// "Implémentation du cœur du moteur d'inférence haute performance vLLM",
// ch. 4 §4.1, §4.3, §4.4 and "Khám phá vLLM: Giải phẫu hệ thống suy luận LLM
// thông lượng cao", "KV cache manager" / "allocate_slots" (see the header for
// the behaviour each follows).
//
// Data structures, all O(1) per block operation:
//  * the free queue is an intrusive doubly linked list over block ids with a
//    sentinel (index num_blocks), so a cache hit can unlink any block;
//  * the prefix cache maps a 64-bit chained block hash to the blocks filed
//    under it, oldest first (almost always one): an open-addressing table
//    (linear probing, backward-shift deletion, doubled when half full) whose
//    entries hold the first and last block of a chain linked through
//    per-block arrays, so filing and evicting a block allocate nothing;
//  * a request keeps its token ids, its block ids and the hashes of its full
//    blocks, extended incrementally as tokens become computed.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_pool.h"

namespace {

constexpr uint64_t kFnvOffset = 0xCBF29CE484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001B3ull;

inline uint64_t fnv_byte(uint64_t h, uint8_t b) { return (h ^ b) * kFnvPrime; }

// h_i = FNV-1a-64(parent as 8 little-endian bytes, then each token id as 4
// little-endian bytes).
uint64_t block_hash(uint64_t parent, const int32_t* tokens, int n) {
  uint64_t h = kFnvOffset;
  for (int i = 0; i < 8; ++i) h = fnv_byte(h, static_cast<uint8_t>(parent >> (8 * i)));
  for (int t = 0; t < n; ++t) {
    const uint32_t u = static_cast<uint32_t>(tokens[t]);
    for (int i = 0; i < 4; ++i) h = fnv_byte(h, static_cast<uint8_t>(u >> (8 * i)));
  }
  return h;
}

struct Request {
  std::vector<int32_t> tokens;
  std::vector<int32_t> blocks;    // position order; the null block where released
  std::vector<uint64_t> hashes;   // chained hashes of the leading full blocks
  int32_t num_computed = 0;
  int32_t num_filed = 0;          // leading full blocks already offered to the cache
};

}  // namespace

struct pkv_pool {
  int32_t nb = 0, bs = 0;
  bool caching = true;
  int32_t null_block = 0;
  std::vector<int32_t> ref, prev, next;  // prev/next: free-queue links, sentinel = nb
  std::vector<uint8_t> in_free, has_hash;
  std::vector<uint64_t> hash;
  int32_t num_free = 0, num_cached = 0;
  // prefix cache: table entries (head < 0: empty) and the chains' links
  struct Entry {
    uint64_t key;
    int32_t head, tail;
  };
  std::vector<Entry> table;
  int shift = 0;           // index = (key * golden) >> shift; table.size() = 2^(64 - shift)
  int64_t entries = 0;
  std::vector<int32_t> hnext, hprev;
  std::unordered_map<int64_t, Request> reqs;

  size_t home(uint64_t key) const {
    return static_cast<size_t>((key * 0x9E3779B97F4A7C15ull) >> shift);
  }
  void init_table(int log2_size) {
    shift = 64 - log2_size;
    table.assign(size_t{1} << log2_size, Entry{0, -1, -1});
  }
  // Index of key's entry, or of the empty slot where it would go.
  size_t probe(uint64_t key) const {
    const size_t mask = table.size() - 1;
    size_t i = home(key);
    while (table[i].head >= 0 && table[i].key != key) i = (i + 1) & mask;
    return i;
  }
  void grow() {
    std::vector<Entry> old;
    old.swap(table);
    init_table(65 - shift);
    for (const Entry& e : old)
      if (e.head >= 0) table[probe(e.key)] = e;
  }
  void erase_entry(size_t i) {
    const size_t mask = table.size() - 1;
    size_t j = i;
    while (true) {
      j = (j + 1) & mask;
      if (table[j].head < 0) break;
      const size_t k = home(table[j].key);
      // the entry at j may stay if its home lies cyclically in (i, j]
      const bool stays = i <= j ? (i < k && k <= j) : (i < k || k <= j);
      if (stays) continue;
      table[i] = table[j];
      i = j;
    }
    table[i].head = -1;
    --entries;
  }
  // First block filed under key, or -1.
  int32_t lookup(uint64_t key) const {
    const Entry& e = table[probe(key)];
    return e.head >= 0 ? e.head : -1;
  }

  // ---- free queue
  void link_before(int32_t b, int32_t at) {  // insert b before `at`
    const int32_t p = prev[at];
    next[p] = b;
    prev[b] = p;
    next[b] = at;
    prev[at] = b;
    in_free[b] = 1;
    ++num_free;
  }
  void push_head(int32_t b) { link_before(b, next[nb]); }
  void push_tail(int32_t b) { link_before(b, nb); }
  void unlink(int32_t b) {
    next[prev[b]] = next[b];
    prev[next[b]] = prev[b];
    in_free[b] = 0;
    --num_free;
  }
  int32_t pop_head() {
    const int32_t b = next[nb];
    unlink(b);
    return b;
  }

  // ---- prefix cache
  void evict_hash(int32_t b) {
    if (!has_hash[b]) return;
    const size_t i = probe(hash[b]);
    Entry& e = table[i];
    const int32_t p = hprev[b], n = hnext[b];
    if (p >= 0) hnext[p] = n;
    else e.head = n;
    if (n >= 0) hprev[n] = p;
    else e.tail = p;
    if (e.head < 0) erase_entry(i);
    has_hash[b] = 0;
    --num_cached;
  }
  void file_block(int32_t b, uint64_t h) {
    if (has_hash[b] && hash[b] == h) return;
    evict_hash(b);
    hash[b] = h;
    has_hash[b] = 1;
    hnext[b] = -1;
    size_t i = probe(h);
    if (table[i].head >= 0) {  // append to the chain: lookups return the oldest
      hprev[b] = table[i].tail;
      hnext[table[i].tail] = b;
      table[i].tail = b;
    } else {
      if (2 * (entries + 1) > static_cast<int64_t>(table.size())) {
        grow();
        i = probe(h);
      }
      hprev[b] = -1;
      table[i] = Entry{h, b, b};
      ++entries;
    }
    ++num_cached;
  }

  // ---- block lifecycle
  int32_t get_new_block() {
    const int32_t b = pop_head();
    evict_hash(b);
    ++ref[b];
    return b;
  }
  void touch(int32_t b) {
    if (ref[b] == 0) unlink(b);
    ++ref[b];
  }
  void release(int32_t b) {
    if (b == null_block) return;
    if (--ref[b] == 0) {
      if (has_hash[b]) push_tail(b);
      else push_head(b);
    }
  }

  // Extends r's chained hashes to its first n full blocks of known tokens.
  void extend_hashes(Request& r, int32_t n) {
    while (static_cast<int32_t>(r.hashes.size()) < n) {
      const size_t i = r.hashes.size();
      const uint64_t parent = i ? r.hashes[i - 1] : 0;
      r.hashes.push_back(block_hash(parent, r.tokens.data() + i * bs, bs));
    }
  }
};

extern "C" {

pkv_pool* pkv_pool_create(int32_t num_blocks, int32_t block_size, int32_t enable_caching) {
  if (num_blocks < 1 || block_size < 1) return nullptr;
  pkv_pool* p = new (std::nothrow) pkv_pool;
  if (!p) return nullptr;
  try {
    p->nb = num_blocks;
    p->bs = block_size;
    p->caching = enable_caching != 0;
    p->ref.assign(num_blocks, 0);
    p->prev.assign(num_blocks + 1, num_blocks);
    p->next.assign(num_blocks + 1, num_blocks);
    p->in_free.assign(num_blocks, 0);
    p->has_hash.assign(num_blocks, 0);
    p->hash.assign(num_blocks, 0);
    p->hnext.assign(num_blocks, -1);
    p->hprev.assign(num_blocks, -1);
    p->init_table(10);
  } catch (...) {
    delete p;
    return nullptr;
  }
  for (int32_t b = 0; b < num_blocks; ++b) p->push_tail(b);  // eviction order = id order
  p->null_block = p->pop_head();                              // first block off the head
  return p;
}

void pkv_pool_destroy(pkv_pool* pool) { delete pool; }

int32_t pkv_pool_num_free(const pkv_pool* pool) { return pool ? pool->num_free : -1; }
int32_t pkv_pool_null_block(const pkv_pool* pool) { return pool ? pool->null_block : -1; }
int32_t pkv_pool_num_cached(const pkv_pool* pool) { return pool ? pool->num_cached : -1; }

int pkv_pool_add_request(pkv_pool* pool, int64_t req_id, const int32_t* tokens,
                         int32_t num_tokens) {
  if (!pool || (num_tokens > 0 && !tokens)) return PKV_E_NULL;
  if (num_tokens < 0) return PKV_E_SHAPE;
  if (pool->reqs.count(req_id)) return PKV_E_REQUEST;
  Request& r = pool->reqs[req_id];
  r.tokens.assign(tokens, tokens + num_tokens);
  return PKV_OK;
}

int pkv_pool_append_tokens(pkv_pool* pool, int64_t req_id, const int32_t* tokens,
                           int32_t num_tokens) {
  if (!pool || (num_tokens > 0 && !tokens)) return PKV_E_NULL;
  if (num_tokens < 0) return PKV_E_SHAPE;
  auto it = pool->reqs.find(req_id);
  if (it == pool->reqs.end()) return PKV_E_REQUEST;
  it->second.tokens.insert(it->second.tokens.end(), tokens, tokens + num_tokens);
  return PKV_OK;
}

int pkv_pool_append_token_batch(pkv_pool* pool, const int64_t* req_ids, const int32_t* tokens,
                                int32_t num_reqs) {
  if (!pool || (num_reqs > 0 && (!req_ids || !tokens))) return PKV_E_NULL;
  if (num_reqs < 0) return PKV_E_SHAPE;
  for (int32_t i = 0; i < num_reqs; ++i) {
    auto it = pool->reqs.find(req_ids[i]);
    if (it == pool->reqs.end()) return PKV_E_REQUEST;
    it->second.tokens.push_back(tokens[i]);
  }
  return PKV_OK;
}

int pkv_pool_admit(pkv_pool* pool, int64_t req_id, int32_t* num_cached_tokens) {
  if (!pool || !num_cached_tokens) return PKV_E_NULL;
  auto it = pool->reqs.find(req_id);
  if (it == pool->reqs.end()) return PKV_E_REQUEST;
  Request& r = it->second;
  if (!r.blocks.empty() || r.num_computed != 0) return PKV_E_REQUEST;
  *num_cached_tokens = 0;
  if (!pool->caching || r.tokens.empty()) return PKV_OK;
  // at most num_tokens - 1 tokens come from the cache
  const int32_t cap = (static_cast<int32_t>(r.tokens.size()) - 1) / pool->bs;
  pool->extend_hashes(r, cap);
  for (int32_t i = 0; i < cap; ++i) {
    const int32_t b = pool->lookup(r.hashes[i]);
    if (b < 0) break;
    r.blocks.push_back(b);
  }
  for (int32_t b : r.blocks) pool->touch(b);
  r.num_computed = static_cast<int32_t>(r.blocks.size()) * pool->bs;
  r.num_filed = static_cast<int32_t>(r.blocks.size());
  *num_cached_tokens = r.num_computed;
  return PKV_OK;
}

int pkv_pool_allocate_slots(pkv_pool* pool, int64_t req_id, int32_t num_new_tokens,
                            int32_t sliding_window, int64_t* slot_mapping) {
  if (!pool) return PKV_E_NULL;
  if (num_new_tokens < 0 || sliding_window < 0) return PKV_E_SHAPE;
  auto it = pool->reqs.find(req_id);
  if (it == pool->reqs.end()) return PKV_E_REQUEST;
  Request& r = it->second;
  const int32_t bs = pool->bs;
  const int64_t first = r.num_computed;
  const int64_t end = first + num_new_tokens;
  if (end > INT32_MAX) return PKV_E_SHAPE;
  // phase 1: blocks wholly before every new token's window
  std::vector<int32_t> drop;
  int32_t freeable = 0;
  if (sliding_window > 0) {
    const int64_t keep_from = first - sliding_window + 1 > 0 ? first - sliding_window + 1 : 0;
    const int64_t n = keep_from / bs < static_cast<int64_t>(r.blocks.size())
                          ? keep_from / bs
                          : static_cast<int64_t>(r.blocks.size());
    for (int64_t i = 0; i < n; ++i)
      if (r.blocks[i] != pool->null_block) {
        drop.push_back(static_cast<int32_t>(i));
        if (pool->ref[r.blocks[i]] == 1) ++freeable;
      }
  }
  const int64_t need = (end + bs - 1) / bs - static_cast<int64_t>(r.blocks.size());
  if (need > pool->num_free + freeable) return PKV_POOL_NO_SPACE;
  // released last to first, replaced by the null block
  for (size_t k = drop.size(); k-- > 0;) {
    const int32_t b = r.blocks[drop[k]];
    r.blocks[drop[k]] = pool->null_block;
    pool->release(b);
  }
  // phase 3: new blocks for the new tokens
  for (int64_t i = 0; i < need; ++i) r.blocks.push_back(pool->get_new_block());
  if (slot_mapping)
    for (int64_t p = first; p < end; ++p)
      slot_mapping[p - first] = static_cast<int64_t>(r.blocks[p / bs]) * bs + p % bs;
  r.num_computed = static_cast<int32_t>(end);
  // newly full blocks whose tokens are known go into the prefix cache
  if (pool->caching) {
    const int64_t known = end < static_cast<int64_t>(r.tokens.size())
                              ? end : static_cast<int64_t>(r.tokens.size());
    const int32_t n_full = static_cast<int32_t>(known / bs);
    if (n_full > r.num_filed) {
      pool->extend_hashes(r, n_full);
      for (int32_t i = r.num_filed; i < n_full; ++i)
        if (r.blocks[i] != pool->null_block) pool->file_block(r.blocks[i], r.hashes[i]);
      r.num_filed = n_full;
    }
  }
  return PKV_OK;
}

int pkv_pool_allocate_slots_batch(pkv_pool* pool, const int64_t* req_ids,
                                  const int32_t* num_new_tokens, int32_t num_reqs,
                                  int32_t sliding_window, int64_t* slot_mapping,
                                  int32_t* num_done) {
  if (!pool || !num_done || (num_reqs > 0 && (!req_ids || !num_new_tokens))) return PKV_E_NULL;
  if (num_reqs < 0) return PKV_E_SHAPE;
  *num_done = 0;
  int64_t off = 0;
  for (int32_t i = 0; i < num_reqs; ++i) {
    const int st = pkv_pool_allocate_slots(pool, req_ids[i], num_new_tokens[i], sliding_window,
                                           slot_mapping ? slot_mapping + off : nullptr);
    if (st != PKV_OK) return st;
    off += num_new_tokens[i];
    *num_done = i + 1;
  }
  return PKV_OK;
}

int pkv_pool_free_request(pkv_pool* pool, int64_t req_id) {
  if (!pool) return PKV_E_NULL;
  auto it = pool->reqs.find(req_id);
  if (it == pool->reqs.end()) return PKV_E_REQUEST;
  const std::vector<int32_t>& blocks = it->second.blocks;
  for (size_t k = blocks.size(); k-- > 0;) pool->release(blocks[k]);
  pool->reqs.erase(it);
  return PKV_OK;
}

int pkv_pool_block_table(const pkv_pool* pool, int64_t req_id, int32_t* row, int32_t capacity,
                         int32_t* num_blocks) {
  if (!pool || !num_blocks || (capacity > 0 && !row)) return PKV_E_NULL;
  auto it = pool->reqs.find(req_id);
  if (it == pool->reqs.end()) return PKV_E_REQUEST;
  const std::vector<int32_t>& b = it->second.blocks;
  *num_blocks = static_cast<int32_t>(b.size());
  for (int32_t i = 0; i < capacity && i < static_cast<int32_t>(b.size()); ++i) row[i] = b[i];
  return PKV_OK;
}

int pkv_pool_build_block_tables(const pkv_pool* pool, const int64_t* req_ids, int32_t num_reqs,
                                int32_t* block_tables, int32_t stride) {
  if (!pool || (num_reqs > 0 && (!req_ids || !block_tables))) return PKV_E_NULL;
  if (num_reqs < 0 || stride < 1) return PKV_E_SHAPE;
  for (int32_t s = 0; s < num_reqs; ++s) {
    auto it = pool->reqs.find(req_ids[s]);
    if (it == pool->reqs.end()) return PKV_E_REQUEST;
    const std::vector<int32_t>& b = it->second.blocks;
    if (static_cast<int64_t>(b.size()) > stride) return PKV_E_SHAPE;
    int32_t* row = block_tables + static_cast<int64_t>(s) * stride;
    for (int32_t i = 0; i < stride; ++i) row[i] = i < static_cast<int32_t>(b.size()) ? b[i] : -1;
  }
  return PKV_OK;
}

int pkv_pool_num_computed(const pkv_pool* pool, int64_t req_id, int32_t* num_computed) {
  if (!pool || !num_computed) return PKV_E_NULL;
  auto it = pool->reqs.find(req_id);
  if (it == pool->reqs.end()) return PKV_E_REQUEST;
  *num_computed = it->second.num_computed;
  return PKV_OK;
}

int pkv_pool_block_state(const pkv_pool* pool, int32_t block, int32_t* ref_cnt, uint64_t* hash,
                         int32_t* has_hash) {
  if (!pool || !ref_cnt || !hash || !has_hash) return PKV_E_NULL;
  if (block < 0 || block >= pool->nb) return PKV_E_SHAPE;
  *ref_cnt = pool->ref[block];
  *hash = pool->hash[block];
  *has_hash = pool->has_hash[block];
  return PKV_OK;
}

int pkv_pool_free_queue(const pkv_pool* pool, int32_t* out, int32_t capacity, int32_t* n) {
  if (!pool || !n || (capacity > 0 && !out)) return PKV_E_NULL;
  *n = pool->num_free;
  int32_t i = 0;
  for (int32_t b = pool->next[pool->nb]; b != pool->nb && i < capacity; b = pool->next[b])
    out[i++] = b;
  return PKV_OK;
}

}  // extern "C"
