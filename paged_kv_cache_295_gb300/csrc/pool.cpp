// Host block pool: FIFO free list, per-block reference counts, per-sequence
// block tables and slot arithmetic.
//
// Behaviour follows "LLM inference tutorial" section 4.2 (class PagedKVCache:
// free list 0..N-1, allocate_sequence takes the front block at once,
// append_token's block/offset rule, free_sequence returns blocks to the tail,
// memory_usage), section 4.3 (prefix sharing by reference count; a block is
// released when its count reaches zero) and "nano-vLLM architecture" section
// 4.3 (block_bytes and available_blocks = free_memory // block_bytes).
//
// The free list is a ring buffer of capacity num_blocks: a block id is in it
// at most once, so it never overflows and both ends are O(1).
//
// Copy-on-write ("LLM inference tutorial" section 4.2, the class docstring:
// beam search): forks share blocks, including a partly filled last block; the
// first write into a block whose count is above one moves the writer to a new
// block from the free-list front and records (old, new) in a pending-copy list
// that the caller drains (pool_take_copies) and executes on the device
// (copy_blocks) before writing the token.
//
// Swap ("ToPG framework" section 2.3: LRU-managed pages, contexts beyond
// device memory): sequences are ordered by their last create / fork / append
// (least recently used first); a swap-out moves a sequence's private blocks
// (count 1) to slots of a host area (FIFO free list) and leaves its shared
// blocks on the device; a swapped-out sequence takes no append, fork, prefix
// insert or batch view until its swap-in gives each host block a device block
// from the free-list front.  Both return the pairs the caller copies
// (swap_blocks) on its stream.
//
// Prefix cache (section 4.3, PrefixCacheManager): entries map a token prefix
// to the blocks holding it, with a count that starts at 1 (cache_prefix),
// rises on every hit of the longest-prefix lookup (get_cached_prefix) and
// falls on release (release_prefix); at zero the entry is dropped together
// with the block references it held.  Lookup hashes every prefix of the query
// in one pass (a 64-bit mix per token) and probes from the longest down; a
// probe hit is confirmed by comparing the tokens, so collisions cannot match.
#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <utility>
#include <vector>

#include "pagedkv.h"

namespace {

int dtype_size(int32_t dt) {
  switch (dt) {
    case PKV_F32: return 4;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
    case PKV_INT8: return 1;
    default: return 0;
  }
}

struct Seq {
  std::vector<int32_t> table;     // device block ids; host slot ids where on_host[j]
  std::vector<uint8_t> on_host;   // empty while resident
  int32_t len = 0;
  uint64_t last_use = 0;          // pool clock at the last create / fork / append
};

struct PrefixEntry {
  std::vector<int32_t> tokens;
  std::vector<int32_t> blocks;
  int32_t count = 0;
};

// Hash of every prefix of tokens[0..n): out[k] covers the first k+1 tokens.
void prefix_hashes(const int32_t* tokens, int32_t n, std::vector<uint64_t>& out) {
  out.resize(n);
  uint64_t h = 0x243F6A8885A308D3ull;
  for (int32_t i = 0; i < n; ++i) {
    uint64_t x = h ^ (static_cast<uint64_t>(static_cast<uint32_t>(tokens[i])) + 0x9E3779B97F4A7C15ull);
    x ^= x >> 30;
    x *= 0xBF58476D1CE4E5B9ull;
    x ^= x >> 27;
    x *= 0x94D049BB133111EBull;
    x ^= x >> 31;
    h = x;
    out[i] = h;
  }
}

}  // namespace

struct pkv_pool {
  pkv_pool_config cfg{};
  int64_t num_blocks = 0;
  int64_t block_bytes = 0;
  std::vector<int32_t> ring;   // free list storage
  int64_t head = 0;            // index of the front
  int64_t count = 0;           // number of free blocks
  std::vector<int32_t> ref;    // reference count per block (0 = free)
  std::unordered_map<int64_t, Seq> seqs;
  std::vector<std::pair<int32_t, int32_t>> copies;   // pending copy-on-write (src, dst)
  std::vector<int32_t> host_ring;   // host swap slots, FIFO free list
  int64_t host_head = 0, host_count = 0, host_blocks = 0;
  uint64_t clock = 0;

  void touch(Seq& s) { s.last_use = ++clock; }
  int32_t host_pop() {
    const int32_t h = host_ring[host_head];
    host_head = (host_head + 1) % host_blocks;
    --host_count;
    return h;
  }
  void host_push(int32_t h) {
    host_ring[(host_head + host_count) % host_blocks] = h;
    ++host_count;
  }
  std::unordered_map<uint64_t, std::vector<PrefixEntry>> prefix;   // prefix hash -> entries

  // The entry cached for exactly tokens[0..n) (hash h), or nullptr.
  PrefixEntry* find_prefix(uint64_t h, const int32_t* tokens, int32_t n) {
    auto it = prefix.find(h);
    if (it == prefix.end()) return nullptr;
    for (PrefixEntry& e : it->second)
      if (static_cast<int32_t>(e.tokens.size()) == n &&
          std::equal(e.tokens.begin(), e.tokens.end(), tokens))
        return &e;
    return nullptr;
  }

  int32_t pop_front() {
    int32_t b = ring[head];
    head = (head + 1) % num_blocks;
    --count;
    return b;
  }
  void push_back(int32_t b) {
    ring[(head + count) % num_blocks] = b;
    ++count;
  }
  bool valid(int64_t b) const { return b >= 0 && b < num_blocks; }
};

namespace {

// The block the sequence's next token goes to exists and is shared.
bool shared_target(const pkv_pool* p, const Seq& s) {
  const int64_t blk = s.len / p->cfg.block_size;
  return blk < static_cast<int64_t>(s.table.size()) && p->ref[s.table[blk]] > 1;
}

bool seq_needs_block(const pkv_pool* p, const Seq& s) {
  return static_cast<int64_t>(s.len / p->cfg.block_size) >=
             static_cast<int64_t>(s.table.size()) ||
         shared_target(p, s);
}

// Advance a sequence by one token, taking a block from the free-list front
// when the token's logical block is not in the table yet, or when it is
// shared (copy-on-write: the pending copy is recorded).  Capacity for the
// table entry and the copy record is reserved by the callers.
void append_one(pkv_pool* p, Seq& s) {
  const int32_t blk = s.len / p->cfg.block_size;
  if (blk >= static_cast<int32_t>(s.table.size())) {
    const int32_t b = p->pop_front();
    p->ref[b] = 1;
    s.table.push_back(b);
  } else if (p->ref[s.table[blk]] > 1) {
    const int32_t b = p->pop_front();
    p->ref[b] = 1;
    p->copies.emplace_back(s.table[blk], b);
    --p->ref[s.table[blk]];
    s.table[blk] = b;
  }
  ++s.len;
}

int64_t slot_of(const pkv_pool* p, const Seq& s, int32_t pos) {
  const int32_t bs = p->cfg.block_size;
  return static_cast<int64_t>(s.table[pos / bs]) * bs + pos % bs;
}

}  // namespace

extern "C" {

const char* pkv_status_string(int32_t st) {
  switch (st) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_NO_FREE_BLOCK: return "no free block";
    case PKV_ERR_BAD_BLOCK: return "block id out of range";
    case PKV_ERR_REFCOUNT: return "reference count error";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_HOST_MEMORY: return "host allocation failed";
    case PKV_ERR_SCRATCH_LIMIT: return "request exceeds the library's built-in decode scratch";
    default: return "unknown status";
  }
}

int64_t pkv_block_bytes(const pkv_pool_config* c) {
  if (!c) return -1;
  const int es = dtype_size(c->kv_dtype);
  if (c->num_layers <= 0 || c->block_size <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0 ||
      es == 0)
    return -1;
  return 2LL * c->num_layers * c->block_size * c->num_kv_heads * c->head_dim * es;
}

pkv_status kv_pool_init(const pkv_pool_config* cfg, pkv_pool** out) {
  if (!cfg || !out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  const int64_t bb = pkv_block_bytes(cfg);
  if (bb <= 0) return PKV_ERR_INVALID_ARG;
  int64_t nb = cfg->num_blocks;
  if (nb == 0) nb = cfg->free_bytes > 0 ? cfg->free_bytes / bb : 0;
  if (nb <= 0 || nb > INT32_MAX) return PKV_ERR_INVALID_ARG;
  pkv_pool* p = new (std::nothrow) pkv_pool();
  if (!p) return PKV_ERR_HOST_MEMORY;
  try {
    p->cfg = *cfg;
    p->cfg.initial_free_order = nullptr;
    p->cfg.num_blocks = nb;
    p->num_blocks = nb;
    p->block_bytes = bb;
    p->ring.resize(nb);
    p->ref.assign(nb, 0);
    if (cfg->initial_free_order) {
      std::vector<char> seen(nb, 0);
      for (int64_t i = 0; i < nb; ++i) {
        const int32_t b = cfg->initial_free_order[i];
        if (b < 0 || b >= nb || seen[b]) {
          delete p;
          return PKV_ERR_INVALID_ARG;
        }
        seen[b] = 1;
        p->ring[i] = b;
      }
    } else {
      for (int64_t i = 0; i < nb; ++i) p->ring[i] = static_cast<int32_t>(i);
    }
    p->head = 0;
    p->count = nb;
  } catch (const std::bad_alloc&) {
    delete p;
    return PKV_ERR_HOST_MEMORY;
  }
  *out = p;
  return PKV_OK;
}

void kv_pool_destroy(pkv_pool* p) { delete p; }

pkv_status block_alloc(pkv_pool* p, int32_t* id) {
  if (!p || !id) return PKV_ERR_INVALID_ARG;
  if (p->count == 0) return PKV_ERR_NO_FREE_BLOCK;
  const int32_t b = p->pop_front();
  p->ref[b] = 1;
  *id = b;
  return PKV_OK;
}

pkv_status block_ref(pkv_pool* p, int32_t id) {
  if (!p) return PKV_ERR_INVALID_ARG;
  if (!p->valid(id)) return PKV_ERR_BAD_BLOCK;
  if (p->ref[id] <= 0) return PKV_ERR_REFCOUNT;
  ++p->ref[id];
  return PKV_OK;
}

pkv_status block_free(pkv_pool* p, int32_t id) {
  if (!p) return PKV_ERR_INVALID_ARG;
  if (!p->valid(id)) return PKV_ERR_BAD_BLOCK;
  if (p->ref[id] <= 0) return PKV_ERR_REFCOUNT;
  if (--p->ref[id] == 0) p->push_back(id);
  return PKV_OK;
}

pkv_status block_refcount(const pkv_pool* p, int32_t id, int32_t* count) {
  if (!p || !count) return PKV_ERR_INVALID_ARG;
  if (!p->valid(id)) return PKV_ERR_BAD_BLOCK;
  *count = p->ref[id];
  return PKV_OK;
}

pkv_status kv_pool_stats(const pkv_pool* p, pkv_pool_stats* o) {
  if (!p || !o) return PKV_ERR_INVALID_ARG;
  o->total_blocks = p->num_blocks;
  o->free_blocks = p->count;
  o->used_blocks = p->num_blocks - p->count;
  o->utilization = static_cast<double>(o->used_blocks) / static_cast<double>(p->num_blocks) * 100.0;
  o->block_bytes = p->block_bytes;
  o->total_bytes = p->num_blocks * p->block_bytes;
  o->used_bytes = o->used_blocks * p->block_bytes;
  return PKV_OK;
}

pkv_status kv_pool_free_list(const pkv_pool* p, int32_t* out, int64_t cap, int64_t* n) {
  if (!p || !n) return PKV_ERR_INVALID_ARG;
  *n = p->count;
  if (cap < p->count || (!out && p->count > 0)) return PKV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < p->count; ++i) out[i] = p->ring[(p->head + i) % p->num_blocks];
  return PKV_OK;
}

pkv_status seq_create(pkv_pool* p, int64_t sid) {
  if (!p) return PKV_ERR_INVALID_ARG;
  if (p->seqs.count(sid)) return PKV_ERR_INVALID_ARG;
  if (p->count == 0) return PKV_ERR_NO_FREE_BLOCK;
  try {
    Seq s;
    s.table.reserve(8);
    const int32_t b = p->pop_front();
    p->ref[b] = 1;
    s.table.push_back(b);
    p->touch(s);
    p->seqs.emplace(sid, std::move(s));
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  return PKV_OK;
}

pkv_status seq_fork_prefix(pkv_pool* p, int64_t dst, int64_t src, int32_t ntok) {
  if (!p) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(src);
  if (it == p->seqs.end() || p->seqs.count(dst) || !it->second.on_host.empty())
    return PKV_ERR_INVALID_ARG;
  const int32_t bs = p->cfg.block_size;
  if (ntok <= 0 || ntok > it->second.len) return PKV_ERR_INVALID_ARG;
  try {
    Seq s;
    s.table.assign(it->second.table.begin(), it->second.table.begin() + (ntok + bs - 1) / bs);
    s.len = ntok;
    p->touch(s);
    for (int32_t b : s.table) ++p->ref[b];
    p->seqs.emplace(dst, std::move(s));
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  return PKV_OK;
}

pkv_status seq_append_slots(pkv_pool* p, const int64_t* ids, int32_t n, int64_t* slots) {
  if (!p || n < 0 || (n > 0 && (!ids || !slots))) return PKV_ERR_INVALID_ARG;
  std::vector<Seq*> v;
  try {
    v.reserve(n);
    std::unordered_set<int64_t> seen;
    seen.reserve(static_cast<size_t>(n) * 2);
    int64_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
      auto it = p->seqs.find(ids[i]);
      if (it == p->seqs.end() || !seen.insert(ids[i]).second || !it->second.on_host.empty())
        return PKV_ERR_INVALID_ARG;
      if (seq_needs_block(p, it->second)) ++need;
      v.push_back(&it->second);
    }
    if (need > p->count) return PKV_ERR_NO_FREE_BLOCK;
    for (int32_t i = 0; i < n; ++i) {
      Seq& s = *v[i];
      if (seq_needs_block(p, s)) s.table.reserve(s.table.size() + 1);
    }
    p->copies.reserve(p->copies.size() + static_cast<size_t>(need));
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  for (int32_t i = 0; i < n; ++i) {
    Seq& s = *v[i];
    const int32_t pos = s.len;
    append_one(p, s);
    slots[i] = slot_of(p, s, pos);
    p->touch(s);
  }
  return PKV_OK;
}

pkv_status seq_append_tokens(pkv_pool* p, int64_t sid, int32_t n, int64_t* slots) {
  if (!p || n < 0) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(sid);
  if (it == p->seqs.end() || !it->second.on_host.empty()) return PKV_ERR_INVALID_ARG;
  Seq& s = it->second;
  const int64_t bs = p->cfg.block_size;
  const int64_t have = static_cast<int64_t>(s.table.size()) * bs;
  const int64_t over = static_cast<int64_t>(s.len) + n - have;
  const int64_t cow = (n > 0 && shared_target(p, s)) ? 1 : 0;
  const int64_t need = (over > 0 ? (over + bs - 1) / bs : 0) + cow;
  if (need > p->count) return PKV_ERR_NO_FREE_BLOCK;
  if (static_cast<int64_t>(s.len) + n > INT32_MAX) return PKV_ERR_INVALID_ARG;
  try {
    s.table.reserve(s.table.size() + need);
    p->copies.reserve(p->copies.size() + static_cast<size_t>(cow));
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t pos = s.len;
    append_one(p, s);
    if (slots) slots[i] = slot_of(p, s, pos);
  }
  p->touch(s);
  return PKV_OK;
}

pkv_status seq_length(const pkv_pool* p, int64_t sid, int32_t* len) {
  if (!p || !len) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(sid);
  if (it == p->seqs.end()) return PKV_ERR_INVALID_ARG;
  *len = it->second.len;
  return PKV_OK;
}

pkv_status seq_block_table(const pkv_pool* p, int64_t sid, int32_t* out, int32_t cap,
                           int32_t* nblocks) {
  if (!p || !nblocks) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(sid);
  if (it == p->seqs.end()) return PKV_ERR_INVALID_ARG;
  const auto& t = it->second.table;
  *nblocks = static_cast<int32_t>(t.size());
  if (cap < static_cast<int32_t>(t.size()) || (!out && !t.empty())) return PKV_ERR_INVALID_ARG;
  if (!t.empty()) std::memcpy(out, t.data(), t.size() * sizeof(int32_t));
  return PKV_OK;
}

pkv_status seq_batch_tables(const pkv_pool* p, const int64_t* ids, int32_t n, int32_t mb,
                            int32_t* tables, int32_t* lens) {
  if (!p || n < 0 || mb < 0 || (n > 0 && (!ids || !lens || (mb > 0 && !tables))))
    return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    auto it = p->seqs.find(ids[i]);
    if (it == p->seqs.end() || !it->second.on_host.empty()) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(it->second.table.size()) > mb) return PKV_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    const Seq& s = p->seqs.find(ids[i])->second;
    int32_t* row = tables + static_cast<int64_t>(i) * mb;
    const int32_t k = static_cast<int32_t>(s.table.size());
    for (int32_t j = 0; j < k; ++j) row[j] = s.table[j];
    for (int32_t j = k; j < mb; ++j) row[j] = -1;
    lens[i] = s.len;
  }
  return PKV_OK;
}

pkv_status seq_free(pkv_pool* p, int64_t sid) {
  if (!p) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(sid);
  if (it == p->seqs.end()) return PKV_ERR_INVALID_ARG;
  const Seq& s = it->second;
  for (size_t j = 0; j < s.table.size(); ++j) {
    const int32_t b = s.table[j];
    if (!s.on_host.empty() && s.on_host[j])
      p->host_push(b);
    else if (--p->ref[b] == 0)
      p->push_back(b);
  }
  p->seqs.erase(it);
  return PKV_OK;
}

pkv_status pool_take_copies(pkv_pool* p, int32_t* pairs, int32_t cap, int32_t* n) {
  if (!p || !n || cap < 0) return PKV_ERR_INVALID_ARG;
  const int64_t k = static_cast<int64_t>(p->copies.size());
  if (k > INT32_MAX) return PKV_ERR_INVALID_ARG;
  *n = static_cast<int32_t>(k);
  if (cap < k || (!pairs && k > 0)) return PKV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < k; ++i) {
    pairs[2 * i] = p->copies[i].first;
    pairs[2 * i + 1] = p->copies[i].second;
  }
  p->copies.clear();
  return PKV_OK;
}

pkv_status prefix_cache_insert(pkv_pool* p, const int32_t* tokens, int32_t n, int64_t sid) {
  if (!p || n <= 0 || !tokens) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(sid);
  if (it == p->seqs.end() || n > it->second.len || !it->second.on_host.empty())
    return PKV_ERR_INVALID_ARG;
  try {
    std::vector<uint64_t> h;
    prefix_hashes(tokens, n, h);
    if (p->find_prefix(h[n - 1], tokens, n)) return PKV_ERR_INVALID_ARG;
    const int32_t bs = p->cfg.block_size;
    PrefixEntry e;
    e.tokens.assign(tokens, tokens + n);
    e.blocks.assign(it->second.table.begin(), it->second.table.begin() + (n + bs - 1) / bs);
    e.count = 1;
    auto& bucket = p->prefix[h[n - 1]];
    bucket.reserve(bucket.size() + 1);
    for (int32_t b : e.blocks) ++p->ref[b];
    bucket.push_back(std::move(e));
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  return PKV_OK;
}

namespace {

// Longest cached prefix of tokens[0..n): its entry and length, or nullptr.
PrefixEntry* longest_prefix(pkv_pool* p, const int32_t* tokens, int32_t n, int32_t* len) {
  std::vector<uint64_t> h;
  prefix_hashes(tokens, n, h);
  for (int32_t k = n; k >= 1; --k) {
    if (PrefixEntry* e = p->find_prefix(h[k - 1], tokens, k)) {
      *len = k;
      return e;
    }
  }
  *len = 0;
  return nullptr;
}

}  // namespace

pkv_status prefix_cache_lookup(pkv_pool* p, const int32_t* tokens, int32_t n, int32_t* matched,
                               int32_t* blocks, int32_t cap, int32_t* nblocks) {
  if (!p || n < 0 || (n > 0 && !tokens) || !matched || !nblocks || cap < 0)
    return PKV_ERR_INVALID_ARG;
  try {
    int32_t len = 0;
    PrefixEntry* e = n > 0 ? longest_prefix(p, tokens, n, &len) : nullptr;
    *matched = len;
    *nblocks = e ? static_cast<int32_t>(e->blocks.size()) : 0;
    if (!e) return PKV_OK;
    if (blocks && cap < *nblocks) return PKV_ERR_INVALID_ARG;
    if (blocks) std::memcpy(blocks, e->blocks.data(), e->blocks.size() * sizeof(int32_t));
    ++e->count;
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  return PKV_OK;
}

pkv_status seq_create_from_prefix(pkv_pool* p, int64_t sid, const int32_t* tokens, int32_t n,
                                  int32_t* matched) {
  if (!p || n < 0 || (n > 0 && !tokens) || !matched) return PKV_ERR_INVALID_ARG;
  if (p->seqs.count(sid)) return PKV_ERR_INVALID_ARG;
  try {
    int32_t len = 0;
    PrefixEntry* e = n > 0 ? longest_prefix(p, tokens, n, &len) : nullptr;
    *matched = 0;
    if (!e) return seq_create(p, sid);
    Seq s;
    s.table = e->blocks;
    s.len = len;
    p->touch(s);
    p->seqs.emplace(sid, std::move(s));
    for (int32_t b : e->blocks) ++p->ref[b];
    ++e->count;
    *matched = len;
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  return PKV_OK;
}

pkv_status prefix_cache_release(pkv_pool* p, const int32_t* tokens, int32_t n) {
  if (!p || n <= 0 || !tokens) return PKV_ERR_INVALID_ARG;
  try {
    std::vector<uint64_t> h;
    prefix_hashes(tokens, n, h);
    auto it = p->prefix.find(h[n - 1]);
    if (it == p->prefix.end()) return PKV_ERR_INVALID_ARG;
    auto& bucket = it->second;
    for (size_t i = 0; i < bucket.size(); ++i) {
      PrefixEntry& e = bucket[i];
      if (static_cast<int32_t>(e.tokens.size()) != n ||
          !std::equal(e.tokens.begin(), e.tokens.end(), tokens))
        continue;
      if (--e.count == 0) {
        for (int32_t b : e.blocks)
          if (--p->ref[b] == 0) p->push_back(b);
        bucket.erase(bucket.begin() + static_cast<std::ptrdiff_t>(i));
        if (bucket.empty()) p->prefix.erase(it);
      }
      return PKV_OK;
    }
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  return PKV_ERR_INVALID_ARG;
}

pkv_status prefix_cache_count(const pkv_pool* p, const int32_t* tokens, int32_t n,
                              int32_t* count) {
  if (!p || n <= 0 || !tokens || !count) return PKV_ERR_INVALID_ARG;
  try {
    std::vector<uint64_t> h;
    prefix_hashes(tokens, n, h);
    const PrefixEntry* e = const_cast<pkv_pool*>(p)->find_prefix(h[n - 1], tokens, n);
    *count = e ? e->count : 0;
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  return PKV_OK;
}

pkv_status kv_pool_host_init(pkv_pool* p, int64_t num_host_blocks) {
  if (!p || num_host_blocks <= 0 || num_host_blocks > INT32_MAX || p->host_blocks)
    return PKV_ERR_INVALID_ARG;
  try {
    p->host_ring.resize(num_host_blocks);
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  for (int64_t i = 0; i < num_host_blocks; ++i) p->host_ring[i] = static_cast<int32_t>(i);
  p->host_blocks = num_host_blocks;
  p->host_head = 0;
  p->host_count = num_host_blocks;
  return PKV_OK;
}

pkv_status pool_lru_order(const pkv_pool* p, int64_t* ids, int64_t cap, int64_t* n) {
  if (!p || !n || cap < 0) return PKV_ERR_INVALID_ARG;
  try {
    std::vector<std::pair<uint64_t, int64_t>> v;
    v.reserve(p->seqs.size());
    for (const auto& kv : p->seqs)
      if (kv.second.on_host.empty()) v.emplace_back(kv.second.last_use, kv.first);
    std::sort(v.begin(), v.end());
    *n = static_cast<int64_t>(v.size());
    if (cap < *n || (!ids && *n > 0)) return PKV_ERR_INVALID_ARG;
    for (size_t i = 0; i < v.size(); ++i) ids[i] = v[i].second;
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  return PKV_OK;
}

pkv_status seq_is_swapped(const pkv_pool* p, int64_t sid, int32_t* swapped) {
  if (!p || !swapped) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(sid);
  if (it == p->seqs.end()) return PKV_ERR_INVALID_ARG;
  *swapped = it->second.on_host.empty() ? 0 : 1;
  return PKV_OK;
}

pkv_status seq_swap_out(pkv_pool* p, int64_t sid, int32_t* pairs, int32_t cap, int32_t* n) {
  if (!p || !n || cap < 0) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(sid);
  if (it == p->seqs.end() || !it->second.on_host.empty()) return PKV_ERR_INVALID_ARG;
  Seq& s = it->second;
  int32_t k = 0;
  for (int32_t b : s.table)
    if (p->ref[b] == 1) ++k;
  *n = k;
  if (cap < k || (!pairs && k > 0)) return PKV_ERR_INVALID_ARG;
  if (k > p->host_count) return PKV_ERR_NO_FREE_BLOCK;
  try {
    s.on_host.assign(s.table.size(), 0);
  } catch (const std::bad_alloc&) {
    return PKV_ERR_HOST_MEMORY;
  }
  int32_t i = 0;
  for (size_t j = 0; j < s.table.size(); ++j) {
    const int32_t b = s.table[j];
    if (p->ref[b] != 1) continue;
    const int32_t h = p->host_pop();
    pairs[2 * i] = b;
    pairs[2 * i + 1] = h;
    ++i;
    p->ref[b] = 0;
    p->push_back(b);
    s.table[j] = h;
    s.on_host[j] = 1;
  }
  return PKV_OK;
}

pkv_status seq_swap_in(pkv_pool* p, int64_t sid, int32_t* pairs, int32_t cap, int32_t* n) {
  if (!p || !n || cap < 0) return PKV_ERR_INVALID_ARG;
  auto it = p->seqs.find(sid);
  if (it == p->seqs.end() || it->second.on_host.empty()) return PKV_ERR_INVALID_ARG;
  Seq& s = it->second;
  int32_t k = 0;
  for (uint8_t f : s.on_host) k += f;
  *n = k;
  if (cap < k || (!pairs && k > 0)) return PKV_ERR_INVALID_ARG;
  if (k > p->count) return PKV_ERR_NO_FREE_BLOCK;
  int32_t i = 0;
  for (size_t j = 0; j < s.table.size(); ++j) {
    if (!s.on_host[j]) continue;
    const int32_t b = p->pop_front();
    p->ref[b] = 1;
    pairs[2 * i] = s.table[j];
    pairs[2 * i + 1] = b;
    ++i;
    p->host_push(s.table[j]);
    s.table[j] = b;
  }
  s.on_host.clear();
  p->touch(s);
  return PKV_OK;
}

}  // extern "C"
