// Host page allocator and block-table builder (the KV block manager of a
// continuous-batching engine).
//
// Pages are handed out from a free list and returned when a sequence finishes, is
// preempted or rolls back rejected drafts ("Continuous Batching and Speculative
// Decoding: How Modern LLM Serving Engines Actually Work", sections "PagedAttention:
// making the KV cache schedulable" and "Continuous batching: scheduling per
// iteration"; "llm-inference-optimization-batching", sections "Anatomy of the KV
// Cache" -- reference counts keep shared prefix pages alive -- and "Speculative
// Decoding: Turning Verification Parallelism into Latency Wins" -- rollback of the
// rejected drafts).  A sequence of L tokens always owns exactly ceil(L / P) pages, so
// waste is bounded by one partially filled page per sequence.
#include <cstdint>
#include <map>
#include <unordered_map>
#include <vector>

#include "../../include/vas.h"

namespace {

struct Seq {
  int32_t len = 0;
  std::vector<int32_t> pages;
  uint64_t admitted = 0;  // admission order (larger = newer)
};

// splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
// OOPSLA 2014): a portable stream for the initial permutation of the free list.
uint64_t splitmix64(uint64_t& s) {
  uint64_t z = (s += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

int32_t pages_for(int64_t tokens, int32_t page_size) {
  return static_cast<int32_t>((tokens + page_size - 1) / page_size);
}

}  // namespace

struct vas_pool {
  int32_t num_pages = 0;
  int32_t page_size = 0;
  std::vector<int32_t> free_list;  // stack: back() is handed out next
  std::vector<int32_t> refcount;   // per page; 0 = free
  std::unordered_map<int64_t, Seq> seqs;
  std::map<uint64_t, int64_t> by_age;  // admission order -> id
  uint64_t clock = 0;

  int32_t take() {
    const int32_t id = free_list.back();
    free_list.pop_back();
    refcount[id] = 1;
    return id;
  }
  void release(int32_t id) {
    if (--refcount[id] == 0) free_list.push_back(id);
  }
  void drop(std::unordered_map<int64_t, Seq>::iterator it) {
    for (int32_t pg : it->second.pages) release(pg);
    by_age.erase(it->second.admitted);
    seqs.erase(it);
  }
};

extern "C" {

vas_pool* vas_pool_create(int32_t num_pages, int32_t page_size, uint64_t seed) {
  if (num_pages < 0 || page_size <= 0) return nullptr;
  vas_pool* p = new vas_pool;
  p->num_pages = num_pages;
  p->page_size = page_size;
  p->refcount.assign(static_cast<size_t>(num_pages), 0);
  std::vector<int32_t> order(static_cast<size_t>(num_pages));
  for (int32_t i = 0; i < num_pages; ++i) order[i] = i;
  if (seed != 0) {
    uint64_t s = seed;
    for (int32_t i = num_pages - 1; i > 0; --i) {
      const int32_t j = static_cast<int32_t>(splitmix64(s) % static_cast<uint64_t>(i + 1));
      const int32_t t = order[i];
      order[i] = order[j];
      order[j] = t;
    }
  }
  // hand pages out in `order`: the stack's back is order[0]
  p->free_list.assign(order.rbegin(), order.rend());
  return p;
}

void vas_pool_destroy(vas_pool* pool) { delete pool; }

int32_t vas_pool_free_pages(const vas_pool* pool) {
  return pool ? static_cast<int32_t>(pool->free_list.size()) : VAS_E_INVALID_ARG;
}

int32_t vas_pool_num_seqs(const vas_pool* pool) {
  return pool ? static_cast<int32_t>(pool->seqs.size()) : VAS_E_INVALID_ARG;
}

int vas_pool_can_allocate(const vas_pool* pool, int32_t n_tokens) {
  if (!pool || n_tokens < 0) return 0;
  return pages_for(n_tokens, pool->page_size) <= static_cast<int32_t>(pool->free_list.size());
}

int32_t vas_seq_pages_needed(const vas_pool* pool, int64_t seq_id, int32_t n_tokens) {
  if (!pool || n_tokens < 0) return VAS_E_INVALID_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return VAS_E_NOT_FOUND;
  const Seq& s = it->second;
  return pages_for(static_cast<int64_t>(s.len) + n_tokens, pool->page_size) -
         static_cast<int32_t>(s.pages.size());
}

int32_t vas_seq_len(const vas_pool* pool, int64_t seq_id) {
  if (!pool) return VAS_E_INVALID_ARG;
  auto it = pool->seqs.find(seq_id);
  return it == pool->seqs.end() ? VAS_E_NOT_FOUND : it->second.len;
}

int vas_seq_admit(vas_pool* pool, int64_t seq_id, int32_t n_tokens) {
  if (!pool || n_tokens < 0) return VAS_E_INVALID_ARG;
  if (pool->seqs.count(seq_id)) return VAS_E_EXISTS;
  const int32_t need = pages_for(n_tokens, pool->page_size);
  if (need > static_cast<int32_t>(pool->free_list.size())) return VAS_E_NOMEM;
  Seq s;
  s.len = n_tokens;
  s.pages.reserve(static_cast<size_t>(need));
  for (int32_t i = 0; i < need; ++i) s.pages.push_back(pool->take());
  s.admitted = ++pool->clock;
  pool->by_age[s.admitted] = seq_id;
  pool->seqs.emplace(seq_id, std::move(s));
  return VAS_OK;
}

int vas_seq_grow(vas_pool* pool, int64_t seq_id, int32_t n_tokens) {
  if (!pool || n_tokens < 0) return VAS_E_INVALID_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return VAS_E_NOT_FOUND;
  Seq& s = it->second;
  const int64_t new_len = static_cast<int64_t>(s.len) + n_tokens;
  if (new_len > INT32_MAX) return VAS_E_INVALID_ARG;
  // Appending into a partially filled page that another sequence shares would write
  // into the other sequence's prefix; forks never share a partial page, so this only
  // arises after a rollback into shared pages, which vas_seq_rollback refuses.
  const int32_t need = pages_for(new_len, pool->page_size) - static_cast<int32_t>(s.pages.size());
  if (need > static_cast<int32_t>(pool->free_list.size())) return VAS_E_NOMEM;
  for (int32_t i = 0; i < need; ++i) s.pages.push_back(pool->take());
  s.len = static_cast<int32_t>(new_len);
  return VAS_OK;
}

int vas_seq_rollback(vas_pool* pool, int64_t seq_id, int32_t n_tokens) {
  if (!pool || n_tokens < 0) return VAS_E_INVALID_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return VAS_E_NOT_FOUND;
  Seq& s = it->second;
  if (n_tokens > s.len) return VAS_E_INVALID_ARG;
  const int32_t new_len = s.len - n_tokens;
  const int32_t keep = pages_for(new_len, pool->page_size);
  // The page that becomes the partially filled last page must be exclusively owned,
  // otherwise the next append would overwrite a shared prefix.
  if (new_len % pool->page_size != 0 && keep > 0 && pool->refcount[s.pages[keep - 1]] > 1)
    return VAS_E_INVALID_ARG;
  while (static_cast<int32_t>(s.pages.size()) > keep) {
    pool->release(s.pages.back());
    s.pages.pop_back();
  }
  s.len = new_len;
  return VAS_OK;
}

int vas_seq_free(vas_pool* pool, int64_t seq_id) {
  if (!pool) return VAS_E_INVALID_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return VAS_E_NOT_FOUND;
  pool->drop(it);
  return VAS_OK;
}

int vas_pool_preempt_newest(vas_pool* pool, int64_t* victim) {
  if (!pool || !victim) return VAS_E_INVALID_ARG;
  if (pool->by_age.empty()) return VAS_E_NOT_FOUND;
  const int64_t id = pool->by_age.rbegin()->second;
  *victim = id;
  pool->drop(pool->seqs.find(id));
  return VAS_OK;
}

int vas_seq_fork(vas_pool* pool, int64_t parent_id, int64_t child_id, int32_t n_tokens) {
  if (!pool || n_tokens < 0) return VAS_E_INVALID_ARG;
  auto it = pool->seqs.find(parent_id);
  if (it == pool->seqs.end()) return VAS_E_NOT_FOUND;
  if (pool->seqs.count(child_id)) return VAS_E_EXISTS;
  const Seq& parent = it->second;
  if (n_tokens > parent.len) return VAS_E_INVALID_ARG;
  const int32_t shared = n_tokens / pool->page_size;  // full pages only
  const int32_t fresh = pages_for(n_tokens, pool->page_size) - shared;
  if (fresh > static_cast<int32_t>(pool->free_list.size())) return VAS_E_NOMEM;
  Seq c;
  c.len = n_tokens;
  for (int32_t i = 0; i < shared; ++i) {
    ++pool->refcount[parent.pages[i]];
    c.pages.push_back(parent.pages[i]);
  }
  for (int32_t i = 0; i < fresh; ++i) c.pages.push_back(pool->take());
  c.admitted = ++pool->clock;
  pool->by_age[c.admitted] = child_id;
  pool->seqs.emplace(child_id, std::move(c));
  return VAS_OK;
}

int32_t vas_page_refcount(const vas_pool* pool, int32_t page) {
  if (!pool || page < 0 || page >= pool->num_pages) return VAS_E_INVALID_ARG;
  return pool->refcount[page];
}

int vas_build_block_table(const vas_pool* pool, const int64_t* seq_ids, int32_t n,
                          int32_t* block_table, int32_t max_pages, int32_t* seq_lens) {
  if (!pool || n < 0 || max_pages < 0 || (n > 0 && (!seq_ids || !block_table || !seq_lens)))
    return VAS_E_INVALID_ARG;
  for (int32_t r = 0; r < n; ++r) {
    auto it = pool->seqs.find(seq_ids[r]);
    if (it == pool->seqs.end()) return VAS_E_NOT_FOUND;
    if (static_cast<int32_t>(it->second.pages.size()) > max_pages) return VAS_E_INVALID_ARG;
  }
  for (int32_t r = 0; r < n; ++r) {
    const Seq& s = pool->seqs.find(seq_ids[r])->second;
    int32_t* row = block_table + static_cast<int64_t>(r) * max_pages;
    const int32_t np = static_cast<int32_t>(s.pages.size());
    for (int32_t c = 0; c < max_pages; ++c) row[c] = c < np ? s.pages[c] : -1;
    seq_lens[r] = s.len;
  }
  return VAS_OK;
}

}  // extern "C"
