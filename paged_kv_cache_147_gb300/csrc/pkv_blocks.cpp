// pkv_blocks.cpp -- the host KV block pool: fixed-size blocks, a FIFO free list, reference
// counts, a prefix index of full blocks keyed by an FNV-1a hash chain over token ids, and
// copy-on-write of shared blocks before an append (the Ollama memory-management page, §三 KV
// Cache内存管理的工程实现 and its copy-on-write paragraph). It produces the block tables and
// the copy pairs that the CUDA entry points take (pkv_copy_blocks, the slot mapping, decode).
//
// Readings of the page (it leaves them open): a block's index key is the FNV-1a state after
// its last token continued from its parent block's (a chain over the whole prefix); only full
// blocks are indexed; a candidate is accepted only if its token ids and its parent block match
// (the token-level verification the page asks for against collisions); a block that leaves the
// index takes its indexed descendants with it (their parent id may be reused for other tokens,
// so the parent check would no longer prove the prefix), and those nobody holds are freed;
// releasing the last reference frees a block and removes it from the index; warm() indexes a
// prompt's blocks with no reference (the page's pre-warmed system prompt); when the free list
// is short, indexed unreferenced blocks are reclaimed oldest allocation first, and referenced
// blocks never are.
#include <algorithm>
#include <cstdint>
#include <deque>
#include <mutex>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/pkv.h"

struct pkv_block_pool {
  int nb = 0, bs = 0;
  uint64_t mask = ~0ull;
  std::vector<int> ref, parent;
  std::vector<uint8_t> indexed;
  std::vector<uint64_t> key, chain;
  std::vector<int64_t> stamp;
  std::vector<std::vector<int32_t>> toks;
  std::vector<std::vector<int>> kids;                    // indexed children, registration order
  std::deque<int> free_list;
  std::unordered_map<uint64_t, std::vector<int>> index;   // key -> blocks, registration order
  std::set<std::pair<int64_t, int>> warm;                // (allocation stamp, block) of the
                                                         // indexed blocks nobody holds
  int64_t clock = 0;
  std::mutex mu;
};

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

uint64_t fnv1a(const int32_t* t, int n, uint64_t h) {
  for (int i = 0; i < n; ++i) {
    h ^= static_cast<uint64_t>(static_cast<uint32_t>(t[i]));
    h *= kFnvPrime;
  }
  return h;
}

// Removes b from the index. Its indexed descendants leave the index with it: once b's id can
// be handed out for other tokens, a child's (parent id, tokens) check no longer proves that the
// child follows the same prefix. A descendant nobody holds goes to the back of the free list
// (pre-order: a block before its own descendants, children in registration order).
void unindex(pkv_block_pool* p, int b) {
  if (!p->indexed[b]) return;
  if (p->ref[b] == 0) p->warm.erase({p->stamp[b], b});
  auto it = p->index.find(p->key[b]);
  if (it != p->index.end()) {
    auto& v = it->second;
    v.erase(std::find(v.begin(), v.end(), b));
    if (v.empty()) p->index.erase(it);
  }
  const int par = p->parent[b];
  if (par >= 0) {
    auto& k = p->kids[par];
    auto kt = std::find(k.begin(), k.end(), b);
    if (kt != k.end()) k.erase(kt);
  }
  p->indexed[b] = 0;
  p->toks[b].clear();
  std::vector<int> kids;
  kids.swap(p->kids[b]);
  for (int c : kids) {
    if (!p->indexed[c]) continue;
    p->parent[c] = -1;                    // b's list is already detached
    if (p->ref[c] == 0) p->free_list.push_back(c);
    unindex(p, c);
  }
}

void index_block(pkv_block_pool* p, int b, int parent, uint64_t chain, const int32_t* t) {
  p->indexed[b] = 1;
  p->key[b] = chain & p->mask;
  p->chain[b] = chain;
  p->parent[b] = parent;
  p->toks[b].assign(t, t + p->bs);
  p->index[p->key[b]].push_back(b);
  if (parent >= 0) p->kids[parent].push_back(b);
}

// Reference changes keep the warm set: an indexed block enters it at reference 0 and leaves it
// when it is held again (or unindexed).
void inc_ref(pkv_block_pool* p, int b) {
  if (p->ref[b]++ == 0 && p->indexed[b]) p->warm.erase({p->stamp[b], b});
}

void dec_ref(pkv_block_pool* p, int b) {
  if (--p->ref[b] == 0 && p->indexed[b]) p->warm.insert({p->stamp[b], b});
}

int match(pkv_block_pool* p, int parent, uint64_t chain, const int32_t* t) {
  auto it = p->index.find(chain & p->mask);
  if (it == p->index.end()) return -1;
  for (int b : it->second)
    if (p->parent[b] == parent && std::equal(t, t + p->bs, p->toks[b].begin())) return b;
  return -1;
}

// Takes n blocks from the front of the free list, first reclaiming indexed unreferenced
// blocks (oldest allocation first) if it is short. All or nothing.
bool take(pkv_block_pool* p, int n, std::vector<int>& out) {
  // eviction moves warm blocks (and orphaned warm descendants) to the free list, so free +
  // warm is what can be had
  if (static_cast<int>(p->free_list.size() + p->warm.size()) < n) return false;
  while (static_cast<int>(p->free_list.size()) < n) {
    const int b = p->warm.begin()->second;        // oldest allocation first
    p->free_list.push_back(b);
    unindex(p, b);
  }
  for (int i = 0; i < n; ++i) {
    const int b = p->free_list.front();
    p->free_list.pop_front();
    p->stamp[b] = ++p->clock;
    out.push_back(b);
  }
  return true;
}

bool valid_table(const pkv_block_pool* p, const int32_t* table, int n) {
  if (n < 0 || (n > 0 && !table)) return false;
  for (int i = 0; i < n; ++i)
    if (table[i] < 0 || table[i] >= p->nb || p->ref[table[i]] < 1) return false;
  return true;
}

// allocate without locking; refs of the matched prefix are taken before new blocks
int allocate_locked(pkv_block_pool* p, const int32_t* tokens, int n_tokens, int max_tokens,
                    int32_t* table, int table_cap, int* n_blocks, int* reused) {
  const int bs = p->bs;
  if (max_tokens < n_tokens) max_tokens = n_tokens;
  std::vector<int> got;
  int parent = -1, pos = 0;
  uint64_t h = kFnvOffset;
  while (pos + bs <= n_tokens) {
    const uint64_t h2 = fnv1a(tokens + pos, bs, h);
    const int b = match(p, parent, h2, tokens + pos);
    if (b < 0) break;
    got.push_back(b);
    parent = b;
    h = h2;
    pos += bs;
  }
  const int n_reused = static_cast<int>(got.size());
  const int need = (max_tokens - pos + bs - 1) / bs;
  if (n_reused + need > table_cap) return PKV_EINVAL;
  for (int b : got) inc_ref(p, b);
  std::vector<int> fresh;
  if (!take(p, need, fresh)) {
    for (int b : got) dec_ref(p, b);
    return PKV_ENOSPC;
  }
  for (int b : fresh) {
    p->ref[b] = 1;
    if (pos + bs <= n_tokens) {
      const uint64_t h2 = fnv1a(tokens + pos, bs, h);
      index_block(p, b, parent, h2, tokens + pos);
      parent = b;
      h = h2;
    }
    pos += bs;
    got.push_back(b);
  }
  for (size_t i = 0; i < got.size(); ++i) table[i] = got[i];
  *n_blocks = static_cast<int>(got.size());
  if (reused) *reused = n_reused;
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_pool_create(int num_blocks, int block_size, int hash_bits, pkv_block_pool** out) {
  if (!out || num_blocks < 1 || block_size < 1 || hash_bits < 1 || hash_bits > 64)
    return PKV_EINVAL;
  auto* p = new (std::nothrow) pkv_block_pool;
  if (!p) return PKV_ENOSPC;
  p->nb = num_blocks;
  p->bs = block_size;
  p->mask = hash_bits >= 64 ? ~0ull : ((1ull << hash_bits) - 1);
  p->ref.assign(num_blocks, 0);
  p->parent.assign(num_blocks, -1);
  p->indexed.assign(num_blocks, 0);
  p->key.assign(num_blocks, 0);
  p->chain.assign(num_blocks, 0);
  p->stamp.assign(num_blocks, 0);
  p->toks.assign(num_blocks, {});
  p->kids.assign(num_blocks, {});
  for (int b = 0; b < num_blocks; ++b) p->free_list.push_back(b);
  *out = p;
  return PKV_OK;
}

void pkv_pool_destroy(pkv_block_pool* pool) { delete pool; }

int pkv_pool_allocate(pkv_block_pool* pool, const int32_t* tokens, int n_tokens, int max_tokens,
                      int32_t* table, int table_cap, int* n_blocks, int* reused) {
  if (!pool || n_tokens < 0 || (n_tokens > 0 && !tokens) || !table || !n_blocks ||
      table_cap < 0)
    return PKV_EINVAL;
  std::lock_guard<std::mutex> lock(pool->mu);
  return allocate_locked(pool, tokens, n_tokens, max_tokens, table, table_cap, n_blocks, reused);
}

int pkv_pool_warm(pkv_block_pool* pool, const int32_t* tokens, int n_tokens) {
  if (!pool || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PKV_EINVAL;
  std::lock_guard<std::mutex> lock(pool->mu);
  const int full = (n_tokens / pool->bs) * pool->bs;
  std::vector<int32_t> table(full / pool->bs + 1);
  int n = 0;
  const int st = allocate_locked(pool, tokens, full, full, table.data(),
                                 static_cast<int>(table.size()), &n, nullptr);
  if (st != PKV_OK) return st;
  for (int i = 0; i < n; ++i) dec_ref(pool, table[i]);
  return PKV_OK;
}

int pkv_pool_release(pkv_block_pool* pool, const int32_t* table, int n_blocks) {
  if (!pool) return PKV_EINVAL;
  std::lock_guard<std::mutex> lock(pool->mu);
  if (!valid_table(pool, table, n_blocks)) return PKV_EINVAL;
  for (int i = 0; i < n_blocks; ++i) {
    const int b = table[i];
    dec_ref(pool, b);
    if (pool->ref[b] == 0) {
      pool->free_list.push_back(b);
      unindex(pool, b);
    }
  }
  return PKV_OK;
}

int pkv_pool_fork(pkv_block_pool* pool, const int32_t* table, int n_blocks) {
  if (!pool) return PKV_EINVAL;
  std::lock_guard<std::mutex> lock(pool->mu);
  if (!valid_table(pool, table, n_blocks)) return PKV_EINVAL;
  for (int i = 0; i < n_blocks; ++i) inc_ref(pool, table[i]);
  return PKV_OK;
}

int pkv_pool_append(pkv_block_pool* pool, int32_t* table, int* n_blocks, int table_cap,
                    int length, int n_new, const int32_t* all_tokens, int32_t* copy_src,
                    int32_t* copy_dst, int copy_cap, int* n_copies) {
  if (!pool || !table || !n_blocks || !n_copies || length < 0 || n_new < 0 || copy_cap < 0 ||
      (copy_cap > 0 && (!copy_src || !copy_dst)))
    return PKV_EINVAL;
  std::lock_guard<std::mutex> lock(pool->mu);
  const int bs = pool->bs;
  const int nb0 = *n_blocks;
  if (!valid_table(pool, table, nb0) || nb0 > table_cap) return PKV_EINVAL;
  *n_copies = 0;
  if (n_new == 0) return PKV_OK;
  const int first = length / bs, last = (length + n_new - 1) / bs;
  if (first > nb0 || last + 1 > table_cap) return PKV_EINVAL;
  // count the blocks needed first: all or nothing
  int need = 0, copies = 0;
  for (int j = first; j <= last; ++j) {
    if (j >= nb0) ++need;
    else if (pool->ref[table[j]] > 1) { ++need; ++copies; }
  }
  if (copies > copy_cap) return PKV_EINVAL;
  std::vector<int> fresh;
  if (!take(pool, need, fresh)) return PKV_ENOSPC;
  int used = 0, nb = nb0;
  for (int j = first; j <= last; ++j) {
    if (j < nb0 && pool->ref[table[j]] > 1) {
      const int d = fresh[used++];
      pool->ref[d] = 1;
      dec_ref(pool, table[j]);
      copy_src[*n_copies] = table[j];
      copy_dst[*n_copies] = d;
      ++*n_copies;
      table[j] = d;
    } else if (j >= nb0) {
      const int d = fresh[used++];
      pool->ref[d] = 1;
      table[nb++] = d;
    }
  }
  *n_blocks = nb;
  // index the blocks this append filled, when their parent is indexed
  if (all_tokens) {
    for (int j = length / bs; j < (length + n_new) / bs; ++j) {
      const int b = table[j];
      if (pool->indexed[b]) continue;
      const int parent = j > 0 ? table[j - 1] : -1;
      if (j > 0 && !pool->indexed[parent]) continue;
      const uint64_t h = j > 0 ? pool->chain[parent] : kFnvOffset;
      index_block(pool, b, parent, fnv1a(all_tokens + static_cast<int64_t>(j) * bs, bs, h),
                  all_tokens + static_cast<int64_t>(j) * bs);
    }
  }
  return PKV_OK;
}

int pkv_pool_stats(pkv_block_pool* pool, int* total, int* used, int* shared, int* free_blocks,
                   int* warm) {
  if (!pool) return PKV_EINVAL;
  std::lock_guard<std::mutex> lock(pool->mu);
  int u = 0, s = 0;
  for (int b = 0; b < pool->nb; ++b) {
    u += pool->ref[b] > 0;
    s += pool->ref[b] > 1;
  }
  const int w = static_cast<int>(pool->warm.size());
  if (total) *total = pool->nb;
  if (used) *used = u;
  if (shared) *shared = s;
  if (free_blocks) *free_blocks = static_cast<int>(pool->free_list.size());
  if (warm) *warm = w;
  return PKV_OK;
}

int pkv_pool_refcount(pkv_block_pool* pool, int block) {
  if (!pool || block < 0 || block >= pool->nb) return PKV_EINVAL;
  std::lock_guard<std::mutex> lock(pool->mu);
  return pool->ref[block];
}

}  // extern "C"
