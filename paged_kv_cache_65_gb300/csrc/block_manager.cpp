// Host control plane of the paged KV cache: FIFO free list, per-block
// reference counts, per-sequence block tables, fork, release and
// copy-on-write decisions.
//
// Semantics follow "PagedAttention 的块表与碎片控制" §03-§05 (address
// translation, allocate only when the tail block is full, FIFO free list,
// MemoryError on an empty list), §10 (reserve a whole step atomically before
// launching) and §13 (conservation checks), and "KV 缓存管理", section
// "通过写时复制分支实现零复制审慎推理" (fork = table copy + one more count
// per block + child length = parent length; copy-on-write of a shared tail;
// release walks the table and returns blocks at count 0).
//
// Every mutating call first checks that it can succeed (ids, duplicates,
// handles, free blocks needed) and only then changes state, so a failing
// call changes nothing.

#include <cmath>
#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>

#include "pool.h"

namespace {

int64_t blocks_for(int64_t tokens, int B) { return (tokens + B - 1) / B; }

bool valid_id(const kvPool* p, int32_t id) { return id >= 0 && id < p->N; }

void push_free(kvPool* p, int32_t id) { p->free_list.push_back(id); }

// ------------------------------------------------------------ prefix cache
// ("KV 缓存管理", radix-tree section: full blocks only, block-aligned
// truncation, leaf-first LRU eviction of dormant nodes.)

// splitmix64's finalizer, a 64-bit mixing step
uint64_t mix64(uint64_t x) {
  x ^= x >> 30;
  x *= 0xbf58476d1ce4e5b9ULL;
  x ^= x >> 27;
  x *= 0x94d049bb133111ebULL;
  x ^= x >> 31;
  return x;
}
// h_k = H(h_{k-1} || tokens of block k); lookups verify the tokens and the
// parent, so the hash only has to spread the keys
uint64_t pc_chain(uint64_t h, const int32_t* t, int B) {
  h = mix64(h + 0x9e3779b97f4a7c15ULL);
  for (int i = 0; i < B; ++i) h = mix64(h ^ static_cast<uint32_t>(t[i]));
  return h;
}
uint64_t pc_root(const kvPool* p) { return mix64(p->pc_salt ^ 0x632be59bd9b4e019ULL); }

int64_t available(const kvPool* p) {
  return static_cast<int64_t>(p->free_list.size()) + p->pc_n_dormant;
}

void pc_tick(kvPool* p, int32_t id) { p->pc_nodes[id].last = ++p->pc_clock; }

// the cached child of `parent` holding `t` (one block of tokens), or -1
int32_t pc_find(const kvPool* p, uint64_t h, int32_t parent, const int32_t* t) {
  auto r = p->pc_index.equal_range(h);
  for (auto it = r.first; it != r.second; ++it) {
    const kvPrefixNode& n = p->pc_nodes.at(it->second);
    if (n.parent == parent && std::equal(n.tokens.begin(), n.tokens.end(), t)) return it->second;
  }
  return -1;
}

// Evict the least recently used dormant leaf: its block returns to the free
// list, and its parent becomes a candidate if it is left without children
// and is itself dormant.
bool pc_evict_one(kvPool* p) {
  if (p->pc_lru.empty()) return false;
  const int32_t id = p->pc_lru.begin()->second;
  p->pc_lru.erase(p->pc_lru.begin());
  const kvPrefixNode n = p->pc_nodes.at(id);
  auto r = p->pc_index.equal_range(n.hash);
  for (auto it = r.first; it != r.second; ++it)
    if (it->second == id) {
      p->pc_index.erase(it);
      break;
    }
  p->pc_nodes.erase(id);
  p->pc_dormant[id] = 0;
  p->pc_n_dormant -= 1;
  if (n.parent >= 0) {
    kvPrefixNode& q = p->pc_nodes.at(n.parent);
    q.children -= 1;
    if (q.children == 0 && p->pc_dormant[n.parent]) p->pc_lru.insert({q.last, n.parent});
  }
  push_free(p, id);
  return true;
}

// Caller has checked available(p) > 0: with an empty free list a dormant
// leaf exists, since every descendant of a dormant node is dormant.
int32_t pop_free(kvPool* p) {
  if (p->free_list.empty()) pc_evict_one(p);
  int32_t id = p->free_list.front();
  p->free_list.pop_front();
  return id;
}

// A block's count reached zero: a cached block turns dormant, others free.
void count_zero(kvPool* p, int32_t id) {
  auto it = p->pc_on ? p->pc_nodes.find(id) : p->pc_nodes.end();
  if (it == p->pc_nodes.end()) {
    push_free(p, id);
    return;
  }
  p->pc_dormant[id] = 1;
  p->pc_n_dormant += 1;
  pc_tick(p, id);
  if (it->second.children == 0) p->pc_lru.insert({it->second.last, id});
}

// Publish the blocks of a sequence that are full now, from logical block
// `first_full` on: a block joins the cache when its tokens are known, its key
// is not cached yet and the block before it in the table is a cached node
// (or it is the first block).
void pc_publish(kvPool* p, int32_t seq_id, int64_t first_full) {
  if (!p->pc_on) return;
  kvSeq& s = p->seqs[seq_id];
  const int B = p->B;
  const int64_t n_full = s.len / B;
  for (int64_t k = first_full; k < n_full; ++k) {
    const int32_t id = s.table[k];
    if (p->pc_nodes.count(id)) continue;
    bool all_known = true;
    for (int64_t i = k * B; i < (k + 1) * B; ++i) all_known = all_known && s.known[i];
    if (!all_known) continue;
    const int32_t parent = k > 0 ? s.table[k - 1] : -1;
    if (k > 0 && !p->pc_nodes.count(parent)) continue;
    const uint64_t h = pc_chain(k > 0 ? p->pc_nodes.at(parent).hash : pc_root(p), &s.tok[k * B], B);
    if (pc_find(p, h, parent, &s.tok[k * B]) >= 0) continue;
    kvPrefixNode n;
    n.hash = h;
    n.parent = parent;
    n.tokens.assign(s.tok.begin() + k * B, s.tok.begin() + (k + 1) * B);
    p->pc_nodes.emplace(id, std::move(n));
    p->pc_index.insert({h, id});
    if (parent >= 0) p->pc_nodes.at(parent).children += 1;
    pc_tick(p, id);
  }
}

void record_tokens(kvPool* p, kvSeq& s, const int32_t* ids, int n) {
  if (!p->pc_on) return;
  for (int i = 0; i < n; ++i) {
    s.tok.push_back(ids ? ids[i] : 0);
    s.known.push_back(ids ? 1 : 0);
  }
}

// One token for sequence s.  Caller has already checked that a free block
// is available whenever this needs one.
void append_one(kvPool* p, kvSeq& s, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
  const int64_t j = s.len / p->B;  // logical block
  const int64_t o = s.len % p->B;  // offset in block
  *cow_src = -1;
  *cow_dst = -1;
  if (j == static_cast<int64_t>(s.table.size())) {
    int32_t id = pop_free(p);
    p->ref[id] = 1;
    s.table.push_back(id);
  } else if (p->ref[s.table[j]] > 1) {
    int32_t old = s.table[j];
    int32_t id = pop_free(p);
    p->ref[old] -= 1;
    p->ref[id] = 1;
    s.table[j] = id;
    *cow_src = old;
    *cow_dst = id;
  }
  s.len += 1;
  *slot = static_cast<int64_t>(s.table[j]) * p->B + o;
}

// Blocks a batch of single-token appends would take from the free list,
// counting copy-on-writes with the counts as they evolve inside the batch
// (seqs[i]: the i-th listed sequence, nullptr for a new one).
int64_t blocks_needed(const kvPool* p, kvSeq* const* seqs, int n) {
  std::unordered_map<int32_t, int32_t> drop;  // shared tail id -> counts dropped so far
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    const kvSeq* s = seqs[i];
    if (!s) {
      need += 1;
      continue;
    }
    const int64_t j = s->len / p->B;
    if (j == static_cast<int64_t>(s->table.size())) {
      need += 1;
    } else {
      const int32_t tail = s->table[j];
      if (p->ref[tail] <= 1) continue;  // a private tail takes the token in place
      int32_t& d = drop[tail];
      if (p->ref[tail] - d > 1) {
        need += 1;
        d += 1;
      }
    }
  }
  return need;
}

// Per-thread working arrays of the batch reservation (reused across calls).
struct AppendScratch {
  std::vector<int32_t> sorted;
  std::vector<kvSeq*> seqs;
  std::vector<const kvSeq*> cseqs;
  std::vector<int64_t> first_full;
};
thread_local AppendScratch t_append;

}  // namespace

extern "C" {

const char* kv_status_string(kvStatus s) {
  switch (s) {
    case KV_OK: return "ok";
    case KV_ERR_NO_FREE_BLOCK: return "no free KV block";
    case KV_ERR_INVALID_ARG: return "invalid argument";
    case KV_ERR_REFCOUNT: return "reference count error";
    case KV_ERR_CUDA: return "CUDA error";
    case KV_ERR_DEVICE_CHECK: return "device check failed";
    case KV_ERR_UNSUPPORTED: return "unsupported shape";
    case KV_ERR_SCRATCH_TOO_SMALL: return "request exceeds the static scratch size";
    default: return "unknown status";
  }
}

kvStatus kv_pool_create(int n_layers, int n_blocks, int block_size, int n_kv_heads, int head_dim,
                        int dtype, void* k_cache, void* v_cache, int32_t* d_status,
                        const int32_t* free_order, kvPool** out) {
  if (!out) return KV_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_layers <= 0 || n_blocks <= 0 || block_size <= 0 || block_size > 256 || n_kv_heads <= 0 ||
      head_dim <= 0 ||
      (dtype != KV_DTYPE_F32 && dtype != KV_DTYPE_BF16 && dtype != KV_DTYPE_FP8_E4M3 &&
       dtype != KV_DTYPE_Q8_0))
    return KV_ERR_INVALID_ARG;
  // q8_0: whole groups of 32 per head row, and one block's scales of a head
  // (B * D_h / 32 fp16) times H_kv in whole 16-byte vectors
  if (dtype == KV_DTYPE_Q8_0 &&
      (head_dim % 32 != 0 ||
       (static_cast<int64_t>(n_kv_heads) * block_size * (head_dim / 32) * 2) % 16 != 0))
    return KV_ERR_INVALID_ARG;
  if ((k_cache == nullptr) != (v_cache == nullptr)) return KV_ERR_INVALID_ARG;
  const int esize = dtype == KV_DTYPE_F32 ? 4 : (dtype == KV_DTYPE_BF16 ? 2 : 1);
  if (k_cache && ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15))
    return KV_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(n_kv_heads) * head_dim * esize) % 16 != 0) return KV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_layers) * n_blocks * block_size >= (int64_t(1) << 31))
    return KV_ERR_INVALID_ARG;
  if (free_order) {
    std::vector<char> seen(n_blocks, 0);
    for (int i = 0; i < n_blocks; ++i) {
      int32_t id = free_order[i];
      if (id < 0 || id >= n_blocks || seen[id]) return KV_ERR_INVALID_ARG;
      seen[id] = 1;
    }
  }
  kvPool* p = new (std::nothrow) kvPool();
  if (!p) return KV_ERR_INVALID_ARG;
  p->L = n_layers;
  p->N = n_blocks;
  p->B = block_size;
  p->H = n_kv_heads;
  p->D = head_dim;
  p->dtype = dtype;
  p->esize = esize;
  p->in_esize = dtype == KV_DTYPE_F32 ? 4 : 2;
  p->k = k_cache;
  p->v = v_cache;
  p->d_status = d_status;
  p->ref.assign(n_blocks, 0);
  p->ext.assign(n_blocks, 0);
  for (int i = 0; i < n_blocks; ++i) p->free_list.push_back(free_order ? free_order[i] : i);
  *out = p;
  return KV_OK;
}

void kv_pool_destroy(kvPool* pool) { delete pool; }

kvStatus kv_pool_stats(const kvPool* p, int* n_free, int* n_allocated, int* n_shared) {
  if (!p) return KV_ERR_INVALID_ARG;
  int shared = 0;
  for (int32_t c : p->ref) shared += c > 1;
  if (n_free) *n_free = static_cast<int>(p->free_list.size());
  if (n_allocated) *n_allocated = p->N - static_cast<int>(p->free_list.size());
  if (n_shared) *n_shared = shared;
  return KV_OK;
}

kvStatus kv_pool_check(const kvPool* p) {
  if (!p) return KV_ERR_INVALID_ARG;
  std::vector<char> is_free(p->N, 0);
  for (int32_t id : p->free_list) {
    if (!valid_id(p, id) || is_free[id]) return KV_ERR_REFCOUNT;
    is_free[id] = 1;
  }
  std::vector<int64_t> table_refs(p->N, 0);
  for (const auto& kv : p->seqs) {
    const kvSeq& s = kv.second;
    if (static_cast<int64_t>(s.table.size()) != blocks_for(s.len, p->B)) return KV_ERR_REFCOUNT;
    for (int32_t id : s.table) {
      if (!valid_id(p, id)) return KV_ERR_REFCOUNT;
      table_refs[id] += 1;
    }
  }
  int64_t n_alloc = 0, n_dormant = 0;
  for (int i = 0; i < p->N; ++i) {
    const bool dormant = p->pc_on && p->pc_dormant[i];
    if ((p->ref[i] > 0) + static_cast<int>(is_free[i]) + static_cast<int>(dormant) != 1)
      return KV_ERR_REFCOUNT;
    if (p->ref[i] < 0 || p->ext[i] < 0) return KV_ERR_REFCOUNT;
    if (p->ref[i] != table_refs[i] + p->ext[i]) return KV_ERR_REFCOUNT;
    n_alloc += p->ref[i] > 0;
    n_dormant += dormant;
  }
  if (static_cast<int64_t>(p->free_list.size()) + n_alloc + n_dormant != p->N)
    return KV_ERR_REFCOUNT;
  if (n_dormant != p->pc_n_dormant) return KV_ERR_REFCOUNT;
  // the cache is a tree of cached blocks; the eviction set is exactly the
  // dormant leaves
  std::unordered_map<int32_t, int32_t> kids;
  size_t n_leaves = 0;
  for (const auto& kv : p->pc_nodes) {
    const int32_t id = kv.first;
    if (!valid_id(p, id) || is_free[id]) return KV_ERR_REFCOUNT;
    if (kv.second.parent >= 0) {
      if (!p->pc_nodes.count(kv.second.parent)) return KV_ERR_REFCOUNT;
      kids[kv.second.parent] += 1;
    }
    if (static_cast<bool>(p->pc_dormant[id]) != (p->ref[id] == 0)) return KV_ERR_REFCOUNT;
  }
  for (const auto& kv : p->pc_nodes) {
    const int32_t want = kids.count(kv.first) ? kids.at(kv.first) : 0;
    if (kv.second.children != want) return KV_ERR_REFCOUNT;
    const bool leaf = p->pc_dormant[kv.first] && want == 0;
    if (leaf != static_cast<bool>(p->pc_lru.count({kv.second.last, kv.first})))
      return KV_ERR_REFCOUNT;
    n_leaves += leaf;
  }
  if (n_leaves != p->pc_lru.size()) return KV_ERR_REFCOUNT;
  return KV_OK;
}

kvStatus kv_pool_set_option(kvPool* p, int option, int value) {
  if (!p) return KV_ERR_INVALID_ARG;
  if (option == KV_OPT_DECODE_PATH && value >= 0 && value <= 3) {
    p->decode_path = value;
    for (int& g : p->grid_by_g) g = 0;  // grid sizes depend on the kernel
    p->grid_tc = 0;
    return KV_OK;
  }
  if (option == KV_OPT_PDL && (value == 0 || value == 1)) {
    p->pdl = value == 1;
    return KV_OK;
  }
  if (option == KV_OPT_PLAN_GRID && value >= 0 && value <= kMaxDecodeCtas) {
    p->plan_grid = value;
    return KV_OK;
  }
  return KV_ERR_INVALID_ARG;
}

kvStatus kv_pool_set_q8_scales(kvPool* p, void* k_scales, void* v_scales) {
  if (!p || p->dtype != KV_DTYPE_Q8_0 || !k_scales || !v_scales) return KV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_scales) | reinterpret_cast<uintptr_t>(v_scales)) & 15)
    return KV_ERR_INVALID_ARG;
  p->k_sc = k_scales;
  p->v_sc = v_scales;
  return KV_OK;
}

kvStatus kv_pool_set_fp8_scales(kvPool* p, float k_scale, float v_scale) {
  if (!p || p->dtype != KV_DTYPE_FP8_E4M3) return KV_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return KV_ERR_INVALID_ARG;
  p->k_scale = k_scale;
  p->v_scale = v_scale;
  return KV_OK;
}

kvStatus kv_block_refcount(const kvPool* p, int32_t id, int* out) {
  if (!p || !out || !valid_id(p, id)) return KV_ERR_INVALID_ARG;
  *out = p->ref[id];
  return KV_OK;
}

// ------------------------------------------------------------ block level

kvStatus block_alloc(kvPool* p, int n, int32_t* out_ids) {
  if (!p || n < 0 || (n > 0 && !out_ids)) return KV_ERR_INVALID_ARG;
  if (static_cast<size_t>(n) > p->free_list.size()) return KV_ERR_NO_FREE_BLOCK;
  for (int i = 0; i < n; ++i) {
    int32_t id = pop_free(p);
    p->ref[id] = 1;
    p->ext[id] = 1;
    out_ids[i] = id;
  }
  return KV_OK;
}

kvStatus block_free(kvPool* p, const int32_t* ids, int n) {
  if (!p || n < 0 || (n > 0 && !ids)) return KV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!valid_id(p, ids[i])) return KV_ERR_INVALID_ARG;
  std::unordered_map<int32_t, int32_t> need;
  for (int i = 0; i < n; ++i) need[ids[i]] += 1;
  for (const auto& kv : need)
    if (p->ext[kv.first] < kv.second) return KV_ERR_REFCOUNT;
  for (int i = 0; i < n; ++i) {
    int32_t id = ids[i];
    p->ref[id] -= 1;
    p->ext[id] -= 1;
    if (p->ref[id] == 0) count_zero(p, id);
  }
  return KV_OK;
}

kvStatus block_fork(kvPool* p, const int32_t* ids, int n) {
  if (!p || n < 0 || (n > 0 && !ids)) return KV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!valid_id(p, ids[i])) return KV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (p->ref[ids[i]] == 0) return KV_ERR_REFCOUNT;
  for (int i = 0; i < n; ++i) {
    p->ref[ids[i]] += 1;
    p->ext[ids[i]] += 1;
  }
  return KV_OK;
}

kvStatus block_cow(kvPool* p, int32_t id, int32_t* out_id) {
  if (!p || !out_id || !valid_id(p, id)) return KV_ERR_INVALID_ARG;
  if (p->ext[id] < 1) return KV_ERR_REFCOUNT;
  if (p->ref[id] == 1) {
    *out_id = id;
    return KV_OK;
  }
  if (available(p) == 0) return KV_ERR_NO_FREE_BLOCK;
  int32_t nid = pop_free(p);
  p->ref[id] -= 1;
  p->ext[id] -= 1;
  p->ref[nid] = 1;
  p->ext[nid] = 1;
  *out_id = nid;
  return KV_OK;
}

// --------------------------------------------------------- sequence level

kvStatus seq_append_slots(kvPool* p, const int32_t* seq_ids, int n_seq, int64_t* out_slots,
                          int32_t* out_cow_pairs, int* out_n_cow) {
  return seq_append_slots_ids(p, seq_ids, n_seq, nullptr, out_slots, out_cow_pairs, out_n_cow);
}

kvStatus seq_append_slots_ids(kvPool* p, const int32_t* seq_ids, int n_seq,
                              const int32_t* token_ids, int64_t* out_slots,
                              int32_t* out_cow_pairs, int* out_n_cow) {
  if (!p || n_seq < 0 || (n_seq > 0 && (!seq_ids || !out_slots || !out_cow_pairs)))
    return KV_ERR_INVALID_ARG;
  AppendScratch& sc = t_append;
  {
    std::vector<int32_t>& sorted = sc.sorted;
    sorted.assign(seq_ids, seq_ids + n_seq);
    std::sort(sorted.begin(), sorted.end());
    if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return KV_ERR_INVALID_ARG;
  }
  // each listed sequence looked up once (elements of the map keep their
  // addresses when others are inserted)
  std::vector<kvSeq*>& seqs = sc.seqs;
  seqs.assign(n_seq, nullptr);
  for (int i = 0; i < n_seq; ++i) {
    auto it = p->seqs.find(seq_ids[i]);
    if (it == p->seqs.end()) continue;
    if (it->second.len >= (int64_t(1) << 40)) return KV_ERR_INVALID_ARG;
    seqs[i] = &it->second;
  }
  if (blocks_needed(p, seqs.data(), n_seq) > available(p)) return KV_ERR_NO_FREE_BLOCK;
  std::vector<int64_t>& first_full = sc.first_full;
  first_full.assign(n_seq, 0);
  for (int i = 0; i < n_seq; ++i) first_full[i] = seqs[i] ? seqs[i]->len / p->B : 0;
  int n_cow = 0;
  for (int i = 0; i < n_seq; ++i) {
    if (!seqs[i]) seqs[i] = &p->seqs[seq_ids[i]];  // a new sequence
    int32_t src, dst;
    append_one(p, *seqs[i], &out_slots[i], &src, &dst);
    if (src >= 0) {
      out_cow_pairs[2 * n_cow] = src;
      out_cow_pairs[2 * n_cow + 1] = dst;
      ++n_cow;
    }
  }
  if (p->pc_on) {
    for (int i = 0; i < n_seq; ++i)
      record_tokens(p, *seqs[i], token_ids ? token_ids + i : nullptr, 1);
    for (int i = 0; i < n_seq; ++i) pc_publish(p, seq_ids[i], first_full[i]);
  }
  if (out_n_cow) *out_n_cow = n_cow;
  return KV_OK;
}

kvStatus seq_append_tokens(kvPool* p, int32_t seq, int n_tokens, int64_t* out_slots,
                           int32_t* out_cow_pair, int* out_n_cow) {
  return seq_append_tokens_ids(p, seq, n_tokens, nullptr, out_slots, out_cow_pair, out_n_cow);
}

kvStatus seq_append_tokens_ids(kvPool* p, int32_t seq, int n_tokens, const int32_t* token_ids,
                               int64_t* out_slots, int32_t* out_cow_pair, int* out_n_cow) {
  if (!p || n_tokens < 0 || (n_tokens > 0 && (!out_slots || !out_cow_pair)))
    return KV_ERR_INVALID_ARG;
  int64_t len = 0, have = 0;
  bool cow = false;
  auto it = p->seqs.find(seq);
  if (it != p->seqs.end()) {
    len = it->second.len;
    have = static_cast<int64_t>(it->second.table.size());
    if (n_tokens > 0 && len % p->B != 0 && p->ref[it->second.table[len / p->B]] > 1) cow = true;
  }
  const int64_t need = blocks_for(len + n_tokens, p->B) - have + (cow ? 1 : 0);
  if (need > available(p)) return KV_ERR_NO_FREE_BLOCK;
  const int64_t first_full = len / p->B;
  int n_cow = 0;
  for (int i = 0; i < n_tokens; ++i) {
    int32_t src, dst;
    append_one(p, p->seqs[seq], &out_slots[i], &src, &dst);
    if (src >= 0) {
      out_cow_pair[0] = src;
      out_cow_pair[1] = dst;
      n_cow = 1;
    }
  }
  if (n_tokens > 0 || p->seqs.count(seq)) {
    record_tokens(p, p->seqs[seq], token_ids, n_tokens);
    pc_publish(p, seq, first_full);
  }
  if (out_n_cow) *out_n_cow = n_cow;
  return KV_OK;
}

kvStatus seq_fork(kvPool* p, int32_t parent, int32_t child) {
  if (!p) return KV_ERR_INVALID_ARG;
  auto it = p->seqs.find(parent);
  if (it == p->seqs.end() || p->seqs.count(child)) return KV_ERR_INVALID_ARG;
  kvSeq c = it->second;  // table copy + length
  for (int32_t id : c.table) p->ref[id] += 1;
  p->seqs.emplace(child, std::move(c));
  return KV_OK;
}

kvStatus seq_release(kvPool* p, int32_t seq) {
  if (!p) return KV_ERR_INVALID_ARG;
  auto it = p->seqs.find(seq);
  if (it == p->seqs.end()) return KV_ERR_INVALID_ARG;
  for (int32_t id : it->second.table) {
    p->ref[id] -= 1;
    if (p->ref[id] == 0) count_zero(p, id);
  }
  p->seqs.erase(it);
  return KV_OK;
}

// ---------------------------------------------------------- prefix cache

kvStatus kv_prefix_cache_enable(kvPool* p, uint64_t salt) {
  if (!p) return KV_ERR_INVALID_ARG;
  if (p->pc_on) return p->pc_salt == salt ? KV_OK : KV_ERR_INVALID_ARG;
  p->pc_on = true;
  p->pc_salt = salt;
  p->pc_dormant.assign(p->N, 0);
  for (auto& kv : p->seqs) {  // positions written before: unknown tokens
    kv.second.tok.assign(kv.second.len, 0);
    kv.second.known.assign(kv.second.len, 0);
  }
  return KV_OK;
}

kvStatus seq_match_prefix(kvPool* p, int32_t seq, const int32_t* tokens, int n_tokens,
                          int* out_matched) {
  if (!p || !p->pc_on || !out_matched || n_tokens < 0 || (n_tokens > 0 && !tokens))
    return KV_ERR_INVALID_ARG;
  if (p->seqs.count(seq)) return KV_ERR_INVALID_ARG;
  const int B = p->B;
  std::vector<int32_t> blocks;
  uint64_t h = pc_root(p);
  int32_t prev = -1;
  for (int k = 0; (k + 1) * B <= n_tokens; ++k) {
    h = pc_chain(h, tokens + k * B, B);
    const int32_t c = pc_find(p, h, prev, tokens + k * B);
    if (c < 0) break;
    blocks.push_back(c);
    prev = c;
  }
  for (int32_t c : blocks) {
    if (p->pc_dormant[c]) {
      p->pc_lru.erase({p->pc_nodes.at(c).last, c});
      p->pc_dormant[c] = 0;
      p->pc_n_dormant -= 1;
    }
    p->ref[c] += 1;
    pc_tick(p, c);
  }
  kvSeq s;
  s.table = blocks;
  s.len = static_cast<int64_t>(blocks.size()) * B;
  s.tok.assign(tokens, tokens + s.len);
  s.known.assign(s.len, 1);
  p->seqs.emplace(seq, std::move(s));
  *out_matched = static_cast<int>(blocks.size()) * B;
  return KV_OK;
}

kvStatus kv_prefix_evict(kvPool* p, int target_free, int* out_n_evicted) {
  if (!p || target_free < 0) return KV_ERR_INVALID_ARG;
  int n = 0;
  while (static_cast<int64_t>(p->free_list.size()) < target_free && pc_evict_one(p)) ++n;
  if (out_n_evicted) *out_n_evicted = n;
  return KV_OK;
}

kvStatus kv_prefix_stats(const kvPool* p, int* n_cached, int* n_dormant) {
  if (!p) return KV_ERR_INVALID_ARG;
  if (n_cached) *n_cached = static_cast<int>(p->pc_nodes.size());
  if (n_dormant) *n_dormant = static_cast<int>(p->pc_n_dormant);
  return KV_OK;
}

kvStatus seq_length(const kvPool* p, int32_t seq, int* out_len) {
  if (!p || !out_len) return KV_ERR_INVALID_ARG;
  auto it = p->seqs.find(seq);
  if (it == p->seqs.end()) return KV_ERR_INVALID_ARG;
  *out_len = static_cast<int>(it->second.len);
  return KV_OK;
}

kvStatus seq_block_table(const kvPool* p, const int32_t* seq_ids, int n_seq, int max_blocks,
                         int32_t* out_table, int32_t* out_context_lens) {
  if (!p || n_seq < 0 || max_blocks < 0 || (n_seq > 0 && (!seq_ids || !out_context_lens)))
    return KV_ERR_INVALID_ARG;
  if (n_seq > 0 && max_blocks > 0 && !out_table) return KV_ERR_INVALID_ARG;
  std::vector<const kvSeq*>& seqs = t_append.cseqs;
  seqs.assign(n_seq, nullptr);
  for (int i = 0; i < n_seq; ++i) {
    auto it = p->seqs.find(seq_ids[i]);
    if (it == p->seqs.end()) return KV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(it->second.table.size()) > max_blocks) return KV_ERR_INVALID_ARG;
    if (it->second.len > INT32_MAX) return KV_ERR_INVALID_ARG;
    seqs[i] = &it->second;
  }
  for (int i = 0; i < n_seq; ++i) {
    const kvSeq& s = *seqs[i];
    int32_t* row = out_table + static_cast<int64_t>(i) * max_blocks;
    const int nb = static_cast<int>(s.table.size());
    if (nb) std::memcpy(row, s.table.data(), sizeof(int32_t) * nb);
    for (int j = nb; j < max_blocks; ++j) row[j] = -1;
    out_context_lens[i] = static_cast<int32_t>(s.len);
  }
  return KV_OK;
}

}  // extern "C"
