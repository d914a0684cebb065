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

int32_t pop_free(kvPool* p) {
  int32_t id = p->free_list.front();
  p->free_list.pop_front();
  return id;
}

void push_free(kvPool* p, int32_t id) { p->free_list.push_back(id); }

// One token for `seq` (creating it if new).  Caller has already checked
// that a free block is available whenever this needs one.
void append_one(kvPool* p, int32_t seq_id, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
  kvSeq& s = p->seqs[seq_id];
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
// counting copy-on-writes with the counts as they evolve inside the batch.
int64_t blocks_needed(const kvPool* p, const int32_t* seq_ids, int n) {
  std::unordered_map<int32_t, int32_t> drop;  // tail id -> counts dropped so far
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    auto it = p->seqs.find(seq_ids[i]);
    if (it == p->seqs.end()) {
      need += 1;
      continue;
    }
    const kvSeq& s = it->second;
    const int64_t j = s.len / p->B;
    if (j == static_cast<int64_t>(s.table.size())) {
      need += 1;
    } else {
      int32_t tail = s.table[j];
      int32_t cnt = p->ref[tail] - drop[tail];
      if (cnt > 1) {
        need += 1;
        drop[tail] += 1;
      }
    }
  }
  return need;
}

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
      (dtype != KV_DTYPE_F32 && dtype != KV_DTYPE_BF16 && dtype != KV_DTYPE_FP8_E4M3))
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
  int64_t n_alloc = 0;
  for (int i = 0; i < p->N; ++i) {
    if ((p->ref[i] > 0) == static_cast<bool>(is_free[i])) return KV_ERR_REFCOUNT;
    if (p->ref[i] < 0 || p->ext[i] < 0) return KV_ERR_REFCOUNT;
    if (p->ref[i] != table_refs[i] + p->ext[i]) return KV_ERR_REFCOUNT;
    n_alloc += p->ref[i] > 0;
  }
  if (static_cast<int64_t>(p->free_list.size()) + n_alloc != p->N) return KV_ERR_REFCOUNT;
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
  return KV_ERR_INVALID_ARG;
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
    if (p->ref[id] == 0) push_free(p, id);
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
  if (p->free_list.empty()) return KV_ERR_NO_FREE_BLOCK;
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
  if (!p || n_seq < 0 || (n_seq > 0 && (!seq_ids || !out_slots || !out_cow_pairs)))
    return KV_ERR_INVALID_ARG;
  {
    std::vector<int32_t> sorted(seq_ids, seq_ids + n_seq);
    std::sort(sorted.begin(), sorted.end());
    if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return KV_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_seq; ++i) {
    auto it = p->seqs.find(seq_ids[i]);
    if (it != p->seqs.end() && it->second.len >= (int64_t(1) << 40)) return KV_ERR_INVALID_ARG;
  }
  if (blocks_needed(p, seq_ids, n_seq) > static_cast<int64_t>(p->free_list.size()))
    return KV_ERR_NO_FREE_BLOCK;
  int n_cow = 0;
  for (int i = 0; i < n_seq; ++i) {
    int32_t src, dst;
    append_one(p, seq_ids[i], &out_slots[i], &src, &dst);
    if (src >= 0) {
      out_cow_pairs[2 * n_cow] = src;
      out_cow_pairs[2 * n_cow + 1] = dst;
      ++n_cow;
    }
  }
  if (out_n_cow) *out_n_cow = n_cow;
  return KV_OK;
}

kvStatus seq_append_tokens(kvPool* p, int32_t seq, int n_tokens, int64_t* out_slots,
                           int32_t* out_cow_pair, int* out_n_cow) {
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
  if (need > static_cast<int64_t>(p->free_list.size())) return KV_ERR_NO_FREE_BLOCK;
  int n_cow = 0;
  for (int i = 0; i < n_tokens; ++i) {
    int32_t src, dst;
    append_one(p, seq, &out_slots[i], &src, &dst);
    if (src >= 0) {
      out_cow_pair[0] = src;
      out_cow_pair[1] = dst;
      n_cow = 1;
    }
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
    if (p->ref[id] == 0) push_free(p, id);
  }
  p->seqs.erase(it);
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
  for (int i = 0; i < n_seq; ++i) {
    auto it = p->seqs.find(seq_ids[i]);
    if (it == p->seqs.end()) return KV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(it->second.table.size()) > max_blocks) return KV_ERR_INVALID_ARG;
    if (it->second.len > INT32_MAX) return KV_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_seq; ++i) {
    const kvSeq& s = p->seqs.find(seq_ids[i])->second;
    int32_t* row = out_table + static_cast<int64_t>(i) * max_blocks;
    const int nb = static_cast<int>(s.table.size());
    if (nb) std::memcpy(row, s.table.data(), sizeof(int32_t) * nb);
    for (int j = nb; j < max_blocks; ++j) row[j] = -1;
    out_context_lens[i] = static_cast<int32_t>(s.len);
  }
  return KV_OK;
}

}  // extern "C"
