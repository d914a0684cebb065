// Internal pool state shared by the host block manager and the device
// entry points.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <deque>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/pagedkv.h"

struct kvSeq {
  std::vector<int32_t> table;  // logical block -> physical block
  int64_t len = 0;             // tokens with K/V present
  // prefix cache on: the token id of every position (known[i] = 0: unknown)
  std::vector<int32_t> tok;
  std::vector<uint8_t> known;
};

// A cached full block of the prefix cache: its identity is the whole token
// prefix up to its end, held as (parent node, this block's tokens); `hash`
// chains the salt and every block's tokens for the lookup.
struct kvPrefixNode {
  uint64_t hash = 0;
  int32_t parent = -1;    // cached block of the previous B tokens (-1: root)
  int32_t children = 0;   // cached blocks whose parent this is
  uint64_t last = 0;      // logical access clock
  std::vector<int32_t> tokens;
};

struct kvPool {
  // shape
  int L = 0, N = 0, B = 0, H = 0, D = 0, dtype = 0, esize = 0;
  int in_esize = 0;                 // bytes of a q / new K/V element (bf16 for FP8 pools)
  void* k_sc = nullptr;             // Q8_0: fp16 scales [L][N][H][B][D / 32] of K and V
  void* v_sc = nullptr;
  float k_scale = 1.f, v_scale = 1.f;  // FP8 pools: stored code = e4m3(x / scale)
  // caller-owned device memory
  void* k = nullptr;
  void* v = nullptr;
  int32_t* d_status = nullptr;

  // host control plane
  std::deque<int32_t> free_list;  // FIFO: pop front, push back
  std::vector<int32_t> ref;       // table entries + handles per block
  std::vector<int32_t> ext;       // caller-held handles per block
  std::unordered_map<int32_t, kvSeq> seqs;

  // prefix cache (off until kv_prefix_cache_enable)
  bool pc_on = false;
  uint64_t pc_salt = 0, pc_clock = 0;
  std::unordered_map<int32_t, kvPrefixNode> pc_nodes;    // cached block -> node
  std::unordered_multimap<uint64_t, int32_t> pc_index;   // chain hash -> cached blocks
  std::set<std::pair<uint64_t, int32_t>> pc_lru;         // dormant leaves by last access
  std::vector<uint8_t> pc_dormant;                       // cached block with count 0
  int64_t pc_n_dormant = 0;

  // device-side cache, filled by the first device call
  bool dev_ready = false;
  int device = -1;
  int sm_count = 0;
  int grid_by_g[4] = {0, 0, 0, 0};  // split-pass CTAs per log2(H_q / H_kv)
  int grid_tc = 0;                  // CTAs of the tcgen05 split pass (one per SM)
  int merge_deep_ctas = -1;         // planned-merge CTAs resident at once, deep prefetch
  int plan_grid = 0;                // KV_OPT_PLAN_GRID: CTA count plans build start records for
  alignas(64) unsigned char tmap[4][128];  // TMA descriptors: K, V plain; K, V swizzled
  // staged prefill of an FP8 pool: swizzled TMA descriptors of the bfloat16
  // copies of K and V in the caller's workspace, valid for (stage_base,
  // stage_rows)
  alignas(64) unsigned char tmap_stage[2][128];
  const void* stage_base = nullptr;
  long long stage_rows = -1;
  bool mma_ok = false;                      // swizzled descriptors valid (bf16, B % 8 == 0)
  int decode_path = 0;                      // KV_OPT_DECODE_PATH
  bool pdl = true;                          // programmatic dependent launch

  // host staging of kv_decode_step_host: the step's metadata (slots, copy
  // pairs, tables, lengths, plan) in page-locked memory, laid out as in the
  // device staging buffer so that one copy moves it
  unsigned char* h_pinned = nullptr;
  size_t h_pinned_bytes = 0;
  // kv_decode_step_host of a pool with several layers: a second stream and
  // two events per layer, made on first use, so that each layer's q copy and
  // output copy overlap the other layers' kernels (cudaStream_t / cudaEvent_t)
  void* side_stream = nullptr;
  std::vector<void*> step_events;  // [2 * L]: layer l's q landed; layer l's output written

  ~kvPool();
};

// Tensor-core passes read K/V through 128-byte-swizzled TMA boxes of 64
// elements by min(B, T) rows, T = 64 tokens at D_h = 128 and 128 at 64: each
// box starts on 1 KiB (B a multiple of 8) and a stage holds whole blocks or a
// block whole stages.
// Pools of one-byte codes (FP8 E4M3, q8_0).
inline bool pool_codes8(const kvPool* p) {
  return p->dtype == KV_DTYPE_FP8_E4M3 || p->dtype == KV_DTYPE_Q8_0;
}

inline bool pool_tensor_core_shape(const kvPool* p) {
  if (pool_codes8(p)) {
    // FP8 / q8_0: rows of 128 one-byte codes, one 128-byte swizzled box per row set
    if (p->D != 128 || p->B % 8 != 0) return false;
  } else if (p->dtype != KV_DTYPE_BF16 || (p->D != 64 && p->D != 128) || p->B % 8 != 0) {
    return false;
  }
  const int t = p->D == 64 ? 128 : 64;
  return p->B <= t ? t % p->B == 0 : p->B % t == 0;
}

// The tcgen05 pass: the tensor-core shape with D_h = 128.
inline bool pool_tc_shape(const kvPool* p) {
  return p->dtype == KV_DTYPE_BF16 && pool_tensor_core_shape(p) && p->D == 128;
}

// The tcgen05 decode pass: bfloat16 as above, or FP8 codes with D_h = 128
// (converted to fp16 in the pass: K rows into tensor memory, V rows into
// shared memory).
inline bool pool_tc_decode_shape(const kvPool* p) {
  return (p->dtype == KV_DTYPE_BF16 || p->dtype == KV_DTYPE_FP8_E4M3) &&
         pool_tensor_core_shape(p) && p->D == 128;
}

// Largest CTA count the split pass uses; sizes the decode workspace.
constexpr int kMaxDecodeCtas = 1024;

// SM count of the pool's device, 0 while unknown (device.cu).
int pool_sm_count(const kvPool* p);

// Workspace bytes of a planned decode pass (plan.cpp).
size_t plan_workspace_bytes(int n_segs, int c_max, int D);

// paged_decode_plan with the per-CTA start records optional (plan.cpp): a
// plan without them is valid for any grid (each CTA then finds its first
// piece itself).
kvStatus plan_build(const kvPool* p, const int32_t* seq_ids, int n_seq, int n_q_heads,
                    int max_blocks, int min_shared_tokens, void* h_plan, size_t plan_bytes,
                    size_t* out_workspace_bytes, bool start_records);
