// Internal pool state shared by the host block manager and the device
// entry points.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <deque>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct kvSeq {
  std::vector<int32_t> table;  // logical block -> physical block
  int64_t len = 0;             // tokens with K/V present
};

struct kvPool {
  // shape
  int L = 0, N = 0, B = 0, H = 0, D = 0, dtype = 0, esize = 0;
  // caller-owned device memory
  void* k = nullptr;
  void* v = nullptr;
  int32_t* d_status = nullptr;

  // host control plane
  std::deque<int32_t> free_list;  // FIFO: pop front, push back
  std::vector<int32_t> ref;       // table entries + handles per block
  std::vector<int32_t> ext;       // caller-held handles per block
  std::unordered_map<int32_t, kvSeq> seqs;

  // device-side cache, filled by the first device call
  bool dev_ready = false;
  int device = -1;
  int sm_count = 0;
  int grid_by_g[4] = {0, 0, 0, 0};  // split-pass CTAs per log2(H_q / H_kv)
  alignas(64) unsigned char tmap[4][128];  // TMA descriptors: K, V plain; K, V swizzled
  bool mma_ok = false;                      // swizzled descriptors valid (bf16, B % 8 == 0)
  int decode_path = 0;                      // KV_OPT_DECODE_PATH
  bool pdl = true;                          // programmatic dependent launch

  // host staging reused by kv_decode_step_host
  std::vector<int64_t> h_slots;
  std::vector<int32_t> h_pairs, h_table, h_lens;
  std::vector<unsigned char> h_plan;
};

// Largest CTA count the split pass uses; sizes the decode workspace.
constexpr int kMaxDecodeCtas = 1024;

// Workspace bytes of a planned decode pass (plan.cpp).
size_t plan_workspace_bytes(int n_segs, int c_max, int D);
