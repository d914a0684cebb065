// Arguments of the chunked-prefill attention kernel (prefill_tc.cuh).
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace pkv {

struct PrefillArgs {
  const void* q;               // [n_tok][H_q][D] bf16
  const int32_t* table;        // [n_seq][max_blocks]
  const int32_t* chunk_start;  // [n_seq + 1] query-row offsets
  const int32_t* ctx;          // [n_seq] context lengths (history + chunk)
  float* out_f32;              // [n_tok][H_q][D], or
  __nv_bfloat16* out_bf16;
  int32_t* status;
  // heaviest-first work order, or null for the natural grid: item i is
  // (sequence, tile, the chunk length the order was built for, blocks);
  // CTA x works on item x / H_kv, K/V head x % H_kv
  const int4* sched;
  int n_seq, max_blocks, layer, n_blocks, block_size, n_kv_heads, n_q_heads;
  float qscale;  // scale * log2(e) (times the K scale of an FP8 pool's codes)
  float vscale;  // factor of the outputs: 1, or the V scale of an FP8 pool's codes
};

}  // namespace pkv
