// Decode attention for callers that cannot allocate device memory.
//
// paged_decode_attention() takes its split-K workspace from the caller.  Some
// callers have no way to provide one: serving loops whose device memory is
// entirely pre-reserved by another allocator, or plain C hosts that want no
// allocator at all.  For them this file keeps the
// workspace in a fixed-size array in the library's own static device memory
// and passes its address to the same kernels.
//
// The array exists once per GPU that loads the library and stays allocated
// until the process exits.  Every call on that GPU shares it: two calls that
// overlap on the GPU (different streams without ordering between them) race
// on it.  Nothing in the workspace needs to start at zero: every entry the
// merge reads is written by the split pass of the same call.
#include <cuda_runtime.h>

#include "pool.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per GPU
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of the array on the current device.  The host-side symbol
// is only a stand-in, so the address comes from cudaGetSymbolAddress, with
// that device current, on every call: the call allocates nothing and
// enqueues no work, and an address kept from an earlier call could be stale
// after the device's context was reset.
kvStatus scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KV_ERR_UNSUPPORTED;
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess || !p) return KV_ERR_CUDA;
  *out = p;
  return KV_OK;
}

}  // namespace

extern "C" kvStatus paged_decode_attention_noalloc(kvPool* pool, int layer, const void* d_q,
                                                   int n_q_heads, const int32_t* d_block_table,
                                                   int max_blocks, const int32_t* d_context_lens,
                                                   int n_seq, float scale, void* d_out,
                                                   int out_dtype, void* stream) {
  if (!pool || n_seq < 0 || n_q_heads <= 0) return KV_ERR_INVALID_ARG;
  const size_t need = paged_decode_workspace_bytes(pool, n_seq, n_q_heads);
  if (need == 0) return KV_ERR_INVALID_ARG;
  if (need > kScratchBytes) return KV_ERR_SCRATCH_TOO_SMALL;
  void* ws = nullptr;
  const kvStatus s = scratch_address(&ws);
  if (s != KV_OK) return s;
  return paged_decode_attention(pool, layer, d_q, n_q_heads, d_block_table, max_blocks,
                                d_context_lens, n_seq, scale, d_out, out_dtype, ws, kScratchBytes,
                                stream);
}
