// Launch of the tcgen05 chunked-prefill attention (bfloat16, D_h = 128).
#include "launch.cuh"
#include "prefill_tc.cuh"

namespace pkv {

cudaError_t launch_prefill_tc(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a,
                              int max_chunk, int n_items, cudaStream_t st, bool pdl) {
  constexpr int smem = prefill_tc_smem_bytes();
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int G = a.n_q_heads / a.n_kv_heads;
  const int T = 128 / G;
  // natural grid: (tiles of the longest chunk, K/V heads, sequences); with a
  // work order, one CTA per (item, K/V head), heads fastest
  const dim3 grid = a.sched ? dim3(n_items * a.n_kv_heads)
                            : dim3((max_chunk + T - 1) / T, a.n_kv_heads, a.n_seq);
  return launch_kernel(pdl, prefill_tc_kernel, grid, dim3(kPfThreads), smem, st, tk, tv, a);
}

}  // namespace pkv
