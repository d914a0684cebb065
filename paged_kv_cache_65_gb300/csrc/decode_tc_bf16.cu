// Instantiations and launch of the tcgen05 split pass (bfloat16, D_h = 128).
#include "decode_launch.cuh"
#include "decode_tc.cuh"

namespace pkv {

cudaError_t launch_tc_bf16(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a_in,
                           int sm_count, int max_grid, int* grid_io, cudaStream_t st, bool pdl) {
  constexpr int smem = decode_tc_smem_bytes();
  auto k_plain = decode_tc_kernel<false>;
  auto k_plan = decode_tc_kernel<true>;
  static bool attr_set[2][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int v = a_in.segs ? 1 : 0;
  if (!attr_set[v][dev]) {
    e = cudaFuncSetAttribute(v ? k_plan : k_plain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    attr_set[v][dev] = true;
  }
  if (*grid_io <= 0) *grid_io = sm_count < max_grid ? sm_count : max_grid;
  DecodeArgs a = a_in;
  a.grid = *grid_io;
  return launch_kernel(pdl, v ? k_plan : k_plain, dim3(a.grid), dim3(kTcThreads), smem, st, tk,
                       tv, a);
}

}  // namespace pkv
