// Instantiations and launch of the tcgen05 split pass over FP8 (E4M3) K/V
// (D_h = 128): codes converted to fp16 in shared memory, f16 MMAs.
#include "decode_launch.cuh"
#include "decode_tc.cuh"

namespace pkv {

cudaError_t launch_tc_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                          int sm_count, int max_grid, int* grid_io, cudaStream_t st, bool pdl) {
  return launch_tc<true>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
}

}  // namespace pkv
