// Instantiations and launch of the tcgen05 split pass (bfloat16, D_h = 128).
#include "decode_launch.cuh"
#include "decode_tc.cuh"

namespace pkv {

cudaError_t launch_tc_bf16(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                           int sm_count, int max_grid, int* grid_io, cudaStream_t st, bool pdl) {
  return launch_tc<false>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
}

}  // namespace pkv
