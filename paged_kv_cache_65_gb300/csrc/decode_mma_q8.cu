// Instantiations of the warp-level MMA split pass over q8_0 K/V (int8 codes,
// one fp16 scale per 32 values).
#include "decode_launch.cuh"

namespace pkv {

cudaError_t launch_mma_q8(int D, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeArgs& a, int sm_count, int max_grid, int* grid_io,
                          cudaStream_t st, bool pdl, bool* supported) {
  *supported = true;
  if (D == 128) {
    switch (G) {
      case 1: return launch_mma<128, 1, true, true>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
      case 2: return launch_mma<128, 2, true, true>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
      case 4: return launch_mma<128, 4, true, true>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
      case 8: return launch_mma<128, 8, true, true>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
      default: break;
    }
  }
  *supported = false;
  return cudaSuccess;
}

}  // namespace pkv
