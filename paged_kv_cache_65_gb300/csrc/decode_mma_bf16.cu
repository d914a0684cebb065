// Instantiations of the tensor-core split pass (bfloat16 K/V).
#include "decode_launch.cuh"

namespace pkv {

cudaError_t launch_mma_bf16(int D, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeArgs& a, int sm_count, int max_grid, int* grid_io,
                            cudaStream_t st, bool pdl, bool* supported) {
  *supported = true;
  switch (D * 16 + G) {
    case 64 * 16 + 1: return launch_mma<64, 1>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
    case 64 * 16 + 2: return launch_mma<64, 2>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
    case 64 * 16 + 4: return launch_mma<64, 4>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
    case 64 * 16 + 8: return launch_mma<64, 8>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
    case 128 * 16 + 1: return launch_mma<128, 1>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
    case 128 * 16 + 2: return launch_mma<128, 2>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
    case 128 * 16 + 4: return launch_mma<128, 4>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
    case 128 * 16 + 8: return launch_mma<128, 8>(tk, tv, a, sm_count, max_grid, grid_io, st, pdl);
    default: break;
  }
  *supported = false;
  return cudaSuccess;
}

}  // namespace pkv
