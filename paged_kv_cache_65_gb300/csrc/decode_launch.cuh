// Launch helper for one instantiation of the split pass.
#pragma once

#include "decode.cuh"
#include "decode_mma.cuh"
#include "launch.cuh"

namespace pkv {

// Launches decode_split_kernel<ESIZE, D, G>.  On the first call for a pool
// (*grid_io <= 0) it raises the kernel's dynamic shared-memory limit and sizes
// the persistent grid as (resident CTAs per SM) x (SM count), capped at
// max_grid; later calls reuse *grid_io.
template <int ESIZE, int D, int G>
cudaError_t launch_split(const CUtensorMap& tk, const CUtensorMap& tv, DecodeArgs a, int sm_count,
                         int max_grid, int* grid_io, cudaStream_t st, bool pdl) {
  constexpr int smem = decode_smem_bytes<ESIZE, D, G>();
  auto kern = decode_split_kernel<ESIZE, D, G>;
  if (*grid_io <= 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    int g = occ * sm_count;
    *grid_io = g > max_grid ? max_grid : g;
  }
  a.grid = *grid_io;
  return launch_kernel(pdl, kern, dim3(a.grid), dim3(kThreads), smem, st, tk, tv, a);
}

template <int D, int G, bool F8 = false, bool Q8 = false>
cudaError_t launch_mma(const CUtensorMap& tk, const CUtensorMap& tv, DecodeArgs a, int sm_count,
                       int max_grid, int* grid_io, cudaStream_t st, bool pdl) {
  constexpr int smem = decode_mma_smem_bytes<D, G, F8, Q8>();
  auto k_plain = decode_mma_kernel<D, G, false, F8, Q8>;
  auto k_plan = decode_mma_kernel<D, G, true, F8, Q8>;
  // the dynamic shared-memory limit is a per-function, per-device attribute
  static bool attr_set[2][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int v = a.segs ? 1 : 0;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[v][dev]) {
    e = cudaFuncSetAttribute(v ? k_plan : k_plain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    attr_set[v][dev] = true;
  }
  if (*grid_io <= 0) {
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, v ? k_plan : k_plain, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    int g = occ * sm_count;
    *grid_io = g > max_grid ? max_grid : g;
  }
  a.grid = *grid_io;
  return launch_kernel(pdl, v ? k_plan : k_plain, dim3(a.grid), dim3(kThreads), smem, st, tk, tv,
                       a);
}

struct PrefillArgs;
// tcgen05 chunked-prefill attention: one CTA per (sequence, K/V head, 128
// query rows); in the natural grid sized by max_chunk, or one per work item
// of a.sched (n_items of them) and K/V head.
cudaError_t launch_prefill_tc(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a,
                              int max_chunk, int n_items, cudaStream_t st, bool pdl);

// tcgen05 variant (bfloat16, D_h = 128, the swizzled TMA maps); one CTA per SM.
cudaError_t launch_tc_bf16(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                           int sm_count, int max_grid, int* grid_io, cudaStream_t st, bool pdl);

// The same over an FP8 (E4M3) pool (the code tensor maps: one 128-code box
// per row set).
cudaError_t launch_tc_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                          int sm_count, int max_grid, int* grid_io, cudaStream_t st, bool pdl);

// Tensor-core variant for bfloat16 (swizzled TMA maps, B a multiple of 8).
cudaError_t launch_mma_bf16(int D, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeArgs& a, int sm_count, int max_grid, int* grid_io,
                            cudaStream_t st, bool pdl, bool* supported);

// The same pass over an FP8 (E4M3) pool, D_h = 128.
cudaError_t launch_mma_fp8(int D, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                           const DecodeArgs& a, int sm_count, int max_grid, int* grid_io,
                           cudaStream_t st, bool pdl, bool* supported);

// The same pass over a q8_0 pool (int8 codes, fp16 scales per 32 values,
// a.k_sc / a.v_sc), D_h = 128.
cudaError_t launch_mma_q8(int D, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeArgs& a, int sm_count, int max_grid, int* grid_io,
                          cudaStream_t st, bool pdl, bool* supported);

// Dispatch over (D, G) for one element size; *supported = false when the
// shape has no compiled instantiation.
cudaError_t launch_split_e2(int D, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeArgs& a, int sm_count, int max_grid, int* grid_io,
                            cudaStream_t st, bool pdl, bool* supported);
cudaError_t launch_split_e4(int D, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeArgs& a, int sm_count, int max_grid, int* grid_io,
                            cudaStream_t st, bool pdl, bool* supported);

}  // namespace pkv
