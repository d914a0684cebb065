// Device entry points of the C ABI: TMA descriptors, slot write
// (reshape_and_cache), copy-on-write block copy, the merge pass of split-K
// decode attention, and the whole-step driver over host buffers.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "decode_launch.cuh"
#include "prefill.h"
#include "launch.cuh"
#include "plan.h"
#include "pool.h"
#include "ptx.cuh"

using pkv::record_status;

namespace {

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int ilog2_small(int g) { return g == 1 ? 0 : g == 2 ? 1 : g == 4 ? 2 : g == 8 ? 3 : -1; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2-D TMA descriptor over n_rows rows of `cols` elements (of esize bytes,
// type dt), box inner x rows.
kvStatus encode_rows_map(const void* base, unsigned long long n_rows, unsigned long long cols,
                         int esize, CUtensorMapDataType dt, int inner, int rows, bool swizzle128,
                         CUtensorMap* out) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return KV_ERR_CUDA;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(n_rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * esize};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(inner), static_cast<cuuint32_t>(rows)};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = fn(out, dt, 2, const_cast<void*>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KV_OK : KV_ERR_CUDA;
}

// A 2-D view of one cache: inner dimension H_kv * D_h elements (one token
// row of every head), outer dimension N_layers * N_blocks * B rows; a box is
// `inner` elements of one head by `rows` token rows.
kvStatus encode_cache_map(kvPool* p, void* base, int inner, int rows, bool swizzle128,
                          CUtensorMap* out) {
  const CUtensorMapDataType dt = p->dtype == KV_DTYPE_BF16     ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : p->dtype == KV_DTYPE_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                               : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return encode_rows_map(base, static_cast<unsigned long long>(p->L) * p->N * p->B,
                         static_cast<unsigned long long>(p->H) * p->D, p->esize, dt, inner, rows,
                         swizzle128, out);
}

// Split-pass kernel for a pool (after ensure_device) and its decode-path
// option: CUDA cores, warp-level MMA (mma.sync), or tcgen05 with TMEM
// accumulators (bfloat16 or FP8, D_h = 128).
enum DecodeKernel { kKernelCudaCores, kKernelMma, kKernelTc };

DecodeKernel decode_kernel(const kvPool* p) {
  const bool mma = p->mma_ok;
  const bool tc = p->mma_ok && pool_tc_decode_shape(p);
  switch (p->decode_path) {
    case 1: return kKernelCudaCores;
    case 2: return mma ? kKernelMma : kKernelCudaCores;
    case 3: return tc ? kKernelTc : (mma ? kKernelMma : kKernelCudaCores);
    default: return mma ? kKernelMma : kKernelCudaCores;
  }
}

// First device use of a pool: device, SM count, TMA descriptors.
kvStatus ensure_device(kvPool* p) {
  if (p->dev_ready) return KV_OK;
  if (!p->k || !p->v) return KV_ERR_INVALID_ARG;
  if (cudaGetDevice(&p->device) != cudaSuccess) return KV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) !=
      cudaSuccess)
    return KV_ERR_CUDA;
  if (p->dtype == KV_DTYPE_Q8_0 && (!p->k_sc || !p->v_sc))
    return KV_ERR_INVALID_ARG;  // a q8_0 pool needs its scale arrays
  if (pool_codes8(p)) {
    // FP8 / q8_0 codes: the tensor-core passes (q8_0: the warp-level one),
    // one 128-byte swizzled box (128 codes, all of D_h = 128) by
    // mma_box_rows(B, 128) rows
    if (!pool_tensor_core_shape(p)) return KV_ERR_UNSUPPORTED;
    const int rm = pkv::mma_box_rows(p->B, pkv::mma_stage_tokens(p->D, true));
    kvStatus s = encode_cache_map(p, p->k, 128, rm, true, reinterpret_cast<CUtensorMap*>(p->tmap[2]));
    if (s != KV_OK) return s;
    s = encode_cache_map(p, p->v, 128, rm, true, reinterpret_cast<CUtensorMap*>(p->tmap[3]));
    if (s != KV_OK) return s;
    p->mma_ok = true;
  } else if (p->D == 64 || p->D == 128) {
    const int ts = pkv::stage_tokens(p->esize, p->D);
    if (p->B > ts && p->B % ts != 0) return KV_ERR_UNSUPPORTED;
    const int rows = p->B < ts ? p->B : ts;
    kvStatus s = encode_cache_map(p, p->k, p->D, rows, false,
                                  reinterpret_cast<CUtensorMap*>(p->tmap[0]));
    if (s != KV_OK) return s;
    s = encode_cache_map(p, p->v, p->D, rows, false, reinterpret_cast<CUtensorMap*>(p->tmap[1]));
    if (s != KV_OK) return s;
    // tensor-core passes: rows of 64 bf16 (128 bytes) with the 128-byte swizzle
    if (pool_tensor_core_shape(p)) {
      const int rm = pkv::mma_box_rows(p->B, pkv::mma_stage_tokens(p->D));
      s = encode_cache_map(p, p->k, 64, rm, true, reinterpret_cast<CUtensorMap*>(p->tmap[2]));
      if (s != KV_OK) return s;
      s = encode_cache_map(p, p->v, 64, rm, true, reinterpret_cast<CUtensorMap*>(p->tmap[3]));
      if (s != KV_OK) return s;
      p->mma_ok = true;
    }
  }
  p->dev_ready = true;
  return KV_OK;
}

// ------------------------------------------------------------- kernels

// Two E4M3 codes (low byte first) as two bfloat16 values, exactly (every
// E4M3 value has at most four significant bits and an exponent inside
// bfloat16's range); NaN codes stay NaN.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two)));
  const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
  const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Staged chunked prefill of an FP8 pool: the codes of every block a listed
// sequence reads (its first ceil(ctx / B) table entries, layer `layer`)
// become their exact bfloat16 values in the workspace, logical block j of
// sequence i at copy block i * max_blocks + j, whose table entry the kernel
// writes too; slots past the context are written as zeros.  The scales stay
// out (the attention applies them).  One CTA per (logical block, sequence).
__global__ void __launch_bounds__(128) prefill_stage_fp8_kernel(
    const uint4* __restrict__ k_pool, const uint4* __restrict__ v_pool,
    const int32_t* __restrict__ table, const int32_t* __restrict__ ctx, int max_blocks,
    int layer, int n_blocks, int B, int row_vecs, uint4* __restrict__ k_stage,
    uint4* __restrict__ v_stage, int32_t* __restrict__ stage_table, int32_t* status) {
  const int j = blockIdx.x, i = blockIdx.y;
  const long long sb = static_cast<long long>(i) * max_blocks + j;
  if (threadIdx.x == 0) stage_table[sb] = static_cast<int32_t>(sb);
  pkv::griddep_wait();  // the pool's newest rows come from the kernels before
  pkv::griddep_launch_dependents();
  const int len = ctx[i];
  if (len <= 0 || j >= (len + B - 1) / B) return;
  const int pid = table[sb];
  const bool ok = pid >= 0 && pid < n_blocks;
  if (!ok && threadIdx.x == 0) record_status(status, KV_DEV_BAD_BLOCK_ID);
  const int rows = len - j * B < B ? len - j * B : B;  // slots inside the context
  // row_vecs: 16-code vectors per token row (H_kv * D_h / 16)
  const long long src = (static_cast<long long>(layer) * n_blocks + (ok ? pid : 0)) * B * row_vecs;
  const long long dst = sb * B * row_vecs * 2;
  for (int idx = threadIdx.x; idx < B * row_vecs; idx += blockDim.x) {
    const bool live = ok && idx / row_vecs < rows;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
      if (live) {
        const uint4 c = (kv ? v_pool : k_pool)[src + idx];
        o0 = make_uint4(e4m3x2_to_bf16x2(c.x), e4m3x2_to_bf16x2(c.x >> 16),
                        e4m3x2_to_bf16x2(c.y), e4m3x2_to_bf16x2(c.y >> 16));
        o1 = make_uint4(e4m3x2_to_bf16x2(c.z), e4m3x2_to_bf16x2(c.z >> 16),
                        e4m3x2_to_bf16x2(c.w), e4m3x2_to_bf16x2(c.w >> 16));
      }
      uint4* out = kv ? v_stage : k_stage;
      out[dst + 2 * idx] = o0;
      out[dst + 2 * idx + 1] = o1;
    }
  }
}

// Slot write: one CTA per (token, layer); 16-byte copies of the token's row
// [H_kv][D_h] into K_cache[layer][slot / B][slot % B] and the same for V.
__global__ void slot_write_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                  const int64_t* __restrict__ slots, int n_tok, uint4* kc,
                                  uint4* vc, int layer, long long slots_per_layer, int row_vecs,
                                  int32_t* status) {
  pkv::griddep_wait();
  pkv::griddep_launch_dependents();
  const int i = blockIdx.x;
  const int ly = layer >= 0 ? layer : blockIdx.y;
  const int64_t slot = slots[i];
  if (slot < 0) return;
  if (slot >= slots_per_layer) {
    if (threadIdx.x == 0) record_status(status, KV_DEV_BAD_SLOT);
    return;
  }
  const long long src = ((layer >= 0 ? 0LL : (long long)blockIdx.y * n_tok) + i) * row_vecs;
  const long long dst = ((long long)ly * slots_per_layer + slot) * row_vecs;
  for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
    kc[dst + v] = k_new[src + v];
    vc[dst + v] = v_new[src + v];
  }
}

// Slot write into an FP8 pool: one CTA per (token, layer); each thread turns
// 8 bfloat16 values of the token's K (and V) row into 8 E4M3 codes of
// x / scale: float32 IEEE division, then the nearest code, ties to even,
// saturating at 448 ("第 8 章 推理优化" §8.4.2's narrower KV, in the
// format of the pool's header description).
__global__ void slot_write_fp8_kernel(const uint4* __restrict__ k_new,
                                      const uint4* __restrict__ v_new,
                                      const int64_t* __restrict__ slots, int n_tok, uint2* kc,
                                      uint2* vc, int layer, long long slots_per_layer,
                                      int row_vecs, float k_scale, float v_scale,
                                      int32_t* status) {
  pkv::griddep_wait();
  pkv::griddep_launch_dependents();
  const int i = blockIdx.x;
  const int ly = layer >= 0 ? layer : blockIdx.y;
  const int64_t slot = slots[i];
  if (slot < 0) return;
  if (slot >= slots_per_layer) {
    if (threadIdx.x == 0) record_status(status, KV_DEV_BAD_SLOT);
    return;
  }
  // row_vecs: 8-element groups per token row (H_kv * D_h / 8)
  const long long src = ((layer >= 0 ? 0LL : (long long)blockIdx.y * n_tok) + i) * row_vecs;
  const long long dst = ((long long)ly * slots_per_layer + slot) * row_vecs;
  auto quant8 = [](uint4 x, float scale) -> uint2 {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t out[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t b = 0;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t word = w[2 * h + k];
        const float lo = __fdiv_rn(__uint_as_float(word << 16), scale);
        const float hi = __fdiv_rn(__uint_as_float(word & 0xffff0000u), scale);
        uint16_t c;
        // the first source goes to the upper byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
        b |= static_cast<uint32_t>(c) << (16 * k);
      }
      out[h] = b;
    }
    return make_uint2(out[0], out[1]);
  };
  for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
    kc[dst + v] = quant8(k_new[src + v], k_scale);
    vc[dst + v] = quant8(v_new[src + v], v_scale);
  }
}

// Copy-on-write copy: CTA (pair, layer, part) copies a slice of block src
// into block dst in K and V.  Each thread loads up to four 16-byte vectors of
// K and four of V before storing any, so the loads of cold source blocks are
// in flight together instead of one latency per vector.
// Slot write into a q8_0 pool: one CTA per (token, layer); each thread takes
// one group of 32 bfloat16 values of the token's K (and V) row: amax =
// max |x|, d = the fp16 nearest to amax / 127 (float32 IEEE division), codes
// = the integers nearest to x / d (float32 IEEE division, ties to even)
// clamped to [-127, 127], all zero when d is 0 ("第 8 章 推理优化" §8.4.2's
// q8_0 groups).  Codes go to the row's slot, the scale to
// scales[layer][block][head][slot][group].
__global__ void slot_write_q8_kernel(const uint4* __restrict__ k_new,
                                     const uint4* __restrict__ v_new,
                                     const int64_t* __restrict__ slots, int n_tok, uint4* kc,
                                     uint4* vc, __half* ksc, __half* vsc, int layer,
                                     int n_blocks, int B, int H, int groups_per_head,
                                     int32_t* status) {
  pkv::griddep_wait();
  pkv::griddep_launch_dependents();
  const int i = blockIdx.x;
  const int ly = layer >= 0 ? layer : blockIdx.y;
  const int64_t slot = slots[i];
  if (slot < 0) return;
  const long long slots_per_layer = static_cast<long long>(n_blocks) * B;
  if (slot >= slots_per_layer) {
    if (threadIdx.x == 0) record_status(status, KV_DEV_BAD_SLOT);
    return;
  }
  const int n_groups = H * groups_per_head;  // groups of 32 in a token row
  const long long src = ((layer >= 0 ? 0LL : (long long)blockIdx.y * n_tok) + i) * n_groups * 4;
  const long long dst = ((long long)ly * slots_per_layer + slot) * n_groups * 2;
  const long long blk = slot / B;
  const int o = static_cast<int>(slot - blk * B);
  for (int g = threadIdx.x; g < 2 * n_groups; g += blockDim.x) {
    const bool is_k = g < n_groups;
    const int gg = is_k ? g : g - n_groups;
    const uint4* in = (is_k ? k_new : v_new) + src + gg * 4;
    float x[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 w = in[v];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[v * 8 + 2 * k] = __uint_as_float(ws[k] << 16);
        x[v * 8 + 2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(x[k]));
    const __half d16 = __float2half_rn(__fdiv_rn(amax, 127.f));
    const float d = __half2float(d16);
    uint32_t packed[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t w = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float q = d > 0.f ? rintf(__fdiv_rn(x[4 * k + b], d)) : 0.f;
        q = fminf(fmaxf(q, -127.f), 127.f);
        w |= (static_cast<uint32_t>(static_cast<int>(q)) & 0xffu) << (8 * b);
      }
      packed[k] = w;
    }
    uint4* out = (is_k ? kc : vc) + dst + gg * 2;
    out[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    out[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    const int h = gg / groups_per_head, q = gg - h * groups_per_head;
    (is_k ? ksc : vsc)[(((long long)ly * n_blocks + blk) * H + h) * B * groups_per_head +
                       static_cast<long long>(o) * groups_per_head + q] = d16;
  }
}

__global__ void cow_copy_kernel(const int32_t* __restrict__ pairs, uint4* kc, uint4* vc,
                                int n_blocks, long long block_vecs, int32_t* status) {
  pkv::griddep_wait();
  pkv::griddep_launch_dependents();
  const int i = blockIdx.x;
  const int ly = blockIdx.y;
  const int src = pairs[2 * i], dst = pairs[2 * i + 1];
  if (src < 0 || src >= n_blocks || dst < 0 || dst >= n_blocks) {
    if (threadIdx.x == 0 && ly == 0 && blockIdx.z == 0) record_status(status, KV_DEV_BAD_COW_PAIR);
    return;
  }
  if (src == dst) return;
  const long long s0 = ((long long)ly * n_blocks + src) * block_vecs;
  const long long d0 = ((long long)ly * n_blocks + dst) * block_vecs;
  const long long per = (block_vecs + gridDim.z - 1) / gridDim.z;
  const long long b = (long long)blockIdx.z * per;
  const long long e = b + per < block_vecs ? b + per : block_vecs;
  constexpr int U = 4;
  for (long long v0 = b + threadIdx.x; v0 < e; v0 += (long long)U * blockDim.x) {
    uint4 kx[U], vx[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long v = v0 + (long long)u * blockDim.x;
      if (v < e) {
        kx[u] = kc[s0 + v];
        vx[u] = vc[s0 + v];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long v = v0 + (long long)u * blockDim.x;
      if (v < e) {
        kc[d0 + v] = kx[u];
        vc[d0 + v] = vx[u];
      }
    }
  }
}

// Self-test of the bounded pipeline waits: one thread waits on an mbarrier
// that nothing completes, with the same helper every pipeline wait uses; the
// wait gives up after limit_ns and the status word gets KV_DEV_WAIT_TIMEOUT.
// Nothing else is in flight, so the CTA then just exits.
__global__ void wait_selftest_kernel(int32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    pkv::mbar_init(&bar, 1);
    pkv::fence_barrier_init();
    if (!pkv::mbar_wait_bounded(&bar, 0, limit_ns)) record_status(status, KV_DEV_WAIT_TIMEOUT);
  }
}

// Merge pass: per (sequence, query head) combine the partials of every piece
// of its segment: M = max m_i, L = sum l_i 2^(m_i - M),
// out = sum O_i 2^(m_i - M) / L.  One warp per (sequence, query head), four
// heads per CTA; the max over pieces is a shuffle reduction.
template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const long long* __restrict__ pre,
                                                    const float* __restrict__ ws_ml,
                                                    const float* __restrict__ ws_o, int n_seq,
                                                    int H, int Hq, int grid, float* out_f32,
                                                    __nv_bfloat16* out_bf16) {
  pkv::griddep_wait();
  pkv::griddep_launch_dependents();
  constexpr int DL = D / 32;
  const int s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = Hq / H;
  // blocks of this sequence, as the split pass counted them
  const int nb = static_cast<int>((pre[s + 1] - pre[s]) / H);
  const long long W = pre[n_seq];
  long long chunk = (W + grid - 1) / grid;
  if (chunk == 0) chunk = 1;
  {
    const int hq = blockIdx.y * 4 + warp;
    if (hq >= Hq) return;
    float o[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) o[d] = 0.f;
    if (nb > 0) {
      const int h = hq / G, g = hq - h * G;
      const long long a0 = pre[s] + (long long)h * nb;
      const long long c0 = a0 / chunk, c1 = (a0 + nb - 1) / chunk;
      const long long seg = (long long)s * H + h;
      const int np = static_cast<int>(c1 - c0 + 1);
      float M = -INFINITY;
      for (int i = lane; i < np; i += 32) M = fmaxf(M, ws_ml[((c0 + i + seg) * G + g) * 2]);
#pragma unroll
      for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      float L = 0.f;
      for (int i = 0; i < np; ++i) {
        const long long slot = (c0 + i + seg) * G + g;
        const float f = pkv::exp2_approx(ws_ml[slot * 2] - M);
        L += f * ws_ml[slot * 2 + 1];
        const float* src = ws_o + slot * D + lane * DL;
        if constexpr (DL == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          o[0] += f * v.x;
          o[1] += f * v.y;
          o[2] += f * v.z;
          o[3] += f * v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          o[0] += f * v.x;
          o[1] += f * v.y;
        }
      }
      const float inv = 1.f / L;
#pragma unroll
      for (int d = 0; d < DL; ++d) o[d] *= inv;
    }
    const long long ob = ((long long)s * Hq + hq) * D + lane * DL;
    if (out_f32) {
#pragma unroll
      for (int d = 0; d < DL; ++d) out_f32[ob + d] = o[d];
    } else {
#pragma unroll
      for (int d = 0; d < DL; ++d) out_bf16[ob + d] = __float2bfloat16_rn(o[d]);
    }
  }
}

// Merge pass of a planned decode: per (sequence, query head) combine the
// partials of every piece of every segment its merge entries name (shared
// prefix and private rest), with the same rule as merge_kernel.  The plan
// (written by the host before the stream's kernel chain started) is read
// before waiting for the split pass; then lanes load the pieces' (m, l) side
// by side, once, and the O rows of the first PRE pieces go out with them
// (the rest four pieces at a time), instead of a chain of dependent loads per
// piece.  The sums run in piece order either way.
// Four warps per CTA.  PRE pieces' O rows are loaded ahead: 12 covers the
// rows of a batch sharing a long prefix (about ten pieces each) at 96
// registers a thread, five CTAs an SM; 8 keeps 80 registers, six CTAs an SM.
// The host takes the deeper one only while the whole grid is resident at once
// (a 48-sequence, 64-query-head batch has 768 CTAs: one wave at 8, two at 12).
constexpr int kMergePlanWarps = 4;

template <int D, int PRE>
__global__ void __launch_bounds__(kMergePlanWarps * 32) merge_plan_kernel(
    const PlanSeg* __restrict__ segs, const int32_t* __restrict__ eoff,
    const PlanEntry* __restrict__ ents, long long W, int grid, int c_max,
    const float* __restrict__ ws_ml, const float* __restrict__ ws_o, int H, int Hq,
    float* out_f32, __nv_bfloat16* out_bf16) {
  constexpr int DL = D / 32;
  const int s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.y * kMergePlanWarps + warp;
  const bool live = hq < Hq;
  const int G = Hq / H;
  const int h = live ? hq / G : 0, g = live ? hq - h * G : 0;
  long long chunk = (W + grid - 1) / grid;
  if (chunk == 0) chunk = 1;
  const int e0 = live ? eoff[s * H + h] : 0, e1 = live ? eoff[s * H + h + 1] : 0;
  // workspace slot of the k-th piece over the entries, or -1 past the last
  auto piece_slot = [&](int k) -> int {
    for (int e = e0; e < e1; ++e) {
      const PlanEntry en = ents[e];
      const PlanSeg sg = segs[en.seg];
      const long long units = static_cast<long long>(sg.b1 - sg.b0) * (sg.w > 0 ? sg.w : 1);
      const long long c0 = sg.wpre / chunk, c1 = (sg.wpre + units - 1) / chunk;
      const int n = static_cast<int>(c1 - c0 + 1);
      if (k < n) return static_cast<int>((c0 + k + en.seg) * c_max + en.col_base + g);
      k -= n;
    }
    return -1;
  };
  int np = 0;
  for (int e = e0; e < e1; ++e) {
    const PlanSeg sg = segs[ents[e].seg];
    const long long units = static_cast<long long>(sg.b1 - sg.b0) * (sg.w > 0 ? sg.w : 1);
    np += static_cast<int>((sg.wpre + units - 1) / chunk - sg.wpre / chunk + 1);
  }
  const int slot0 = lane < np ? piece_slot(lane) : -1;
  pkv::griddep_wait();
  pkv::griddep_launch_dependents();
  if (!live) return;
  // (m, l) of the first 32 pieces in one 8-byte load per lane, kept for the
  // weights below
  float2 ml0 = make_float2(-INFINITY, 0.f);
  if (lane < np) ml0 = *reinterpret_cast<const float2*>(&ws_ml[static_cast<long long>(slot0) * 2]);
  // the O rows of the first kPre pieces go out with their (m, l), not after
  // the weights: one dependent latency less after the wait
  constexpr int kPre = PRE;
  float pre[kPre][DL];
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const int sj = __shfl_sync(0xffffffffu, slot0, j);
    if (j < np) {
      const float* src = ws_o + static_cast<long long>(sj) * D + lane * DL;
      if constexpr (DL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        pre[j][0] = v.x;
        pre[j][1] = v.y;
        pre[j][2] = v.z;
        pre[j][3] = v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        pre[j][0] = v.x;
        pre[j][1] = v.y;
      }
    }
  }
  float M = ml0.x;
  for (int k = lane + 32; k < np; k += 32)
    M = fmaxf(M, ws_ml[static_cast<long long>(piece_slot(k)) * 2]);
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float o[DL];
#pragma unroll
  for (int d = 0; d < DL; ++d) o[d] = 0.f;
  float L = 0.f;
  for (int r = 0; r < np; r += 32) {
    // lane k: weight of piece r + k (0 for a CTA whose range held no block
    // start of the segment: m = -inf, O = 0)
    const int k = r + lane;
    int sl = 0;
    float f = 0.f;
    if (k < np) {
      sl = r == 0 ? slot0 : piece_slot(k);
      const float2 mlk =
          r == 0 ? ml0 : *reinterpret_cast<const float2*>(&ws_ml[static_cast<long long>(sl) * 2]);
      f = mlk.x == -INFINITY ? 0.f : pkv::exp2_approx(mlk.x - M);
      L += f * mlk.y;
    }
    const int nr = np - r < 32 ? np - r : 32;
    int j0 = 0;
    if (r == 0) {
#pragma unroll
      for (int j = 0; j < kPre; ++j) {
        const float fj = __shfl_sync(0xffffffffu, f, j);
        if (j < nr) {
#pragma unroll
          for (int d = 0; d < DL; ++d) o[d] += fj * pre[j][d];
        }
      }
      j0 = kPre;
    }
#pragma unroll 4
    for (int j = j0; j < nr; ++j) {
      const float fj = __shfl_sync(0xffffffffu, f, j);
      const int sj = __shfl_sync(0xffffffffu, sl, j);
      const float* src = ws_o + static_cast<long long>(sj) * D + lane * DL;
      if constexpr (DL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        o[0] += fj * v.x;
        o[1] += fj * v.y;
        o[2] += fj * v.z;
        o[3] += fj * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        o[0] += fj * v.x;
        o[1] += fj * v.y;
      }
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const long long ob = ((long long)s * Hq + hq) * D + lane * DL;
  if constexpr (DL == 4) {
    if (out_f32 && (reinterpret_cast<uintptr_t>(out_f32) & 15u) == 0u) {
      // one 16-byte store per lane (the output may be page-locked host
      // memory written in place, which whole vectors cross in fewer writes)
      *reinterpret_cast<float4*>(out_f32 + ob) =
          make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
      return;
    }
  }
#pragma unroll
  for (int d = 0; d < DL; ++d) {
    if (out_f32)
      out_f32[ob + d] = o[d] * inv;
    else
      out_bf16[ob + d] = __float2bfloat16_rn(o[d] * inv);
  }
}

struct WsLayout {
  size_t pre, ml, o, total;
};

WsLayout ws_layout(const kvPool* p, int n_seq, int G) {
  const size_t n_slots = static_cast<size_t>(kMaxDecodeCtas) + static_cast<size_t>(n_seq) * p->H;
  WsLayout w;
  w.pre = 0;
  w.ml = align256(sizeof(long long) * (static_cast<size_t>(n_seq) + 1));
  w.o = w.ml + align256(n_slots * G * 2 * sizeof(float));
  w.total = w.o + n_slots * G * p->D * sizeof(float);
  return w;
}

bool aligned16(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; }

// Checks and launch shared by the natural-grid and the scheduled prefill.
// Staged prefill of an FP8 pool: the bfloat16 copy the attention reads
// instead of the pool (its TMA descriptors, its table, its block count).
struct PrefillStage {
  const CUtensorMap* tk;
  const CUtensorMap* tv;
  const int32_t* table;
  int n_blocks;
};

// Whether a pool can run the chunked-prefill pass: bfloat16 in place, or
// FP8 (D_h = 128, the tensor-core block shapes) through a bfloat16 copy.
bool prefill_shape(const kvPool* p, bool staged) {
  return staged ? p->dtype == KV_DTYPE_FP8_E4M3 && p->D == 128 && pool_tensor_core_shape(p)
                : pool_tc_shape(p);
}

kvStatus prefill_common(kvPool* p, int layer, const void* d_q, int n_q_heads,
                        const int32_t* d_block_table, int max_blocks,
                        const int32_t* d_chunk_start, const int32_t* d_context_lens, int n_seq,
                        int max_chunk, const int4* sched, int n_items, float scale, void* d_out,
                        int out_dtype, void* stream, const PrefillStage* stage = nullptr) {
  if (!p || !p->k || n_seq < 0 || n_q_heads <= 0 || n_q_heads % p->H != 0)
    return KV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= p->L) return KV_ERR_INVALID_ARG;
  if (out_dtype != KV_DTYPE_F32 && out_dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  const int G = n_q_heads / p->H;
  if (ilog2_small(G) < 0 || !prefill_shape(p, stage != nullptr)) return KV_ERR_UNSUPPORTED;
  if (n_seq == 0 || (sched ? n_items == 0 : max_chunk == 0)) return KV_OK;
  if (!d_q || !d_block_table || !d_chunk_start || !d_context_lens || !d_out || max_blocks <= 0)
    return KV_ERR_INVALID_ARG;
  if (!aligned16(d_q) || !aligned16(d_out)) return KV_ERR_INVALID_ARG;
  if (n_seq > 65535 || static_cast<long long>(max_blocks) * p->B >= (1LL << 31))
    return KV_ERR_INVALID_ARG;
  if (sched && static_cast<long long>(n_items) * p->H > 0x7fffffffLL) return KV_ERR_INVALID_ARG;
  kvStatus s = ensure_device(p);
  if (s != KV_OK) return s;
  if (!p->mma_ok) return KV_ERR_UNSUPPORTED;
  pkv::PrefillArgs a;
  a.q = d_q;
  a.table = stage ? stage->table : d_block_table;
  a.chunk_start = d_chunk_start;
  a.ctx = d_context_lens;
  a.out_f32 = out_dtype == KV_DTYPE_F32 ? static_cast<float*>(d_out) : nullptr;
  a.out_bf16 = out_dtype == KV_DTYPE_BF16 ? static_cast<__nv_bfloat16*>(d_out) : nullptr;
  a.status = p->d_status;
  a.sched = sched;
  a.n_seq = n_seq;
  a.max_blocks = max_blocks;
  a.layer = stage ? 0 : layer;
  a.n_blocks = stage ? stage->n_blocks : p->N;
  a.block_size = p->B;
  a.n_kv_heads = p->H;
  a.n_q_heads = n_q_heads;
  if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(p->D));
  // an FP8 copy holds the codes' values: K's scale joins the score scale,
  // V's scales the outputs
  a.qscale = scale * 1.4426950408889634f * (stage ? p->k_scale : 1.f);  // log2(e)
  a.vscale = stage ? p->v_scale : 1.f;
  const CUtensorMap& tk = stage ? *stage->tk : *reinterpret_cast<const CUtensorMap*>(p->tmap[2]);
  const CUtensorMap& tv = stage ? *stage->tv : *reinterpret_cast<const CUtensorMap*>(p->tmap[3]);
  const cudaError_t e =
      pkv::launch_prefill_tc(tk, tv, a, max_chunk, n_items, as_stream(stream), p->pdl);
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kvStatus check_decode_args(const kvPool* p, int layer, const void* q, int n_q_heads,
                           const int32_t* table, int max_blocks, const int32_t* ctx, int n_seq,
                           const void* ws, size_t ws_bytes) {
  if (!p || !p->k) return KV_ERR_INVALID_ARG;
  if (n_seq < 0 || n_q_heads <= 0 || n_q_heads % p->H != 0) return KV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= p->L) return KV_ERR_INVALID_ARG;
  const int G = n_q_heads / p->H;
  if (ilog2_small(G) < 0 || (p->D != 64 && p->D != 128)) return KV_ERR_UNSUPPORTED;
  if (n_seq == 0) return KV_OK;
  if (!q || !table || !ctx || !ws || max_blocks <= 0) return KV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(p, n_seq, G).total) return KV_ERR_INVALID_ARG;
  if (static_cast<long long>(max_blocks) * p->B >= (1LL << 31)) return KV_ERR_INVALID_ARG;
  return KV_OK;
}

}  // namespace

kvPool::~kvPool() {
  if (h_pinned) cudaFreeHost(h_pinned);
  for (void* e : step_events)
    if (e) cudaEventDestroy(static_cast<cudaEvent_t>(e));
  if (side_stream) cudaStreamDestroy(static_cast<cudaStream_t>(side_stream));
}

// SM count of the device a pool with device memory runs on (the current
// device until its first kernel has run); 0 for a host-only pool or without
// a device.
int pool_sm_count(const kvPool* p) {
  if (p->sm_count > 0) return p->sm_count;
  if (!p->k) return 0;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

extern "C" {

kvStatus kv_pool_device_status(kvPool* p, void* stream, int* out_bits) {
  if (!p || !out_bits) return KV_ERR_INVALID_ARG;
  *out_bits = 0;
  if (!p->d_status) return KV_OK;
  cudaStream_t st = as_stream(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KV_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, p->d_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KV_ERR_CUDA;
  if (v && cudaMemset(p->d_status, 0, sizeof(int32_t)) != cudaSuccess) return KV_ERR_CUDA;
  *out_bits = v;
  return v ? KV_ERR_DEVICE_CHECK : KV_OK;
}

kvStatus kv_device_wait_selftest(kvPool* p, int limit_us, void* stream) {
  if (!p || limit_us < 1 || limit_us > 1000000) return KV_ERR_INVALID_ARG;
  kvStatus s = ensure_device(p);
  if (s != KV_OK) return s;
  const cudaError_t e =
      pkv::launch_kernel(false, wait_selftest_kernel, dim3(1), dim3(32), 0, as_stream(stream),
                         p->d_status, static_cast<unsigned long long>(limit_us) * 1000ull);
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kvStatus cow_copy(kvPool* p, const int32_t* d_pairs, int n_pairs, void* stream) {
  if (!p || n_pairs < 0 || (n_pairs > 0 && !d_pairs)) return KV_ERR_INVALID_ARG;
  if (n_pairs == 0) return KV_OK;
  kvStatus s = ensure_device(p);
  if (s != KV_OK) return s;
  const long long block_vecs = static_cast<long long>(p->B) * p->H * p->D * p->esize / 16;
  // about 512 vectors of K (and of V) per CTA: two per thread
  const long long want = (block_vecs + 511) / 512;
  const int parts = static_cast<int>(want < 1 ? 1 : (want > 16 ? 16 : want));
  dim3 grid(n_pairs, p->L, parts);
  cudaError_t e = pkv::launch_kernel(
      p->pdl, cow_copy_kernel, grid, dim3(256), 0, as_stream(stream), d_pairs,
      reinterpret_cast<uint4*>(p->k), reinterpret_cast<uint4*>(p->v), p->N, block_vecs,
      p->d_status);
  if (e == cudaSuccess && p->dtype == KV_DTYPE_Q8_0) {
    // the blocks' scales ([L][N][H][B][D / 32] fp16) go with their codes
    const long long sc_vecs = static_cast<long long>(p->H) * p->B * (p->D / 32) * 2 / 16;
    e = pkv::launch_kernel(p->pdl, cow_copy_kernel, dim3(n_pairs, p->L, 1), dim3(256), 0,
                           as_stream(stream), d_pairs, reinterpret_cast<uint4*>(p->k_sc),
                           reinterpret_cast<uint4*>(p->v_sc), p->N, sc_vecs, p->d_status);
  }
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kvStatus reshape_and_cache(kvPool* p, int layer, const void* d_k_new, const void* d_v_new,
                           const int64_t* d_slot_mapping, int n_tokens, void* stream) {
  if (!p || n_tokens < 0 || layer < -1 || layer >= p->L) return KV_ERR_INVALID_ARG;
  if (n_tokens == 0) return KV_OK;
  if (!d_k_new || !d_v_new || !d_slot_mapping) return KV_ERR_INVALID_ARG;
  if (!aligned16(d_k_new) || !aligned16(d_v_new)) return KV_ERR_INVALID_ARG;
  kvStatus s = ensure_device(p);
  if (s != KV_OK) return s;
  if (p->dtype == KV_DTYPE_Q8_0) {
    const int groups = p->H * p->D / 32;
    dim3 grid(n_tokens, layer >= 0 ? 1 : p->L);
    const int threads = 2 * groups >= 128 ? 128 : (2 * groups >= 64 ? 64 : 32);
    const cudaError_t e = pkv::launch_kernel(
        p->pdl, slot_write_q8_kernel, grid, dim3(threads), 0, as_stream(stream),
        reinterpret_cast<const uint4*>(d_k_new), reinterpret_cast<const uint4*>(d_v_new),
        d_slot_mapping, n_tokens, reinterpret_cast<uint4*>(p->k), reinterpret_cast<uint4*>(p->v),
        reinterpret_cast<__half*>(p->k_sc), reinterpret_cast<__half*>(p->v_sc), layer, p->N,
        p->B, p->H, p->D / 32, p->d_status);
    return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
  }
  if (p->dtype == KV_DTYPE_FP8_E4M3) {
    const int row_vecs = p->H * p->D / 8;
    dim3 grid(n_tokens, layer >= 0 ? 1 : p->L);
    const int threads = row_vecs >= 128 ? 128 : (row_vecs >= 64 ? 64 : 32);
    const cudaError_t e = pkv::launch_kernel(
        p->pdl, slot_write_fp8_kernel, grid, dim3(threads), 0, as_stream(stream),
        reinterpret_cast<const uint4*>(d_k_new), reinterpret_cast<const uint4*>(d_v_new),
        d_slot_mapping, n_tokens, reinterpret_cast<uint2*>(p->k), reinterpret_cast<uint2*>(p->v),
        layer, static_cast<long long>(p->N) * p->B, row_vecs, p->k_scale, p->v_scale,
        p->d_status);
    return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
  }
  const int row_vecs = p->H * p->D * p->esize / 16;
  dim3 grid(n_tokens, layer >= 0 ? 1 : p->L);
  const int threads = row_vecs >= 128 ? 128 : (row_vecs >= 64 ? 64 : 32);
  const cudaError_t e = pkv::launch_kernel(
      p->pdl, slot_write_kernel, grid, dim3(threads), 0, as_stream(stream),
      reinterpret_cast<const uint4*>(d_k_new), reinterpret_cast<const uint4*>(d_v_new),
      d_slot_mapping, n_tokens, reinterpret_cast<uint4*>(p->k), reinterpret_cast<uint4*>(p->v),
      layer, static_cast<long long>(p->N) * p->B, row_vecs, p->d_status);
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

size_t paged_decode_workspace_bytes(const kvPool* p, int n_seq, int n_q_heads) {
  if (!p || n_seq < 0 || n_q_heads <= 0 || n_q_heads % p->H != 0) return 0;
  return ws_layout(p, n_seq, n_q_heads / p->H).total;
}

kvStatus paged_decode_partials(kvPool* p, int layer, const void* d_q, int n_q_heads,
                               const int32_t* d_block_table, int max_blocks,
                               const int32_t* d_context_lens, int n_seq, float scale,
                               void* d_workspace, size_t workspace_bytes, void* stream) {
  kvStatus s = check_decode_args(p, layer, d_q, n_q_heads, d_block_table, max_blocks,
                                 d_context_lens, n_seq, d_workspace, workspace_bytes);
  if (s != KV_OK || n_seq == 0) return s;
  s = ensure_device(p);
  if (s != KV_OK) return s;
  const int G = n_q_heads / p->H;
  const WsLayout w = ws_layout(p, n_seq, G);
  unsigned char* ws = reinterpret_cast<unsigned char*>(d_workspace);
  pkv::DecodeArgs a;
  a.q = d_q;
  a.table = d_block_table;
  a.ctx = d_context_lens;
  a.ws_pre = reinterpret_cast<long long*>(ws + w.pre);
  a.ws_ml = reinterpret_cast<float*>(ws + w.ml);
  a.ws_o = reinterpret_cast<float*>(ws + w.o);
  a.status = p->d_status;
  a.n_seq = n_seq;
  a.max_blocks = max_blocks;
  a.layer = layer;
  a.n_blocks = p->N;
  a.block_size = p->B;
  a.n_kv_heads = p->H;
  a.n_q_heads = n_q_heads;
  if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(p->D));
  a.qscale = scale * 1.4426950408889634f;  // log2(e)
  a.vscale = 1.f;
  if (p->dtype == KV_DTYPE_FP8_E4M3) {  // codes carry x / scale
    a.qscale *= p->k_scale;
    a.vscale = p->v_scale;
  }
  a.grid = 0;
  a.segs = nullptr;
  a.members = nullptr;
  a.n_segs = 0;
  a.c_max = G;
  a.plan_W = 0;
  a.starts = nullptr;
  a.start_grid = 0;
  const DecodeKernel kern = decode_kernel(p);
  int* grid_io = kern == kKernelTc ? &p->grid_tc : &p->grid_by_g[ilog2_small(G)];
  bool supported = false;
  cudaError_t e;
  if (p->dtype == KV_DTYPE_FP8_E4M3 && kern == kKernelTc) {
    const CUtensorMap& tk = *reinterpret_cast<const CUtensorMap*>(p->tmap[2]);
    const CUtensorMap& tv = *reinterpret_cast<const CUtensorMap*>(p->tmap[3]);
    e = pkv::launch_tc_fp8(tk, tv, a, p->sm_count, kMaxDecodeCtas, grid_io, as_stream(stream),
                           p->pdl);
    supported = true;
  } else if (pool_codes8(p)) {
    if (kern != kKernelMma) return KV_ERR_UNSUPPORTED;  // no CUDA-core pass over codes
    const CUtensorMap& tk = *reinterpret_cast<const CUtensorMap*>(p->tmap[2]);
    const CUtensorMap& tv = *reinterpret_cast<const CUtensorMap*>(p->tmap[3]);
    a.k_sc = p->k_sc;
    a.v_sc = p->v_sc;
    e = p->dtype == KV_DTYPE_Q8_0
            ? pkv::launch_mma_q8(p->D, G, tk, tv, a, p->sm_count, kMaxDecodeCtas, grid_io,
                                 as_stream(stream), p->pdl, &supported)
            : pkv::launch_mma_fp8(p->D, G, tk, tv, a, p->sm_count, kMaxDecodeCtas, grid_io,
                                  as_stream(stream), p->pdl, &supported);
  } else if (kern == kKernelTc) {
    const CUtensorMap& tk = *reinterpret_cast<const CUtensorMap*>(p->tmap[2]);
    const CUtensorMap& tv = *reinterpret_cast<const CUtensorMap*>(p->tmap[3]);
    e = pkv::launch_tc_bf16(tk, tv, a, p->sm_count, kMaxDecodeCtas, grid_io, as_stream(stream),
                            p->pdl);
    supported = true;
  } else if (kern == kKernelMma) {
    const CUtensorMap& tk = *reinterpret_cast<const CUtensorMap*>(p->tmap[2]);
    const CUtensorMap& tv = *reinterpret_cast<const CUtensorMap*>(p->tmap[3]);
    e = pkv::launch_mma_bf16(p->D, G, tk, tv, a, p->sm_count, kMaxDecodeCtas, grid_io,
                             as_stream(stream), p->pdl, &supported);
  } else {
    const CUtensorMap& tk = *reinterpret_cast<const CUtensorMap*>(p->tmap[0]);
    const CUtensorMap& tv = *reinterpret_cast<const CUtensorMap*>(p->tmap[1]);
    e = p->esize == 2 ? pkv::launch_split_e2(p->D, G, tk, tv, a, p->sm_count, kMaxDecodeCtas,
                                             grid_io, as_stream(stream), p->pdl, &supported)
                      : pkv::launch_split_e4(p->D, G, tk, tv, a, p->sm_count, kMaxDecodeCtas,
                                             grid_io, as_stream(stream), p->pdl, &supported);
  }
  if (!supported) return KV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kvStatus paged_decode_merge(kvPool* p, int n_q_heads, const int32_t* d_context_lens, int n_seq,
                            void* d_out, int out_dtype, const void* d_workspace,
                            size_t workspace_bytes, void* stream) {
  if (!p || n_seq < 0 || n_q_heads <= 0 || n_q_heads % p->H != 0) return KV_ERR_INVALID_ARG;
  if (out_dtype != KV_DTYPE_F32 && out_dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  const int G = n_q_heads / p->H;
  if (ilog2_small(G) < 0 || (p->D != 64 && p->D != 128)) return KV_ERR_UNSUPPORTED;
  if (n_seq == 0) return KV_OK;
  if (!d_context_lens || !d_out || !d_workspace) return KV_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(p, n_seq, G);
  if (workspace_bytes < w.total || !aligned16(d_workspace)) return KV_ERR_INVALID_ARG;
  // the CTA count of the split pass that wrote the partials
  const int grid = p->dev_ready && decode_kernel(p) == kKernelTc ? p->grid_tc
                                                                 : p->grid_by_g[ilog2_small(G)];
  if (grid <= 0) return KV_ERR_INVALID_ARG;  // no split pass has run on this pool
  const unsigned char* ws = reinterpret_cast<const unsigned char*>(d_workspace);
  const long long* pre = reinterpret_cast<const long long*>(ws + w.pre);
  const float* ml = reinterpret_cast<const float*>(ws + w.ml);
  const float* o = reinterpret_cast<const float*>(ws + w.o);
  float* of = out_dtype == KV_DTYPE_F32 ? reinterpret_cast<float*>(d_out) : nullptr;
  __nv_bfloat16* ob = out_dtype == KV_DTYPE_BF16 ? reinterpret_cast<__nv_bfloat16*>(d_out) : nullptr;
  const dim3 mg(n_seq, (n_q_heads + 3) / 4);
  const cudaError_t e =
      p->D == 128 ? pkv::launch_kernel(p->pdl, merge_kernel<128>, mg, dim3(128), 0,
                                       as_stream(stream), pre, ml, o, n_seq, p->H, n_q_heads,
                                       grid, of, ob)
                  : pkv::launch_kernel(p->pdl, merge_kernel<64>, mg, dim3(128), 0,
                                       as_stream(stream), pre, ml, o, n_seq, p->H, n_q_heads,
                                       grid, of, ob);
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kvStatus paged_decode_attention(kvPool* p, int layer, const void* d_q, int n_q_heads,
                                const int32_t* d_block_table, int max_blocks,
                                const int32_t* d_context_lens, int n_seq, float scale,
                                void* d_out, int out_dtype, void* d_workspace,
                                size_t workspace_bytes, void* stream) {
  if (out_dtype != KV_DTYPE_F32 && out_dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (n_seq > 0 && !d_out) return KV_ERR_INVALID_ARG;
  kvStatus s = paged_decode_partials(p, layer, d_q, n_q_heads, d_block_table, max_blocks,
                                     d_context_lens, n_seq, scale, d_workspace, workspace_bytes,
                                     stream);
  if (s != KV_OK || n_seq == 0) return s;
  return paged_decode_merge(p, n_q_heads, d_context_lens, n_seq, d_out, out_dtype, d_workspace,
                            workspace_bytes, stream);
}

namespace {
// Header of a host plan, checked against the pool and the call.
kvStatus read_plan_header(const kvPool* p, int n_q_heads, const void* h_plan, PlanHeader* hd) {
  if (!p || !p->k || !h_plan) return KV_ERR_INVALID_ARG;
  if (n_q_heads <= 0 || n_q_heads % p->H != 0) return KV_ERR_INVALID_ARG;
  std::memcpy(hd, h_plan, sizeof(*hd));
  const int G = n_q_heads / p->H;
  if (hd->n_kv_heads != p->H || hd->group != G || hd->block_size != p->B || hd->n_seq < 0 ||
      hd->c_max < G || hd->c_max > kPlanMaxCols || hd->n_segs < 0 ||
      (hd->kernel != kPlanKernelMma && hd->kernel != kPlanKernelTc))
    return KV_ERR_INVALID_ARG;
  return KV_OK;
}

size_t plan_ml_bytes(const PlanHeader& hd) {
  const size_t n_slots = static_cast<size_t>(kMaxDecodeCtas) + hd.n_segs;
  return (n_slots * hd.c_max * 2 * sizeof(float) + 255) & ~size_t(255);
}
}  // namespace

namespace {
// The planned split pass; with d_k_new / d_v_new, the step's slot write of
// this layer is fused in (each listed sequence's newest token).
kvStatus partials_planned(kvPool* p, int layer, const void* d_q, int n_q_heads,
                          const int32_t* d_block_table, int max_blocks, const void* d_plan,
                          const void* h_plan, float scale, void* d_workspace,
                          size_t workspace_bytes, void* stream, const void* d_k_new,
                          const void* d_v_new) {
  PlanHeader hd;
  kvStatus s = read_plan_header(p, n_q_heads, h_plan, &hd);
  if (s != KV_OK) return s;
  if (layer < 0 || layer >= p->L) return KV_ERR_INVALID_ARG;
  if (hd.n_seq == 0 || hd.W == 0) return KV_OK;
  if (!d_plan || !d_q || !d_block_table || !d_workspace || max_blocks <= 0)
    return KV_ERR_INVALID_ARG;
  if (!aligned16(d_q) || !aligned16(d_workspace) || !aligned16(d_plan)) return KV_ERR_INVALID_ARG;
  if (workspace_bytes < plan_workspace_bytes(hd.n_segs, hd.c_max, p->D)) return KV_ERR_INVALID_ARG;
  s = ensure_device(p);
  if (s != KV_OK) return s;
  const int G = n_q_heads / p->H;
  // the kernel the plan's work units were weighted for; the CUDA-core
  // option turns the planned pass off
  if (decode_kernel(p) == kKernelCudaCores || ilog2_small(G) < 0) return KV_ERR_UNSUPPORTED;
  const bool tc = hd.kernel == kPlanKernelTc;
  if (tc && !pool_tc_decode_shape(p)) return KV_ERR_UNSUPPORTED;
  const unsigned char* dp = reinterpret_cast<const unsigned char*>(d_plan);
  unsigned char* ws = reinterpret_cast<unsigned char*>(d_workspace);
  pkv::DecodeArgs a;
  a.q = d_q;
  a.table = d_block_table;
  a.ctx = nullptr;
  a.ws_pre = nullptr;
  a.ws_ml = reinterpret_cast<float*>(ws);
  a.ws_o = reinterpret_cast<float*>(ws + plan_ml_bytes(hd));
  a.status = p->d_status;
  a.n_seq = hd.n_seq;
  a.max_blocks = max_blocks;
  a.layer = layer;
  a.n_blocks = p->N;
  a.block_size = p->B;
  a.n_kv_heads = p->H;
  a.n_q_heads = n_q_heads;
  if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(p->D));
  a.qscale = scale * 1.4426950408889634f;  // log2(e)
  a.vscale = 1.f;
  if (p->dtype == KV_DTYPE_FP8_E4M3) {  // codes carry x / scale
    a.qscale *= p->k_scale;
    a.vscale = p->v_scale;
  }
  a.grid = 0;
  a.segs = reinterpret_cast<const PlanSeg*>(dp + hd.seg_off);
  a.members = reinterpret_cast<const int32_t*>(dp + hd.mem_off);
  a.n_segs = hd.n_segs;
  a.c_max = hd.c_max;
  a.plan_W = hd.W;
  a.starts = hd.start_grid > 0 ? reinterpret_cast<const PlanStart*>(dp + hd.start_off) : nullptr;
  a.start_grid = hd.start_grid;
  a.k_new = d_k_new;
  a.v_new = d_v_new;
  a.k_pool = p->k;
  a.v_pool = p->v;
  a.k_scale_w = p->k_scale;
  a.v_scale_w = p->v_scale;
  a.k_sc = p->k_sc;
  a.v_sc = p->v_sc;
  const CUtensorMap& tk = *reinterpret_cast<const CUtensorMap*>(p->tmap[2]);
  const CUtensorMap& tv = *reinterpret_cast<const CUtensorMap*>(p->tmap[3]);
  bool supported = true;
  const cudaError_t e =
      tc ? (p->dtype == KV_DTYPE_FP8_E4M3
                ? pkv::launch_tc_fp8(tk, tv, a, p->sm_count, kMaxDecodeCtas, &p->grid_tc,
                                     as_stream(stream), p->pdl)
                : pkv::launch_tc_bf16(tk, tv, a, p->sm_count, kMaxDecodeCtas, &p->grid_tc,
                                      as_stream(stream), p->pdl))
      : p->dtype == KV_DTYPE_Q8_0
          ? pkv::launch_mma_q8(p->D, G, tk, tv, a, p->sm_count, kMaxDecodeCtas,
                               &p->grid_by_g[ilog2_small(G)], as_stream(stream), p->pdl,
                               &supported)
      : p->dtype == KV_DTYPE_FP8_E4M3
          ? pkv::launch_mma_fp8(p->D, G, tk, tv, a, p->sm_count, kMaxDecodeCtas,
                                &p->grid_by_g[ilog2_small(G)], as_stream(stream), p->pdl,
                                &supported)
          : pkv::launch_mma_bf16(p->D, G, tk, tv, a, p->sm_count, kMaxDecodeCtas,
                                 &p->grid_by_g[ilog2_small(G)], as_stream(stream), p->pdl,
                                 &supported);
  if (!supported) return KV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}
}  // namespace

kvStatus paged_decode_partials_planned(kvPool* p, int layer, const void* d_q, int n_q_heads,
                                       const int32_t* d_block_table, int max_blocks,
                                       const void* d_plan, const void* h_plan, float scale,
                                       void* d_workspace, size_t workspace_bytes, void* stream) {
  return partials_planned(p, layer, d_q, n_q_heads, d_block_table, max_blocks, d_plan, h_plan,
                          scale, d_workspace, workspace_bytes, stream, nullptr, nullptr);
}

kvStatus paged_decode_partials_planned_write(kvPool* p, int layer, const void* d_q, int n_q_heads,
                                             const void* d_k_new, const void* d_v_new,
                                             const int32_t* d_block_table, int max_blocks,
                                             const void* d_plan, const void* h_plan, float scale,
                                             void* d_workspace, size_t workspace_bytes,
                                             void* stream) {
  if (!p || !d_k_new || !d_v_new || !aligned16(d_k_new) || !aligned16(d_v_new))
    return KV_ERR_INVALID_ARG;
  if (p->dtype != KV_DTYPE_BF16 && p->dtype != KV_DTYPE_FP8_E4M3) return KV_ERR_UNSUPPORTED;
  return partials_planned(p, layer, d_q, n_q_heads, d_block_table, max_blocks, d_plan, h_plan,
                          scale, d_workspace, workspace_bytes, stream, d_k_new, d_v_new);
}

kvStatus paged_decode_merge_planned(kvPool* p, int n_q_heads, const void* d_plan,
                                    const void* h_plan, void* d_out, int out_dtype,
                                    const void* d_workspace, size_t workspace_bytes,
                                    void* stream) {
  PlanHeader hd;
  kvStatus s = read_plan_header(p, n_q_heads, h_plan, &hd);
  if (s != KV_OK) return s;
  if (out_dtype != KV_DTYPE_F32 && out_dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (hd.n_seq == 0) return KV_OK;
  if (!d_plan || !d_out || !d_workspace) return KV_ERR_INVALID_ARG;
  if (workspace_bytes < plan_workspace_bytes(hd.n_segs, hd.c_max, p->D)) return KV_ERR_INVALID_ARG;
  const int G = n_q_heads / p->H;
  if (ilog2_small(G) < 0 || (p->D != 64 && p->D != 128)) return KV_ERR_UNSUPPORTED;
  const int grid = hd.kernel == kPlanKernelTc ? p->grid_tc : p->grid_by_g[ilog2_small(G)];
  if (hd.W > 0 && grid <= 0) return KV_ERR_INVALID_ARG;  // no split pass has run on this pool
  const unsigned char* dp = reinterpret_cast<const unsigned char*>(d_plan);
  const unsigned char* ws = reinterpret_cast<const unsigned char*>(d_workspace);
  const float* ml = reinterpret_cast<const float*>(ws);
  const float* o = reinterpret_cast<const float*>(ws + plan_ml_bytes(hd));
  const PlanSeg* segs = reinterpret_cast<const PlanSeg*>(dp + hd.seg_off);
  const int32_t* eoff = reinterpret_cast<const int32_t*>(dp + hd.eoff_off);
  const PlanEntry* ents = reinterpret_cast<const PlanEntry*>(dp + hd.ent_off);
  float* of = out_dtype == KV_DTYPE_F32 ? reinterpret_cast<float*>(d_out) : nullptr;
  __nv_bfloat16* ob = out_dtype == KV_DTYPE_BF16 ? reinterpret_cast<__nv_bfloat16*>(d_out) : nullptr;
  const dim3 mg(hd.n_seq, (n_q_heads + kMergePlanWarps - 1) / kMergePlanWarps);
  const int gr = grid > 0 ? grid : 1;
  const dim3 mb(kMergePlanWarps * 32);
  cudaError_t e = cudaSuccess;
  if (p->merge_deep_ctas < 0) {  // resident CTAs of the deeper variant, once per pool
    int occ = 0;
    e = p->D == 128 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                          &occ, merge_plan_kernel<128, 12>, kMergePlanWarps * 32, 0)
                    : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                          &occ, merge_plan_kernel<64, 12>, kMergePlanWarps * 32, 0);
    if (e != cudaSuccess) return KV_ERR_CUDA;
    p->merge_deep_ctas = occ * pool_sm_count(p);
  }
  const bool deep = static_cast<long long>(mg.x) * mg.y <= p->merge_deep_ctas;
  auto go = [&](auto kern) {
    return pkv::launch_kernel(p->pdl, kern, mg, mb, 0, as_stream(stream), segs, eoff, ents, hd.W,
                              gr, hd.c_max, ml, o, p->H, n_q_heads, of, ob);
  };
  if (p->D == 128)
    e = deep ? go(merge_plan_kernel<128, 12>) : go(merge_plan_kernel<128, 8>);
  else
    e = deep ? go(merge_plan_kernel<64, 12>) : go(merge_plan_kernel<64, 8>);
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kvStatus paged_decode_attention_planned(kvPool* p, int layer, const void* d_q, int n_q_heads,
                                        const int32_t* d_block_table, int max_blocks,
                                        const void* d_plan, const void* h_plan, float scale,
                                        void* d_out, int out_dtype, void* d_workspace,
                                        size_t workspace_bytes, void* stream) {
  if (out_dtype != KV_DTYPE_F32 && out_dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  kvStatus s = paged_decode_partials_planned(p, layer, d_q, n_q_heads, d_block_table, max_blocks,
                                             d_plan, h_plan, scale, d_workspace, workspace_bytes,
                                             stream);
  if (s != KV_OK) return s;
  return paged_decode_merge_planned(p, n_q_heads, d_plan, h_plan, d_out, out_dtype, d_workspace,
                                    workspace_bytes, stream);
}

// ------------------------------------------------------ whole decode step

namespace {
struct StepLayout {
  size_t q, k, v, slots, pairs, table, lens, plan, meta_end, out, ws, total;
};

// The device address of a caller's host buffer that is page-locked and
// mapped into the device's address space (cudaMallocHost / cudaHostAlloc, or
// a mapped cudaHostRegister, under unified addressing), else nullptr.
void* host_mapped(const void* h) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    (void)cudaGetLastError();  // clear this call's own error
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

StepLayout step_layout(const kvPool* p, int n_seq, int n_q_heads, int max_blocks) {
  StepLayout l;
  const size_t L = p->L, n = n_seq;
  size_t off = 0;
  l.q = off;
  off += align256(L * n * n_q_heads * p->D * p->in_esize);
  l.k = off;
  off += align256(L * n * p->H * p->D * p->in_esize);
  l.v = off;
  off += align256(L * n * p->H * p->D * p->in_esize);
  l.slots = off;
  off += align256(n * sizeof(int64_t));
  l.pairs = off;
  off += align256(n * 2 * sizeof(int32_t));
  l.table = off;
  off += align256(n * static_cast<size_t>(max_blocks) * sizeof(int32_t));
  l.lens = off;
  off += align256(n * sizeof(int32_t));
  l.plan = off;
  off += align256(paged_decode_plan_bytes(p, n_seq, n_q_heads));
  l.meta_end = off;  // slots .. plan: the metadata moved by one copy
  l.out = off;
  off += align256(L * n * n_q_heads * p->D * sizeof(float));
  l.ws = off;
  const size_t ws_plain = ws_layout(p, n_seq, n_q_heads / p->H).total;
  const size_t ws_plan = plan_workspace_bytes(plan_max_segs(n_seq, p->H), kPlanMaxCols, p->D);
  off += align256(ws_plain > ws_plan ? ws_plain : ws_plan);
  l.total = off;
  return l;
}
}  // namespace

size_t kv_decode_step_staging_bytes(const kvPool* p, int n_seq, int n_q_heads, int max_blocks) {
  if (!p || n_seq < 0 || n_q_heads <= 0 || n_q_heads % p->H != 0 || max_blocks <= 0) return 0;
  return step_layout(p, n_seq, n_q_heads, max_blocks).total;
}

kvStatus paged_prefill_attention(kvPool* p, int layer, const void* d_q, int n_q_heads,
                                 const int32_t* d_block_table, int max_blocks,
                                 const int32_t* d_chunk_start, const int32_t* d_context_lens,
                                 int n_seq, int max_chunk, float scale, void* d_out,
                                 int out_dtype, void* stream) {
  if (max_chunk < 0) return KV_ERR_INVALID_ARG;
  return prefill_common(p, layer, d_q, n_q_heads, d_block_table, max_blocks, d_chunk_start,
                        d_context_lens, n_seq, max_chunk, nullptr, 0, scale, d_out, out_dtype,
                        stream);
}

kvStatus paged_prefill_attention_scheduled(kvPool* p, int layer, const void* d_q, int n_q_heads,
                                           const int32_t* d_block_table, int max_blocks,
                                           const int32_t* d_chunk_start,
                                           const int32_t* d_context_lens, int n_seq,
                                           const void* d_sched, int n_items, float scale,
                                           void* d_out, int out_dtype, void* stream) {
  if (n_items < 0 || (n_items > 0 && (!d_sched || !aligned16(d_sched))))
    return KV_ERR_INVALID_ARG;
  return prefill_common(p, layer, d_q, n_q_heads, d_block_table, max_blocks, d_chunk_start,
                        d_context_lens, n_seq, 0, static_cast<const int4*>(d_sched), n_items,
                        scale, d_out, out_dtype, stream);
}

namespace {
// Workspace of a staged prefill: bfloat16 copies of K and V as rows
// (copy block, slot) of H_kv * D_h values, then the copy's table.
struct StageLayout {
  long long rows;
  size_t k, v, table, total;
};
StageLayout stage_layout(const kvPool* p, int n_seq, int max_blocks) {
  StageLayout l;
  l.rows = static_cast<long long>(n_seq) * max_blocks * p->B;
  const size_t kv = align256(static_cast<size_t>(l.rows) * p->H * p->D * 2);
  l.k = 0;
  l.v = kv;
  l.table = 2 * kv;
  l.total = l.table + align256(static_cast<size_t>(n_seq) * max_blocks * sizeof(int32_t));
  return l;
}
}  // namespace

size_t paged_prefill_staging_bytes(const kvPool* p, int n_seq, int max_blocks) {
  if (!p || n_seq < 0 || max_blocks <= 0 || p->dtype != KV_DTYPE_FP8_E4M3) return 0;
  return stage_layout(p, n_seq, max_blocks).total;
}

kvStatus paged_prefill_attention_staged(kvPool* p, int layer, const void* d_q, int n_q_heads,
                                        const int32_t* d_block_table, int max_blocks,
                                        const int32_t* d_chunk_start,
                                        const int32_t* d_context_lens, int n_seq, int max_chunk,
                                        const void* d_sched, int n_items, float scale,
                                        void* d_out, int out_dtype, void* d_workspace,
                                        size_t workspace_bytes, void* stream) {
  if (!p || !p->k || n_seq < 0 || max_chunk < 0 || n_items < 0) return KV_ERR_INVALID_ARG;
  if (d_sched && !aligned16(d_sched)) return KV_ERR_INVALID_ARG;
  const int4* sched = static_cast<const int4*>(d_sched);
  if (p->dtype != KV_DTYPE_FP8_E4M3)  // read in place
    return prefill_common(p, layer, d_q, n_q_heads, d_block_table, max_blocks, d_chunk_start,
                          d_context_lens, n_seq, sched ? 0 : max_chunk, sched, n_items, scale,
                          d_out, out_dtype, stream);
  if (layer < 0 || layer >= p->L || n_q_heads <= 0 || n_q_heads % p->H != 0)
    return KV_ERR_INVALID_ARG;
  if (ilog2_small(n_q_heads / p->H) < 0 || !prefill_shape(p, true)) return KV_ERR_UNSUPPORTED;
  if (n_seq == 0 || (sched ? n_items == 0 : max_chunk == 0)) return KV_OK;
  if (!d_block_table || !d_context_lens || max_blocks <= 0 || n_seq > 65535)
    return KV_ERR_INVALID_ARG;
  const StageLayout l = stage_layout(p, n_seq, max_blocks);
  if (l.rows >= (1LL << 31)) return KV_ERR_INVALID_ARG;
  if (!d_workspace || (reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0 ||
      workspace_bytes < l.total)
    return KV_ERR_INVALID_ARG;
  kvStatus s = ensure_device(p);
  if (s != KV_OK) return s;
  unsigned char* w = static_cast<unsigned char*>(d_workspace);
  int32_t* stage_table = reinterpret_cast<int32_t*>(w + l.table);
  const int row_vecs = p->H * p->D / 16;
  const cudaError_t e = pkv::launch_kernel(
      p->pdl, prefill_stage_fp8_kernel, dim3(max_blocks, n_seq), dim3(128), 0, as_stream(stream),
      reinterpret_cast<const uint4*>(p->k), reinterpret_cast<const uint4*>(p->v), d_block_table,
      d_context_lens, max_blocks, layer, p->N, p->B, row_vecs, reinterpret_cast<uint4*>(w + l.k),
      reinterpret_cast<uint4*>(w + l.v), stage_table, p->d_status);
  if (e != cudaSuccess) return KV_ERR_CUDA;
  // descriptors of the copy, kept while the workspace and its size stay
  if (p->stage_base != d_workspace || p->stage_rows != l.rows) {
    const int rm = pkv::mma_box_rows(p->B, pkv::mma_stage_tokens(p->D));
    for (int kv = 0; kv < 2; ++kv) {
      s = encode_rows_map(w + (kv ? l.v : l.k), static_cast<unsigned long long>(l.rows),
                          static_cast<unsigned long long>(p->H) * p->D, 2,
                          CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, rm, true,
                          reinterpret_cast<CUtensorMap*>(p->tmap_stage[kv]));
      if (s != KV_OK) {
        p->stage_base = nullptr;
        return s;
      }
    }
    p->stage_base = d_workspace;
    p->stage_rows = l.rows;
  }
  const PrefillStage st{reinterpret_cast<const CUtensorMap*>(p->tmap_stage[0]),
                        reinterpret_cast<const CUtensorMap*>(p->tmap_stage[1]), stage_table,
                        n_seq * max_blocks};
  return prefill_common(p, layer, d_q, n_q_heads, d_block_table, max_blocks, d_chunk_start,
                        d_context_lens, n_seq, sched ? 0 : max_chunk, sched, n_items, scale,
                        d_out, out_dtype, stream, &st);
}

kvStatus kv_decode_step_host(kvPool* p, const int32_t* seq_ids, int n_seq, int n_q_heads,
                             int max_blocks, const void* h_q, const void* h_k_new,
                             const void* h_v_new, float scale, float* h_out, void* d_staging,
                             size_t staging_bytes, void* stream) {
  if (!p || !p->k || n_seq <= 0 || !seq_ids || !h_q || !h_k_new || !h_v_new || !h_out ||
      !d_staging || max_blocks <= 0)
    return KV_ERR_INVALID_ARG;
  if (n_q_heads <= 0 || n_q_heads % p->H != 0) return KV_ERR_INVALID_ARG;
  const StepLayout l = step_layout(p, n_seq, n_q_heads, max_blocks);
  if (staging_bytes < l.total || !aligned16(d_staging)) return KV_ERR_INVALID_ARG;
  // every table must fit max_blocks after the step
  for (int i = 0; i < n_seq; ++i) {
    auto it = p->seqs.find(seq_ids[i]);
    const long long len = it == p->seqs.end() ? 0 : it->second.len;
    if ((len + 1 + p->B - 1) / p->B > max_blocks) return KV_ERR_INVALID_ARG;
  }
  kvStatus s = ensure_device(p);
  if (s != KV_OK) return s;
  // page-locked host staging of the metadata (slots .. plan)
  const size_t meta = l.meta_end - l.slots;
  if (p->h_pinned_bytes < meta) {
    if (p->h_pinned) cudaFreeHost(p->h_pinned);
    p->h_pinned = nullptr;
    p->h_pinned_bytes = 0;
    void* h = nullptr;
    if (cudaMallocHost(&h, meta) != cudaSuccess) return KV_ERR_CUDA;
    p->h_pinned = static_cast<unsigned char*>(h);
    p->h_pinned_bytes = meta;
  }
  unsigned char* hm = p->h_pinned - l.slots;  // hm + l.x: host copy of region x
  int64_t* h_slots = reinterpret_cast<int64_t*>(hm + l.slots);
  int32_t* h_pairs = reinterpret_cast<int32_t*>(hm + l.pairs);
  int32_t* h_table = reinterpret_cast<int32_t*>(hm + l.table);
  int32_t* h_lens = reinterpret_cast<int32_t*>(hm + l.lens);
  unsigned char* h_plan = hm + l.plan;
  cudaStream_t st = as_stream(stream);
  unsigned char* d = reinterpret_cast<unsigned char*>(d_staging);
  const size_t qb = static_cast<size_t>(p->L) * n_seq * n_q_heads * p->D * p->in_esize;
  const size_t kb = static_cast<size_t>(p->L) * n_seq * p->H * p->D * p->in_esize;
  const size_t ob = static_cast<size_t>(p->L) * n_seq * n_q_heads * p->D * sizeof(float);
  // the caller's buffers, where the device can address them in place
  // (page-locked host memory mapped into its address space): the kernels
  // then read q and the new K / V rows and the merge writes the outputs
  // through the mapping, with no staging copy; other buffers are copied
  const unsigned char* mq = static_cast<const unsigned char*>(host_mapped(h_q));
  const void* mk = host_mapped(h_k_new);
  const void* mv = host_mapped(h_v_new);
  float* mo = static_cast<float*>(host_mapped(h_out));
  const bool kv_direct = mk != nullptr && mv != nullptr;
  // several layers: layer l's q goes over on the side stream (and, when
  // copied back, layer l's output too), each ordered against the attention
  // of that layer by an event, so that the copies overlap the other layers'
  // kernels
  const bool overlap = p->L > 1 && (!mq || !mo);
  cudaStream_t cs = nullptr;
  const size_t q_layer = static_cast<size_t>(n_seq) * n_q_heads * p->D;
  if (overlap) {
    if (!p->side_stream) {
      cudaStream_t ns = nullptr;
      if (cudaStreamCreateWithFlags(&ns, cudaStreamNonBlocking) != cudaSuccess) return KV_ERR_CUDA;
      p->side_stream = ns;
    }
    if (p->step_events.size() != static_cast<size_t>(2 * p->L)) {
      for (void* e : p->step_events)
        if (e) cudaEventDestroy(static_cast<cudaEvent_t>(e));
      p->step_events.assign(2 * p->L, nullptr);
      for (auto& e : p->step_events) {
        cudaEvent_t ne = nullptr;
        if (cudaEventCreateWithFlags(&ne, cudaEventDisableTiming) != cudaSuccess)
          return KV_ERR_CUDA;
        e = ne;
      }
    }
    cs = static_cast<cudaStream_t>(p->side_stream);
  }
  // a step that fails after its copies were issued waits for them before
  // returning, so that the caller may reuse its buffers at once
  auto fail = [&](kvStatus e) {
    if (overlap) cudaStreamSynchronize(cs);
    cudaStreamSynchronize(st);
    return e;
  };
  // host -> device, first: what needs no reservation (q; K and V unless
  // read in place), so that the copies run while the host reserves
  bool ok = true;
  if (!overlap && !mq)
    ok &= cudaMemcpyAsync(d + l.q, h_q, qb, cudaMemcpyHostToDevice, st) == cudaSuccess;
  if (!kv_direct) {
    ok &= cudaMemcpyAsync(d + l.k, h_k_new, kb, cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok &= cudaMemcpyAsync(d + l.v, h_v_new, kb, cudaMemcpyHostToDevice, st) == cudaSuccess;
  }
  if (overlap && !mq) {
    for (int layer = 0; layer < p->L && ok; ++layer) {
      const size_t off = layer * q_layer * p->in_esize;
      ok &= cudaMemcpyAsync(d + l.q + off, static_cast<const unsigned char*>(h_q) + off,
                            q_layer * p->in_esize, cudaMemcpyHostToDevice, cs) == cudaSuccess;
      ok &= cudaEventRecord(static_cast<cudaEvent_t>(p->step_events[2 * layer]), cs) ==
            cudaSuccess;
    }
  }
  if (!ok) return fail(KV_ERR_CUDA);
  // host: reserve (all or nothing), the tables, and the sharing-aware plan
  // of the tensor-core passes (shared blocks read once)
  int n_cow = 0;
  s = seq_append_slots(p, seq_ids, n_seq, h_slots, h_pairs, &n_cow);
  if (s != KV_OK) return fail(s);
  s = seq_block_table(p, seq_ids, n_seq, max_blocks, h_table, h_lens);
  if (s != KV_OK) return fail(s);
  const int G = n_q_heads / p->H;
  const bool planned = decode_kernel(p) != kKernelCudaCores && ilog2_small(G) >= 0 &&
                       (p->D == 64 || p->D == 128);
  if (planned) {
    // the per-CTA start records cost the host about as much as three or
    // four split launches save with them (each CTA otherwise finds its
    // first piece itself): built when the plan serves four or more layers
    size_t ws_need = 0;
    s = plan_build(p, seq_ids, n_seq, n_q_heads, max_blocks, 0, h_plan,
                   paged_decode_plan_bytes(p, n_seq, n_q_heads), &ws_need, p->L >= 4);
    if (s != KV_OK) return fail(s);
  }
  // the step's metadata (slots, copy pairs, tables, lengths, plan) in one copy
  if (cudaMemcpyAsync(d + l.slots, p->h_pinned, (planned ? l.meta_end : l.plan) - l.slots,
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return fail(KV_ERR_CUDA);
  // device: copy shared tails, write the new token in every layer, attend.
  // With a plan on a bfloat16 or FP8 pool the split pass of each layer
  // writes that layer's new rows itself (the CTA reading a sequence's last
  // block writes its newest token first), one launch less per step.
  const bool fused = planned && (p->dtype == KV_DTYPE_BF16 || p->dtype == KV_DTYPE_FP8_E4M3);
  s = cow_copy(p, reinterpret_cast<const int32_t*>(d + l.pairs), n_cow, stream);
  if (s != KV_OK) return fail(s);
  const unsigned char* kn = kv_direct ? static_cast<const unsigned char*>(mk) : d + l.k;
  const unsigned char* vn = kv_direct ? static_cast<const unsigned char*>(mv) : d + l.v;
  if (!fused) {
    s = reshape_and_cache(p, -1, kn, vn, reinterpret_cast<const int64_t*>(d + l.slots), n_seq,
                          stream);
    if (s != KV_OK) return fail(s);
  }
  const size_t kv_layer = static_cast<size_t>(n_seq) * p->H * p->D * p->in_esize;
  for (int layer = 0; layer < p->L; ++layer) {
    if (overlap && !mq &&
        cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(p->step_events[2 * layer]), 0) !=
            cudaSuccess)
      return fail(KV_ERR_CUDA);
    const unsigned char* q = (mq ? mq : d + l.q) + layer * q_layer * p->in_esize;
    float* out = mo ? mo + layer * q_layer
                    : reinterpret_cast<float*>(d + l.out) + layer * q_layer;
    const int32_t* table = reinterpret_cast<const int32_t*>(d + l.table);
    void* ws = d + l.ws;
    const size_t ws_bytes = staging_bytes - l.ws;
    if (fused) {
      s = paged_decode_partials_planned_write(p, layer, q, n_q_heads, kn + layer * kv_layer,
                                              vn + layer * kv_layer, table, max_blocks,
                                              d + l.plan, h_plan, scale, ws, ws_bytes, stream);
      if (s == KV_OK)
        s = paged_decode_merge_planned(p, n_q_heads, d + l.plan, h_plan, out, KV_DTYPE_F32, ws,
                                       ws_bytes, stream);
    } else if (planned) {
      s = paged_decode_attention_planned(p, layer, q, n_q_heads, table, max_blocks, d + l.plan,
                                         h_plan, scale, out, KV_DTYPE_F32, ws, ws_bytes, stream);
    } else {
      s = paged_decode_attention(p, layer, q, n_q_heads, table, max_blocks,
                                 reinterpret_cast<const int32_t*>(d + l.lens), n_seq, scale, out,
                                 KV_DTYPE_F32, ws, ws_bytes, stream);
    }
    if (s != KV_OK) return fail(s);
    if (overlap && !mo) {
      cudaEvent_t done = static_cast<cudaEvent_t>(p->step_events[2 * layer + 1]);
      const size_t off = layer * q_layer * sizeof(float);
      if (cudaEventRecord(done, st) != cudaSuccess || cudaStreamWaitEvent(cs, done, 0) != cudaSuccess ||
          cudaMemcpyAsync(reinterpret_cast<unsigned char*>(h_out) + off, d + l.out + off,
                          q_layer * sizeof(float), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return fail(KV_ERR_CUDA);
    }
  }
  if (!overlap && !mo &&
      cudaMemcpyAsync(h_out, d + l.out, ob, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return fail(KV_ERR_CUDA);
  if (overlap && cudaStreamSynchronize(cs) != cudaSuccess) return KV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KV_ERR_CUDA;
  return KV_OK;
}

}  // extern "C"
