// Split-K paged decode attention, partial pass, bfloat16 K/V on tensor cores.
//
// Same contract, work split and workspace as decode.cuh (see there): per
// piece of a segment (a block range of one table row and one K/V head) it
// emits the base-2 online-softmax statistics m, l and the unnormalised O of
// every query column of the segment.  Without a plan a segment is one
// (sequence, K/V head) and its columns are that sequence's G query heads;
// with a plan (plan.h) a segment of blocks shared by several sequences
// carries all of their columns, so each shared block is read once.
//
// The products of a 16-token tile and an 8-column n-tile are MMAs
// (m16n8k16, bf16 in, f32 accumulate):
//     S^T [16 tokens x 8 cols] = K [16 x D] . Q^T [D x 8]        (D/16 MMAs)
//     O^T [D x 8 cols]        += V^T [D x 16] . P^T [16 x 8]      (2 x D/16)
// K and V^T come straight from shared memory with ldmatrix (V transposed on
// load), Q^T lives in registers for the whole piece, and P^T is the S^T
// accumulator turned into bf16 and transposed inside the warp with movmatrix.
// P is split into a bf16 high part and a bf16 remainder (two MMAs) so that
// the weights keep ~16 mantissa bits.  Columns past the segment's are zero.
//
// Shared memory: each stage holds TS token rows of K and of V for one K/V
// head (64 tokens at D = 128), written by TMA with the 128-byte swizzle (rows
// of 64 elements, the 16-byte chunk c of row r stored at chunk c ^ (r mod 8)),
// so the 8 rows an ldmatrix phase reads fall in 8 different bank groups.  All
// four consumer warps consume every stage.  A piece with NT n-tiles (1, 2 or
// 4) gives warp w the n-tile w mod NT and the stage's tiles w / NT, w / NT +
// 4 / NT, ...; each warp keeps its own running softmax state, and the states
// of warps sharing an n-tile are merged through shared memory at the end of
// the piece.
#pragma once

#include <cuda_fp16.h>

#include "decode.cuh"

namespace pkv {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA on fp16 operands (the FP8 pass: E4M3 codes convert exactly).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (lo, hi) floats -> f16x2, lo in the low half, saturating at +-65504
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// four E4M3 codes (bytes, lowest first) -> two f16x2 words (exact)
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// 8-bit transposing load of a 16 x 16 byte tile (lanes 0-15 give the row
// addresses): lane 4g + t receives the bytes of rows 4t .. 4t + 3 in column g
// (r0) and in column g + 8 (r1), lowest row in the lowest byte (layout
// checked on the GPU with a tile of known bytes).
__device__ __forceinline__ void ldsm8_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x1.trans.shared.b8 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// FP8 pass, token order inside a 16-token tile.  ldsm8_t hands lane (g, t)
// the rows that lanes 4t .. 4t + 3 address, which an fp16 A fragment holds
// in its k-slots 2t, 2t + 1, 2t + 8, 2t + 9; lane i addresses tile row
// f8_vrow(i).  Row k of S^T (= k-slot k of P^T) then stands for token
// f8_srow(k): k itself for k < 8, a rotation of 8 .. 15 above (the sum over
// tokens does not depend on their order).  This choice keeps both the K
// loads (rows f8_srow(g), f8_srow(g + 8) over the eight g) and each 8-row
// phase of ldsm8_t on eight distinct 128-byte swizzle phases: no bank
// conflicts (the order 0, 1, 4, 5, 8, 9, 12, 13 / 2, 3, 6, 7, 10, 11, 14, 15
// of natural row addresses put rows r and r + 8 in one K load).
__device__ __forceinline__ int f8_vrow(int i) {
  return (i & 3) < 2 ? 2 * (i >> 2) + (i & 3) : 8 + ((2 * (i >> 2) + (i & 1) + 4) & 7);
}
__device__ __forceinline__ int f8_srow(int k) { return k < 8 ? k : 8 + ((k + 4) & 7); }

// q8_0 pass: four int8 codes (lowest byte first) as two fp16 pairs, exactly:
// the half 0x6400 | (c + 128) is 1024 + c + 128, and subtracting 1152 leaves
// c (every step exact in fp16's 11-bit significand).
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
  const uint32_t bias = 0x64806480u;  // 1152, 1152
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(bias));
}

// fp16 halves of a 32-bit word as floats
__device__ __forceinline__ float half_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// (lo, hi) floats -> bf16x2 with lo in the low half (round to nearest even)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Tokens per stage of the tensor-core pass: 64 tokens (16 KiB of K and 16
// KiB of V at D = 128 in bf16), 128 in FP8 (16 KiB of codes each).
constexpr int mma_stage_tokens(int D, bool f8 = false) {
  return f8 ? 128 : 16 * 4 * (D == 64 ? 2 : 1);
}

// Rows per TMA box for block size B and TS-token stages: a whole block when
// it divides the stage, else the stage, else half of it (an FP8 stage of 128
// tokens over blocks of 64 k + 64 rows); boxes never cross a block.
constexpr int mma_box_rows(int B, int TS) {
  return B < TS ? B : (B % TS == 0 ? TS : TS / 2);
}

// F8: the pool holds E4M3 codes and the contractions run on fp16 operands
// (codes convert exactly).  S = K . Q^T is unchanged by any permutation of
// the head dimension applied to both operands, so the A fragments of K take
// d = 16 ks + 4 t .. 4 t + 3 (four consecutive codes, one 32-bit load per
// row, two conversions) and Q's fragments the same dimensions; V's transpose
// comes from the 8-bit transposing ldmatrix (ldsm8_t), whose byte order and
// row addresses fix the order of the tile's tokens in both contractions
// (f8_vrow, f8_srow), and is converted to fp16 in registers.  FP8 stages hold 128 tokens (16 KiB of
// codes each of K and V): every consumer warp then takes two 16-token tiles
// of a stage, whose dependency chains the unrolled tile loop interleaves.
template <int D, int G, bool F8 = false, bool Q8 = false>
struct MmaCfg {
  static constexpr int TS = mma_stage_tokens(D, F8);  // tokens per stage
  static constexpr int TILES = TS / 16;           // 16-token tiles per stage
  static constexpr int KS = D / 16;               // k-steps of Q.K and m-tiles of O^T
  static constexpr int ESZ = F8 ? 1 : 2;          // bytes per stored element
  static constexpr int HALVES = F8 ? 1 : D / 64;  // 128-byte swizzled boxes per row set
  static constexpr int HALF_BYTES = TS * 128;     // one box column of a K (or V) stage
  static constexpr int STAGE_BYTES = TS * D * ESZ;  // K (or V) per stage
  // Q8 (with F8's one-byte layout): the codes' fp16 scales of a stage, K or V
  static constexpr int SC_BYTES = Q8 ? TS * (D / 32) * 2 : 0;

  static constexpr int NST = 3;                   // stages in the ring
  static constexpr int CC = 4;                    // columns per combine pass
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!F8 || D == 128, "FP8 rows are 128 codes");
  static_assert(!Q8 || F8, "q8_0 shares the one-byte code layout");
  static_assert(G >= 1 && G <= 8, "group size");
  static_assert(TILES % ((F8 ? 2 : 1) * kConsumerWarps) == 0, "whole tiles (pairs) per warp");
};

// Piece descriptors the producer can publish ahead of the consumers.
constexpr int kPieceRing = 4;

// Fused slot write, by one warp: the newest token's row (rep, head) of the
// step's K (and / or V) of this layer, D bfloat16 values, into slot o of
// physical block pid (bfloat16 pools: a copy; FP8 pools: the E4M3 code
// nearest to x / scale, ties to even, saturating at 448), then a proxy fence
// so that the TMA copies this warp issues next see it.
template <int D, bool F8>
__device__ __forceinline__ void write_new_row(const DecodeArgs& a, int rep, int head, int pid,
                                              int o, bool do_k, bool do_v, int lane) {
  constexpr int VECS = D * 2 / 16;  // 16-byte vectors of bf16 per row
  const long long src = ((long long)rep * a.n_kv_heads + head) * D;
  const long long dst = (((long long)a.layer * a.n_blocks + pid) * a.block_size + o) *
                            a.n_kv_heads * D + (long long)head * D;
  for (int i = lane; i < 2 * VECS; i += 32) {
    const bool is_k = i < VECS;
    if ((is_k && !do_k) || (!is_k && !do_v)) continue;
    const int vi = is_k ? i : i - VECS;
    const uint4 x = reinterpret_cast<const uint4*>(
        reinterpret_cast<const unsigned char*>(is_k ? a.k_new : a.v_new) + src * 2)[vi];
    void* pool = is_k ? a.k_pool : a.v_pool;
    if constexpr (F8) {
      const float scale = is_k ? a.k_scale_w : a.v_scale_w;
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
      reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(pool) + dst)[vi] =
          make_uint2(out[0], out[1]);
    } else {
      reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(pool) + dst * 2)[vi] = x;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <int D, int G, bool F8 = false, bool Q8 = false>
constexpr int decode_mma_smem_bytes() {
  using C = MmaCfg<D, G, F8, Q8>;
  return 2 * C::NST * C::STAGE_BYTES        // K and V stages
         + 2 * C::NST * C::SC_BYTES         // Q8: their scales
         + kConsumerWarps * C::CC * D * 4   // combine: O per warp, CC columns at a time
         + kConsumerWarps * 8 * 2 * 4       // combine: m, l per warp and column
         + 2 * C::NST * 8                   // mbarriers
         + kTableCache * 4                  // producer table cache
         + kPieceRing * (48 + 16)           // piece descriptors and their mbarriers
         + 64 + 128 + 1024;                 // walk state, start record, 1 KiB alignment
}

// swizzled shared address of (row r, 8-element chunk c) inside a half
__device__ __forceinline__ uint32_t swz(uint32_t half_base, int r, int c) {
  return half_base + r * 128 + ((c ^ (r & 7)) << 4);
}

// One piece of work: blocks [b0, b1) of table row `rep` for K/V head `head`,
// tokens below tok_end, `ncols` query columns taken from members mem.. (or
// from `rep` itself without a plan); `seg` numbers the segment.
struct Piece {
  int rep, head, b0, b1, tok_end, ncols, mem, seg;
  int last;  // the piece holds its segment's last block
};

// Walks the plan's segments over the block range [r, r1).
struct PlanWalker {
  const PlanSeg* segs;
  int n_segs, B, s;
  long long r, r1;

  // A piece for every segment whose units meet [r, r1); its blocks are those
  // whose first unit lies in the range, possibly none.
  __device__ bool next(Piece& p) {
    while (r < r1 && s < n_segs) {
      const PlanSeg sg = segs[s];
      const long long len = sg.b1 - sg.b0;
      const long long w = sg.w > 0 ? sg.w : 1;
      if (len <= 0 || r >= sg.wpre + len * w) {
        ++s;
        continue;
      }
      const long long end = r1 < sg.wpre + len * w ? r1 : sg.wpre + len * w;
      const long long jb = (r - sg.wpre + w - 1) / w, je = (end - sg.wpre + w - 1) / w;
      p.rep = sg.rep;
      p.head = sg.head;
      p.b0 = sg.b0 + (int)jb;
      p.b1 = sg.b0 + (int)je;
      p.tok_end = p.b1 * B < sg.tok_end ? p.b1 * B : sg.tok_end;
      p.ncols = sg.ncols;
      p.mem = sg.mem;
      p.seg = s;
      p.last = p.b1 == sg.b1;
      r = end;
      return true;
    }
    return false;
  }
};

// One warp: the segment whose block range holds r0 (segments sorted by wpre).
__device__ inline int plan_find(const PlanSeg* segs, int n_segs, long long r0) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = n_segs;  // wpre[lo] <= r0 holds throughout
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool ok = idx < hi && segs[idx].wpre <= r0;
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    const int L = 31 - __clz(m);
    lo = lo + L * step;
    hi = lo + step < hi ? lo + step : hi;
  }
  return lo;
}

template <int D, int G, bool PLAN, bool F8 = false, bool Q8 = false>
__global__ void __launch_bounds__(kThreads, 2)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
  using C = MmaCfg<D, G, F8, Q8>;
  constexpr int NST = C::NST;
  // the declared alignment stays at 16 so that the explicit round-up to the
  // 1 KiB the 128-byte swizzle needs is never folded away
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* k_st = smem;
  unsigned char* v_st = k_st + NST * C::STAGE_BYTES;
  unsigned char* sc_st = v_st + NST * C::STAGE_BYTES;  // Q8: K scales, then V scales
  float* cmb_o = reinterpret_cast<float*>(sc_st + 2 * NST * C::SC_BYTES);
  float* cmb_ml = cmb_o + kConsumerWarps * C::CC * D;
  uint64_t* full = reinterpret_cast<uint64_t*>(cmb_ml + kConsumerWarps * 8 * 2);
  uint64_t* empty = full + NST;
  long long* walk = reinterpret_cast<long long*>(empty + NST);
  int32_t* tcache = reinterpret_cast<int32_t*>(walk + 4);
  PlanStart* rec_s = reinterpret_cast<PlanStart*>(tcache + kTableCache);
  Piece* ring = reinterpret_cast<Piece*>(rec_s + 1);
  uint64_t* dfull = reinterpret_cast<uint64_t*>(ring + kPieceRing);
  uint64_t* dempty = dfull + kPieceRing;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int H = a.n_kv_heads;
  const int UR = mma_box_rows(B, C::TS);     // rows per TMA box (a multiple of 8)
  const int SB = C::TS / UR;                 // boxes per stage
  const int STG = SB * UR;                   // tokens per stage
  const uint32_t unit_bytes = (uint32_t)UR * D * C::ESZ;  // K (or V) bytes of one box row set

  // self-check: swizzled TMA destinations must sit on 1 KiB boundaries
  if ((smem_u32(k_st) & 1023u) != 0u) {
    if (threadIdx.x == 0) record_status(a.status, 32);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kPieceRing; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&dempty[i], kConsumerWarps);
    }
    fence_barrier_init();
  }
  // The walk start and the producer's first block-table entries read only
  // host-written metadata (plan, context lengths, tables), complete before the
  // first kernel of the stream's programmatic chain started, so they are
  // read before waiting for the previous grid; the pool, q and the workspace
  // only after it.
  // a plan with start records for this grid: the CTA's first piece and its
  // first blocks' ids come with one 128-byte read (no search, no table read)
  const bool use_rec = PLAN && a.starts != nullptr && a.start_grid == a.grid;
  if (warp == 0) {
    if constexpr (PLAN) {
      const long long W = a.plan_W;
      long long chunk = (W + a.grid - 1) / a.grid;
      if (chunk == 0) chunk = 1;
      int s0 = 0;
      if (use_rec) {
        reinterpret_cast<int32_t*>(rec_s)[lane] =
            reinterpret_cast<const int32_t*>(a.starts + blockIdx.x)[lane];
      } else {
        const long long r0 = (long long)blockIdx.x * chunk;
        s0 = r0 < W ? plan_find(a.segs, a.n_segs, r0) : a.n_segs;
      }
      if (lane == 0) {
        walk[0] = s0;
        walk[1] = 0;
        walk[2] = W;
        walk[3] = chunk;
      }
    } else {
      WalkStart w = find_start(a.ctx, a.n_seq, B, H, a.max_blocks, a.grid, blockIdx.x, a.status);
      if (lane == 0) {
        walk[0] = w.s;
        walk[1] = w.pre;
        walk[2] = w.W;
        walk[3] = w.chunk;
      }
    }
  }
  __syncthreads();

  const long long W = walk[2], chunk = walk[3];
  const long long r_begin = (long long)blockIdx.x * chunk;
  const long long r_end = r_begin + chunk < W ? r_begin + chunk : W;
  PieceWalker pw;
  PlanWalker plw;
  if constexpr (PLAN) {
    plw.segs = a.segs;
    plw.n_segs = a.n_segs;
    plw.B = B;
    plw.s = (int)walk[0];
    plw.r = r_begin;
    plw.r1 = r_end;
  } else {
    pw.ctx = a.ctx;
    pw.n_seq = a.n_seq;
    pw.B = B;
    pw.H = H;
    pw.max_blocks = a.max_blocks;
    pw.s = (int)walk[0];
    pw.pre = walk[1];
    pw.r = r_begin;
    pw.r1 = r_end;
  }
  bool rec_first = use_rec;  // the first piece comes from the start record
  auto next_piece = [&](Piece& p) -> bool {
    if constexpr (PLAN) {
      if (rec_first) {
        rec_first = false;
        const PlanStart& R = *rec_s;
        if (R.seg < 0) {
          plw.s = plw.n_segs;
          return false;
        }
        p.rep = R.rep;
        p.head = R.head;
        p.b0 = R.b0;
        p.b1 = R.b1;
        p.tok_end = R.tok_end;
        p.ncols = R.ncols;
        p.mem = R.mem;
        p.seg = R.seg;
        p.last = R.last;
        plw.s = R.seg;
        plw.r = R.r_after;
        return true;
      }
      return plw.next(p);
    } else {
      if (!pw.next()) return false;
      p.rep = pw.seq;
      p.head = pw.head;
      p.b0 = pw.b0;
      p.b1 = pw.b1;
      p.tok_end = pw.b1 * B < pw.ctx_len ? pw.b1 * B : pw.ctx_len;
      p.ncols = G;
      p.mem = -1;
      p.seg = pw.seq * H + pw.head;
      p.last = 0;
      return true;
    }
  };
  auto wait_previous_grid = [&]() {
    griddep_wait();
    griddep_launch_dependents();
    if constexpr (!PLAN) {
      if (blockIdx.x == 0 && warp == 0)
        write_prefix(a.ctx, a.n_seq, B, H, a.max_blocks, a.ws_pre);
    }
  };

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
    }
    bool alive = true;
    int stage = 0;
    TableCache tc;
    tc.ent = tcache;
    // The producer alone walks the work list: each piece goes to the
    // consumers as a descriptor in shared memory, published one piece ahead
    // of its copies, so that no consumer reads the plan or waits on it at a
    // piece boundary.  A descriptor with rep = -1 ends the list.
    int npub = 0;
    auto publish = [&](const Piece& x, bool valid) {
      const int di = npub % kPieceRing;
      if (npub >= kPieceRing && alive) {
        if (!mbar_wait_bounded(&dempty[di], ((npub / kPieceRing) - 1) & 1, kWaitLimitNs)) {
          alive = false;
          if (lane == 0) record_status(a.status, 8);
        }
      }
      if (lane == 0) {
        Piece y = x;
        if (!valid) y.rep = -1;
        ring[di] = y;
        mbar_arrive(&dfull[di]);
      }
      __syncwarp();
      ++npub;
    };
    Piece p, pn;
    bool have = next_piece(p);
    if (have && !use_rec) tc.ensure(a.table, a.max_blocks, p.rep, p.b0, p.b0, lane);
    wait_previous_grid();
    publish(p, have);
    while (have) {
      const bool have_next = next_piece(pn);
      publish(pn, have_next);
      // the next piece's first table entries, loaded while this piece's
      // copies are issued and installed after them
      int32_t tnext[kTableCache / 32];
      if (have_next) {
        const int32_t* row = a.table + (long long)pn.rep * a.max_blocks;
#pragma unroll
        for (int i = 0; i < kTableCache / 32; ++i) {
          const int j = pn.b0 + i * 32 + lane;
          tnext[i] = j < a.max_blocks ? row[j] : 0;
        }
      }
      for (int tok0 = p.b0 * B; tok0 < p.tok_end; tok0 += STG) {
        const int slot = stage % NST;
        if (stage >= NST && alive) {
          if (!mbar_wait_bounded(&empty[slot], ((stage / NST) & 1) ^ 1, kWaitLimitNs)) {
            alive = false;
            if (lane == 0) record_status(a.status, 8);
          }
        }
        const int nvalid = p.tok_end - tok0 < STG ? p.tok_end - tok0 : STG;
        const int nunits = (nvalid + UR - 1) / UR;
        const int jl = (tok0 + (nunits - 1) * UR) / B;
        // the first stage of the record's piece takes the record's block ids
        const bool from_rec = use_rec && stage == 0 && p.seg == rec_s->seg &&
                              tok0 / B >= rec_s->b0 && jl - rec_s->b0 < rec_s->n_pid;
        if (!from_rec) tc.ensure(a.table, a.max_blocks, p.rep, tok0 / B, jl, lane);
        if constexpr (PLAN) {
          // fused slot write: the stage holding a private segment's last
          // token (the sequence's newest) writes that row first
          if (a.k_new != nullptr && p.last && p.ncols == G && tok0 + STG >= p.tok_end) {
            const int t = p.tok_end - 1;
            const int j = t / B;
            const int pid = from_rec ? rec_s->pid[j - rec_s->b0] : tc.ent[j - tc.base];
            if (pid >= 0 && pid < a.n_blocks)
              write_new_row<D, F8>(a, p.rep, p.head, pid, t - j * B, true, true, lane);
          }
        }
        // Q8: each box's rows also bring their scales (D / 32 fp16 a row)
        constexpr uint32_t kScRow = Q8 ? D / 32 * 2 : 0;
        if (lane == 0)
          mbar_arrive_expect_tx(&full[slot], 2u * nunits * (unit_bytes + UR * kScRow));
        __syncwarp();
        for (int u = lane; u < nunits; u += 32) {
          const int t = tok0 + u * UR;
          const int j = t / B;
          const int row = t - j * B;
          int pid = from_rec ? rec_s->pid[j - rec_s->b0] : tc.ent[j - tc.base];
          if (pid < 0 || pid >= a.n_blocks) {
            record_status(a.status, 1);
            pid = 0;  // stay in bounds; the result is flagged as invalid
          }
          const int y = (a.layer * a.n_blocks + pid) * B + row;
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h) {
            const int x = p.head * D + h * 64;
            const int off = slot * C::STAGE_BYTES + h * C::HALF_BYTES + u * UR * 128;
            tma_load_2d(k_st + off, &tmap_k, x, y, &full[slot]);
            tma_load_2d(v_st + off, &tmap_v, x, y, &full[slot]);
          }
          if constexpr (Q8) {
            // scales [L][N][H][B][D / 32]: the box's UR rows side by side
            const long long src =
                (((long long)a.layer * a.n_blocks + pid) * H + p.head) * B + row;
            const int so = slot * C::SC_BYTES + u * UR * kScRow;
            bulk_load(sc_st + so, reinterpret_cast<const unsigned char*>(a.k_sc) + src * kScRow,
                      UR * kScRow, &full[slot]);
            bulk_load(sc_st + NST * C::SC_BYTES + so,
                      reinterpret_cast<const unsigned char*>(a.v_sc) + src * kScRow, UR * kScRow,
                      &full[slot]);
          }
        }
        ++stage;
      }
      if (have_next) {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kTableCache / 32; ++i) tc.ent[i * 32 + lane] = tnext[i];
        tc.seq = pn.rep;
        tc.base = pn.b0;
        __syncwarp();
      }
      p = pn;
      have = have_next;
    }
    const int first = stage > NST ? stage - NST : 0;
    for (int k = first; k < stage; ++k)
      mbar_wait_bounded(&full[k % NST], (k / NST) & 1, kWaitLimitNs);
    return;
  }

  // -------------------------------------------------------------- consumers
  wait_previous_grid();
  const int g = lane >> 2;  // groupID: row of A / C, column of B
  const int t = lane & 3;   // thread in group
  const uint32_t k_base = smem_u32(k_st);
  const uint32_t v_base = smem_u32(v_st);
  const int cstride = PLAN ? a.c_max : G;  // columns per workspace slot
  bool alive = true;
  int stage = 0;
  // Q^T fragments of this warp's column of a piece (column wn*8 + g: dims
  // ks*16 + 2t (+1) and + 8; F8: the dimensions of the permuted K fragments,
  // 16 ks + 4t .. + 3), as raw bf16 pairs.  They are loaded one piece ahead,
  // so that a piece's first MMA does not wait for its member list and q rows
  // to arrive from memory.
  auto load_q = [&](const Piece& pc, uint32_t (&qr)[C::KS][2]) {
    const int NTc = pc.ncols <= 8 ? 1 : (pc.ncols <= 16 ? 2 : 4);
    const int col = (warp % NTc) * 8 + g;
    const bool colv = col < pc.ncols;
    int seqm = pc.rep, gi = col;
    if constexpr (PLAN) {
      const int mi = col / G;
      gi = col - mi * G;
      seqm = colv ? a.members[pc.mem + mi] : 0;
    }
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(
        reinterpret_cast<const unsigned char*>(a.q) +
        ((long long)seqm * a.n_q_heads + (long long)pc.head * G + (colv ? gi : 0)) * D * 2);
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      if constexpr (F8) {
        qr[ks][0] = colv ? qw[(ks * 16 + 4 * t) / 2] : 0u;
        qr[ks][1] = colv ? qw[(ks * 16 + 4 * t + 2) / 2] : 0u;
      } else {
        qr[ks][0] = colv ? qw[(ks * 16 + 2 * t) / 2] : 0u;
        qr[ks][1] = colv ? qw[(ks * 16 + 2 * t + 8) / 2] : 0u;
      }
    }
  };
  // the k-th piece descriptor the producer published (false: the list ended,
  // or the wait gave up)
  int nread = 0;
  auto read_piece = [&](Piece& x) -> bool {
    const int di = nread % kPieceRing;
    if (alive && !mbar_wait_bounded(&dfull[di], (nread / kPieceRing) & 1, kWaitLimitNs)) {
      alive = false;
      if (lane == 0) record_status(a.status, 8);
    }
    alive = __all_sync(0xffffffffu, alive);
    if (!alive) return false;
    x = ring[di];
    __syncwarp();
    if (lane == 0) mbar_arrive(&dempty[di]);
    ++nread;
    return x.rep >= 0;
  };
  Piece p, pn;
  uint32_t qn[C::KS][2];
  bool have = read_piece(p), have_next = false;
  if (have) load_q(p, qn);
  for (; have; p = pn, have = have_next) {
    const int NT = p.ncols <= 8 ? 1 : (p.ncols <= 16 ? 2 : 4);  // n-tiles of the piece
    const int WT = kConsumerWarps / NT;                           // warps per n-tile
    const int wt = warp / NT;
    uint32_t qf[C::KS][2];
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      qf[ks][0] = qn[ks][0];
      qf[ks][1] = qn[ks][1];
      if constexpr (F8) {
        // bf16 pairs -> fp16 pairs (exact in fp16's range)
#pragma unroll
        for (int i = 0; i < 2; ++i)
          qf[ks][i] = pack_f16(__uint_as_float(qf[ks][i] << 16),
                               __uint_as_float(qf[ks][i] & 0xffff0000u));
      }
    }
    have_next = read_piece(pn);
    if (have_next) load_q(pn, qn);
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[C::KS][4];
#pragma unroll
    for (int mt = 0; mt < C::KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int tok0 = p.b0 * B; tok0 < p.tok_end; tok0 += STG, ++stage) {
      // every consumer warp waits on every stage and takes its own tiles of it
      const int slot = stage % NST;
      if (alive && !mbar_wait_bounded(&full[slot], (stage / NST) & 1, kWaitLimitNs)) {
        alive = false;
        if (lane == 0) record_status(a.status, 8);
      }
      alive = __all_sync(0xffffffffu, alive);  // reconverge before ldmatrix / mma.sync
      const int nvalid = p.tok_end - tok0 < STG ? p.tok_end - tok0 : STG;
      const uint32_t kb = k_base + slot * C::STAGE_BYTES;
      const uint32_t vb = v_base + slot * C::STAGE_BYTES;
      if constexpr (F8) {
        // two tiles per pass, tt and tt + WT: their K.Q^T chains, their
        // softmax and their V products interleave, and one running-max
        // update covers both (the second may lie past the context: its
        // scores are masked to -inf and its V rows zeroed)
#pragma unroll 1
        for (int tt = wt; tt < C::TILES; tt += 2 * WT) {
          if (tt * 16 >= nvalid) break;
          int rlo[2], rhi[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            // rows g and g + 8 of S^T stand for tokens f8_srow(g), f8_srow(g + 8)
            rlo[i] = (tt + i * WT) * 16 + f8_srow(g);
            rhi[i] = (tt + i * WT) * 16 + f8_srow(g + 8);
          }
          // ---- S^T = K . Q^T: codes 16 ks + 4 t .. + 3 of each token row,
          // one 32-bit load each, straight into fp16; two chains per tile
          float s[2][4], s2[2][4];
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = s2[i][j] = 0.f;
          // Q8: one accumulator per 32-dimension group (k-steps 2 grp and
          // 2 grp + 1: the dimension permutation stays inside a k-step), each
          // weighted by its rows' K scales afterwards
          float sg[2][Q8 ? 4 : 1][4];
          if constexpr (Q8) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
              for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < 4; ++j) sg[i][q][j] = 0.f;
          }
#pragma unroll
          for (int ks = 0; ks < C::KS; ++ks) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              uint32_t wa, wb, a0, a1, a2, a3;
              asm volatile("ld.shared.b32 %0, [%1];"
                           : "=r"(wa)
                           : "r"(kb + rlo[i] * 128 + t * 4 +
                                 (static_cast<uint32_t>(ks ^ (rlo[i] & 7)) << 4)));
              asm volatile("ld.shared.b32 %0, [%1];"
                           : "=r"(wb)
                           : "r"(kb + rhi[i] * 128 + t * 4 +
                                 (static_cast<uint32_t>(ks ^ (rhi[i] & 7)) << 4)));
              if constexpr (Q8) {
                i8x4_to_f16(wa, a0, a2);
                i8x4_to_f16(wb, a1, a3);
                mma_f16(sg[i][Q8 ? ks >> 1 : 0], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
              } else {
                e4m3x4_to_f16(wa, a0, a2);
                e4m3x4_to_f16(wb, a1, a3);
                if (ks & 1)
                  mma_f16(s2[i], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                else
                  mma_f16(s[i], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
              }
            }
          }
          if constexpr (Q8) {
            // rows rlo / rhi: their four K scales (fp16) side by side
            const uint32_t kscb = smem_u32(sc_st) + slot * C::SC_BYTES;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              uint32_t l0, l1, h0, h1;
              asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                           : "=r"(l0), "=r"(l1)
                           : "r"(kscb + rlo[i] * 8));
              asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                           : "=r"(h0), "=r"(h1)
                           : "r"(kscb + rhi[i] * 8));
              const float kl[4] = {half_lo(l0), half_hi(l0), half_lo(l1), half_hi(l1)};
              const float kh[4] = {half_lo(h0), half_hi(h0), half_lo(h1), half_hi(h1)};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                s[i][0] = fmaf(kl[q], sg[i][Q8 ? q : 0][0], s[i][0]);
                s[i][1] = fmaf(kl[q], sg[i][Q8 ? q : 0][1], s[i][1]);
                s[i][2] = fmaf(kh[q], sg[i][Q8 ? q : 0][2], s[i][2]);
                s[i][3] = fmaf(kh[q], sg[i][Q8 ? q : 0][3], s[i][3]);
              }
            }
          }
          // ---- scale, mask, max over both tiles per column
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const bool v0 = rlo[i] < nvalid, v1 = rhi[i] < nvalid;
            s[i][0] = v0 ? (s[i][0] + s2[i][0]) * a.qscale : -INFINITY;
            s[i][1] = v0 ? (s[i][1] + s2[i][1]) * a.qscale : -INFINITY;
            s[i][2] = v1 ? (s[i][2] + s2[i][2]) * a.qscale : -INFINITY;
            s[i][3] = v1 ? (s[i][3] + s2[i][3]) * a.qscale : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(s[i][0], s[i][2]));
            mx1 = fmaxf(mx1, fmaxf(s[i][1], s[i][3]));
          }
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
          const float al0 = exp2_approx(m_run[0] - mn0), al1 = exp2_approx(m_run[1] - mn1);
          m_run[0] = mn0;
          m_run[1] = mn1;
          // ---- P^T fragments (P <= 1 in fp16: 11 bits, far inside the
          // tolerance), transposed
          // Q8: per 32-dimension group, P times its rows' V scales (a row
          // past the context takes 0, whatever its scale bytes hold)
          uint32_t bh[2][Q8 ? 4 : 1][2];
          float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float p0 = exp2_approx(s[i][0] - mn0), p1 = exp2_approx(s[i][1] - mn1);
            const float p2 = exp2_approx(s[i][2] - mn0), p3 = exp2_approx(s[i][3] - mn1);
            ls0 += p0 + p2;
            ls1 += p1 + p3;
            if constexpr (Q8) {
              const uint32_t vscb = smem_u32(sc_st) + (NST + slot) * C::SC_BYTES;
              uint32_t l0, l1, h0, h1;
              asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                           : "=r"(l0), "=r"(l1)
                           : "r"(vscb + rlo[i] * 8));
              asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                           : "=r"(h0), "=r"(h1)
                           : "r"(vscb + rhi[i] * 8));
              const bool okl = rlo[i] < nvalid, okh = rhi[i] < nvalid;
              const float vl[4] = {half_lo(l0), half_hi(l0), half_lo(l1), half_hi(l1)};
              const float vh[4] = {half_lo(h0), half_hi(h0), half_lo(h1), half_hi(h1)};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float fl = okl ? vl[q] : 0.f, fh = okh ? vh[q] : 0.f;
                bh[i][Q8 ? q : 0][0] = movm_t(pack_f16(p0 * fl, p1 * fl));
                bh[i][Q8 ? q : 0][1] = movm_t(pack_f16(p2 * fh, p3 * fh));
              }
            } else {
              bh[i][0][0] = movm_t(pack_f16(p0, p1));
              bh[i][0][1] = movm_t(pack_f16(p2, p3));
            }
          }
          l_run[0] = l_run[0] * al0 + ls0;
          l_run[1] = l_run[1] * al1 + ls1;
          if (__any_sync(0xffffffffu, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
            for (int mt = 0; mt < C::KS; ++mt) {
              o[mt][0] *= al0;
              o[mt][1] *= al1;
              o[mt][2] *= al0;
              o[mt][3] *= al1;
            }
          }
          // ---- V^T fragments straight from the codes: one 8-bit transposing
          // load per tile and m-tile (16 dimensions = one 16-byte chunk of the
          // 16 token rows, 128-byte swizzle; lane i addresses row f8_vrow(i))
          // gives lane (g, t) tokens f8_vrow(4t .. 4t + 3) = f8_srow of its
          // k-slots, dimensions g and g + 8, converted exactly to fp16;
          // tokens past the context are zeroed (unused slots may hold NaN
          // codes, and 0 * NaN would reach the sum)
          uint32_t vrow[2], vsw[2], mlo[2], mhi[2];
          const int tk0 = 2 * t, tk2 = f8_srow(2 * t + 8), tk3 = f8_srow(2 * t + 9);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int vr = (tt + i * WT) * 16 + f8_vrow(lane & 15);
            const int nv = nvalid - (tt + i * WT) * 16;
            vrow[i] = vb + vr * 128;
            vsw[i] = vr & 7;
            mlo[i] = (tk0 < nv ? 0x0000ffffu : 0u) | (tk0 + 1 < nv ? 0xffff0000u : 0u);
            mhi[i] = (tk2 < nv ? 0x0000ffffu : 0u) | (tk3 < nv ? 0xffff0000u : 0u);
          }
#pragma unroll
          for (int mt = 0; mt < C::KS; ++mt) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              uint32_t r0, r1, a0, a1, a2, a3;
              ldsm8_t(vrow[i] + ((static_cast<uint32_t>(mt) ^ vsw[i]) << 4), r0, r1);
              if constexpr (Q8) {
                i8x4_to_f16(r0, a0, a2);
                i8x4_to_f16(r1, a1, a3);
              } else {
                e4m3x4_to_f16(r0, a0, a2);
                e4m3x4_to_f16(r1, a1, a3);
              }
              const int q = Q8 ? (mt >> 1) : 0;  // Q8: the m-tile's 32-dimension group
              mma_f16(o[mt], a0 & mlo[i], a1 & mlo[i], a2 & mhi[i], a3 & mhi[i], bh[i][q][0],
                      bh[i][q][1]);
            }
          }
        }
      } else {
#pragma unroll 1
      for (int tt = wt; tt < C::TILES; tt += WT) {
        if (tt * 16 >= nvalid) break;
        // ---- S^T = K . Q^T (two independent accumulator chains)
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int r = tt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int ks = 0; ks < C::KS; ++ks) {
            const int d0 = ks * 16 + (lane >> 4) * 8;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(swz(kb + (d0 >> 6) * C::HALF_BYTES, r, (d0 & 63) >> 3), a0, a1, a2, a3);
            if (ks & 1)
              mma_bf16(s2, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            else
              mma_bf16(s, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] += s2[i];
        // ---- scale, mask, tile max per column (columns 2t, 2t+1; tokens g, g+8)
        const int row0 = tt * 16 + g;
        const bool v0 = row0 < nvalid, v1 = row0 + 8 < nvalid;
        s[0] = v0 ? s[0] * a.qscale : -INFINITY;
        s[1] = v0 ? s[1] * a.qscale : -INFINITY;
        s[2] = v1 ? s[2] * a.qscale : -INFINITY;
        s[3] = v1 ? s[3] * a.qscale : -INFINITY;
        float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
        const float al0 = exp2_approx(m_run[0] - mn0), al1 = exp2_approx(m_run[1] - mn1);
        m_run[0] = mn0;
        m_run[1] = mn1;
        const float p0 = exp2_approx(s[0] - mn0), p1 = exp2_approx(s[1] - mn1);
        const float p2 = exp2_approx(s[2] - mn0), p3 = exp2_approx(s[3] - mn1);
        l_run[0] = l_run[0] * al0 + (p0 + p2);
        l_run[1] = l_run[1] * al1 + (p1 + p3);
        // ---- P^T fragments, transposed: bf16 high part and remainder (P
        // keeps ~16 mantissa bits)
        const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
        const uint32_t l01 = pack_bf16(p0 - __uint_as_float(h01 << 16),
                                       p1 - __uint_as_float(h01 & 0xffff0000u));
        const uint32_t l23 = pack_bf16(p2 - __uint_as_float(h23 << 16),
                                       p3 - __uint_as_float(h23 & 0xffff0000u));
        const uint32_t bh0 = movm_t(h01), bh1 = movm_t(h23);
        const uint32_t bl0 = movm_t(l01), bl1 = movm_t(l23);
        // ---- rescale O^T (columns 2t, 2t+1) and accumulate V^T . P^T.  In a
        // partial tile the rows past the context hold whatever the pool held
        // there (possibly NaN bit patterns): their V^T elements are zeroed,
        // since 0 * NaN would reach the sum even with P = 0.
        // The rescale is skipped when no running max of the warp moved (alpha
        // is then exactly 1), which is the common case once the max settles.
        if (__any_sync(0xffffffffu, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
          for (int mt = 0; mt < C::KS; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
          }
        }
        const int nv = nvalid - tt * 16;
        const int r = tt * 16 + (lane & 7) + (lane >> 4) * 8;
        constexpr int hb = C::HALF_BYTES;
        if (nv >= 16) {
#pragma unroll
          for (int mt = 0; mt < C::KS; ++mt) {
            const int d0 = mt * 16 + ((lane >> 3) & 1) * 8;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(swz(vb + (d0 >> 6) * hb, r, (d0 & 63) >> 3), a0, a1, a2, a3);
            mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
            mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
          }
        } else {
          const uint32_t mlo =
              (2 * t < nv ? 0x0000ffffu : 0u) | (2 * t + 1 < nv ? 0xffff0000u : 0u);
          const uint32_t mhi =
              (2 * t + 8 < nv ? 0x0000ffffu : 0u) | (2 * t + 9 < nv ? 0xffff0000u : 0u);
#pragma unroll
          for (int mt = 0; mt < C::KS; ++mt) {
            const int d0 = mt * 16 + ((lane >> 3) & 1) * 8;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(swz(vb + (d0 >> 6) * hb, r, (d0 & 63) >> 3), a0, a1, a2, a3);
            a0 &= mlo;
            a1 &= mlo;
            a2 &= mhi;
            a3 &= mhi;
            mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
            mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
          }
        }
      }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    if constexpr (F8) {  // V codes carry x / v_scale
#pragma unroll
      for (int mt = 0; mt < C::KS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][i] *= a.vscale;
    }
    // ---- combine the states of the warps that share an n-tile
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
      l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
    }
    if (g == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        cmb_ml[(warp * 8 + 2 * t + k) * 2] = m_run[k];
        cmb_ml[(warp * 8 + 2 * t + k) * 2 + 1] = l_run[k];
      }
    }
    const long long slot_id = (long long)blockIdx.x + p.seg;
    if (WT == 1) {
      // one warp per n-tile: its state is already the piece's; each pass
      // hands its CC columns (contiguous in the workspace) to a bulk copy
      // instead of storing them through the registers
      for (int pc = 0; pc < 8; pc += C::CC) {
        const int col0 = warp * 8 + pc;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int c8 = 2 * t + k;
          if (c8 >= pc && c8 < pc + C::CC) {
#pragma unroll
            for (int mt = 0; mt < C::KS; ++mt) {
              cmb_o[(warp * C::CC + c8 - pc) * D + mt * 16 + g] = o[mt][k];
              cmb_o[(warp * C::CC + c8 - pc) * D + mt * 16 + g + 8] = o[mt][2 + k];
            }
            if (g == 0 && col0 + c8 - pc < p.ncols) {
              a.ws_ml[(slot_id * cstride + col0 + c8 - pc) * 2] = m_run[k];
              a.ws_ml[(slot_id * cstride + col0 + c8 - pc) * 2 + 1] = l_run[k];
            }
          }
        }
        fence_async_smem();
        __syncwarp();
        const int cnt = p.ncols - col0 < C::CC ? p.ncols - col0 : C::CC;
        if (lane == 0 && cnt > 0) {
          bulk_store(&a.ws_o[(slot_id * cstride + col0) * D], cmb_o + warp * C::CC * D,
                     static_cast<uint32_t>(cnt) * D * 4);
          bulk_commit();
          bulk_wait_read();
        }
        __syncwarp();
      }
      continue;
    }
    for (int pc = 0; pc < 8; pc += C::CC) {
      if (pc >= p.ncols) break;  // no column of any n-tile in this pass
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c8 = 2 * t + k;
        if (c8 >= pc && c8 < pc + C::CC) {
#pragma unroll
          for (int mt = 0; mt < C::KS; ++mt) {
            cmb_o[(warp * C::CC + c8 - pc) * D + mt * 16 + g] = o[mt][k];
            cmb_o[(warp * C::CC + c8 - pc) * D + mt * 16 + g + 8] = o[mt][2 + k];
          }
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
      // four consecutive dimensions per thread and one 16-byte store: the
      // stores of a piece's partials compete with the stream of K/V loads
      // for the memory system, so their count matters more than their size
      constexpr int D4 = D / 4;
      for (int idx = threadIdx.x; idx < NT * C::CC * D4; idx += kConsumerWarps * 32) {
        const int wni = idx / (C::CC * D4);
        const int rem = idx - wni * C::CC * D4;
        const int cc = rem / D4, d = (rem - cc * D4) * 4;
        const int col = wni * 8 + pc + cc;
        if (col >= p.ncols) continue;
        float M = -INFINITY;
        for (int j = 0; j < WT; ++j) M = fmaxf(M, cmb_ml[((wni + j * NT) * 8 + pc + cc) * 2]);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < WT; ++j) {
          const int w = wni + j * NT;
          const float mw = cmb_ml[(w * 8 + pc + cc) * 2];
          const float f = mw == -INFINITY ? 0.f : exp2_approx(mw - M);
          L += f * cmb_ml[(w * 8 + pc + cc) * 2 + 1];
          const float4 v = *reinterpret_cast<const float4*>(&cmb_o[(w * C::CC + cc) * D + d]);
          O.x += f * v.x;
          O.y += f * v.y;
          O.z += f * v.z;
          O.w += f * v.w;
        }
        *reinterpret_cast<float4*>(&a.ws_o[(slot_id * cstride + col) * D + d]) = O;
        if (d == 0) {
          a.ws_ml[(slot_id * cstride + col) * 2] = M;
          a.ws_ml[(slot_id * cstride + col) * 2 + 1] = L;
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
    }
  }
  if (lane == 0) bulk_wait_all();  // partials handed to bulk copies have landed
}

}  // namespace pkv
