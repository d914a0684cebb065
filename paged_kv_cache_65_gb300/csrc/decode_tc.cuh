// Split-K paged decode attention, partial pass, on the fifth-generation
// tensor cores (tcgen05) with accumulators in tensor memory (TMEM).
//
// Same contract, work split, pieces and workspace as decode_mma.cuh: per
// piece (a block range of one segment) it writes the base-2 online-softmax
// statistics m, l and the unnormalised O of each of the segment's query
// columns ("PagedAttention 的块表与碎片控制" §07 for the attention, "KV 缓存管理"
// chunked-prefill section for the split and merge rule).  bfloat16 or FP8
// (E4M3) K/V, D_h = 128, B a multiple of 8 with whole 64-row boxes per block.
//
// Per stage of 128 token rows of one K/V head:
//     S^T [128 tokens x N] = K [128 x 128] . Q^T [128 x N]          (8 MMAs, K = 16)
//     O^T [128 dims  x 64] += V^T [128 x 128] . [P_hi | P_lo]^T      (8 MMAs)
// N = 16 for pieces with up to 16 query columns, 32 otherwise (the softmax
// handles 8, 16 or 32 columns).  K, V and Q
// are read by the tensor core straight from shared memory (K and Q
// K-major, V^T M-major, all with the 128-byte swizzle the TMA wrote); P is
// written by the softmax warps into the stage's K area, which the S MMA has
// finished with, N-major with the 128-byte swizzle: a bf16 high part in
// columns 0-31 and the bf16 remainder in columns 32-63, so the weights keep
// ~16 mantissa bits and one N = 64 MMA per 16 tokens accumulates both (O^T
// holds the two sums side by side; the readout adds them).  S^T (two
// buffers) and O^T live in TMEM: row r of a 128-row tile is TMEM lane r.
//
// Warp roles (one CTA per SM): warps 0-3 are the softmax warps (thread r owns
// token row r of S^T and, at the end of a piece, dimension r of O^T), warps
// 4 and 5 issue the TMA loads of K and of V (issuing a tensor copy costs the
// issuing warp tens of cycles, so one warp alone cannot keep up with HBM at
// 16-row boxes), warp 4 also stages each piece's Q tile (three buffers, so
// the next pieces' S can start while the current one finishes), lane 0 of
// warp 6 issues the S MMAs and lane 0 of warp 7 the P.V MMAs.  Issuing one
// of these small MMAs costs the issuing thread tens of cycles, so one thread
// issuing both would hold the next stage's S back behind this stage's P.V;
// with two, S of a stage goes out as soon as its K is in and the softmax
// has read the S buffer it overwrites.
// Softmax is
// lazy: the reference max m of a column only moves when a new score exceeds
// it by more than 2^8 (TAU = 8 in base-2 units), so in the steady state a
// stage costs one barrier-reduction to confirm that nothing moved, and the
// weights stay below 2^8.  When m moves, the column maxima of the stage are
// reduced exactly, l is rescaled, and O^T is rescaled in TMEM once the
// previous stage's MMAs have completed.
//
// A parity wait is exact only while the waiter is never two phases ahead of
// the barrier, nor two behind it: each role waits every phase of full,
// s_full, p_full, q_full, q_empty and o_free in order; p_full has one barrier
// per ring slot, so the softmax cannot complete a slot's next phase before
// the P.V issuer has seen this one (that stage's copies wait for its P.V);
// and the MMAs of a stage are awaited through that stage's empty barrier,
// whose phases are NST stages apart.
//
// FP8 (E4M3) pools: the codes take half the bytes, so a stage's converted
// operands must not take the shared memory the copies in flight need.  Four
// converter warps (8-11, a warpgroup of their own; thread r owns token row
// r) turn each stage's codes into fp16: K row r goes to TMEM
// lane r (the S MMA reads K from tensor memory), V row r into the same
// shared-memory layout the bfloat16 pass reads (the V codes land in the
// upper half of that buffer and each row's codes are read before they are
// written over).  A stage then holds 16 KiB of K codes (where the softmax
// later writes P) and 32 KiB of V, four stages in the ring against three.
// Rows past the context become zeros.  E4M3 values convert to fp16 exactly,
// Q is staged as fp16 (exact inside fp16's range), P is split into an fp16
// high part and remainder, and the MMAs run on f16 operands; the K scale is
// folded into the score scale and the V scale into the O readout.  K and V
// copies complete on barriers of their own, and the S MMA waits only for
// the K rows, the P.V MMA for the V rows.  Twelve warps leave 168 registers
// a thread at launch; the converters then give some back and the softmax
// and the producer / MMA warpgroups take them.
//
// Every mbarrier wait is bounded; a wait that gives up records
// KV_DEV_WAIT_TIMEOUT and the role runs the rest of its loops without waiting
// or issuing, so that every named barrier is still reached and the CTA frees
// its TMEM and exits.
#pragma once

#include "decode_mma.cuh"
#include "tc.cuh"

namespace pkv {

// Instruction descriptor of kind::f16 with f16 A and B (format 0 in bits
// 7-9 and 10-12; bf16 is 1, tc.cuh's idesc_bf16), the rest as there.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

constexpr int kTcWarps = 8;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcCvtWarps = 4;  // FP8 converter warps (8-11)
constexpr int kTcCvtWarp0 = 8;
// FP8 register split per warpgroup: softmax, producers and MMA, converters,
// against the 168 a thread that twelve warps are launched with (the launcher
// checks that count)
constexpr int kTcRegsLaunchF8 = 168;
constexpr int kTcRegsSoftmax = 232, kTcRegsHelper = 176, kTcRegsCvt = 96;
static_assert(128 * (kTcRegsSoftmax + kTcRegsHelper + kTcRegsCvt) <= kTcRegsLaunchF8 * 12 * 32,
              "register split within the launch's registers");

// A warpgroup's register count moved from the launch count to N: raised
// (setmaxnreg.inc) or lowered (setmaxnreg.dec), never the other way round.
template <int N>
__device__ __forceinline__ void tc_regs_f8() {
  if constexpr (N > kTcRegsLaunchF8)
    reg_alloc<N>();
  else if constexpr (N < kTcRegsLaunchF8)
    reg_dealloc<N>();
}

template <bool F8>
constexpr int tc_threads() {
  return F8 ? (kTcCvtWarp0 + kTcCvtWarps) * 32 : kTcThreads;
}

struct TcCfg {
  static constexpr int D = 128;
  static constexpr int TS = 128;            // token rows per stage (M of the S MMA)
  static constexpr int HALF = TS * 128;     // one 64-element half of K (or V): 16 KiB
  static constexpr int STAGE = 2 * HALF;    // K (or V) of one stage: 32 KiB
  static constexpr int NST = 3;             // stages in the ring
  static constexpr int QHALF = 32 * 128;    // one half of a Q tile: 4 KiB
  static constexpr int QTILE = 2 * QHALF;   // Q tile: 32 columns x 128 dims
  static constexpr int QBUF = 3;            // Q tiles in flight
  static constexpr int TM_S = 0;            // TMEM columns: S^T buffers at 0 and 32,
  static constexpr int TM_O = 64;           // O^T: high-part sums at 64, remainder at 96
  static constexpr int TM_COLS = 128;
  static constexpr float TAU = 8.f;
  // FP8: four stages of K codes (16 KiB) and fp16 V (32 KiB); K tiles in
  // TMEM after S and O, 64 columns (128 fp16) a stage
  static constexpr int NST_F8 = 4;
  static constexpr int TM_K = 128;
  static constexpr int TM_COLS_F8 = 512;
  static constexpr int NBARS = 40;          // mbarrier slots (the FP8 pass uses 32)
};
static_assert(TcCfg::TM_K + TcCfg::NST_F8 * 64 <= TcCfg::TM_COLS_F8, "TMEM columns");

// Ring depth and shared-memory bytes of a stage's K buffer for each pass.
template <bool F8>
constexpr int tc_stages() {
  return F8 ? TcCfg::NST_F8 : TcCfg::NST;
}
template <bool F8>
constexpr int tc_k_stage_bytes() {
  return F8 ? TcCfg::HALF : TcCfg::STAGE;
}

template <bool F8>
constexpr int decode_tc_smem_bytes() {
  return tc_stages<F8>() * (tc_k_stage_bytes<F8>() + TcCfg::STAGE)  // K, V stages
         + TcCfg::QBUF * TcCfg::QTILE   // Q tiles
         + 3 * 4 * 32 * 4               // column maxima, per-warp broadcast, l sums
         + TcCfg::NBARS * 8             // mbarriers
         + 4 * 8 + 16                   // walk state, TMEM address
         + 2 * kTableCache * 4          // producer table caches
         + 128                          // start record
         + 1024;                        // alignment
}

// Barrier over the 128 softmax threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_or_sync(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 32)
    tmem_ld32(taddr, r);
  else if constexpr (N == 16)
    tmem_ld16(taddr, r);
  else
    tmem_ld8(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 32)
    tmem_st32(taddr, r);
  else if constexpr (N == 16)
    tmem_st16(taddr, r);
  else
    tmem_st8(taddr, r);
}

// Column reduction across a warp: lane i holds v[0..N) (one row per lane);
// returns the reduction over the 32 rows of column (lane mod N).  Halving
// exchange (N - 1 shuffles), then folds over the lanes holding the same
// column (32 / N - 1 more).
template <int N, bool MAX>
__device__ __forceinline__ float warp_column_reduce(float (&v)[N]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int off = N; off < 32; off <<= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, r, off);
    r = MAX ? fmaxf(r, o) : r + o;
  }
  return r;
}

// Shared state of the softmax warps for one CTA.
struct TcSoftmax {
  const DecodeArgs* a;
  unsigned char* k_st;
  unsigned char* v_st;
  float* red;   // [4][32] column maxima per warp
  float* cmx;   // [4][32] per-warp broadcast of the stage maxima
  float* lsum;  // [4][32] column sums of l per warp (end of a piece)
  uint64_t *full, *empty, *s_full, *p_full, *o_free;
  uint32_t tmem;
  int B, cstride;
  bool alive;
  int stage;

  __device__ bool wait(uint64_t* bar, uint32_t parity) {
    if (alive && !mbar_wait_bounded(bar, parity, kWaitLimitNs)) {
      alive = false;
      record_status(a->status, 8);
    }
    return alive;
  }

  // One piece with at least one stage; NCP = 8, 16 or 32 query columns.
  template <int NCP, bool F8>
  __device__ void run(const Piece& p, int n_st) {
    using C = TcCfg;
    constexpr int NST = tc_stages<F8>();
    const int t = threadIdx.x;  // token row of a stage / dimension of O^T
    const int warp = t >> 5, lane = t & 31;
    const uint32_t tl = static_cast<uint32_t>(warp * 32) << 16;
    const int ncols = p.ncols;
    float m_ref[NCP], l_part[NCP];
#pragma unroll
    for (int c = 0; c < NCP; ++c) {
      m_ref[c] = -INFINITY;
      l_part[c] = 0.f;
    }
    const float qs = a->qscale;
    for (int i = 0; i < n_st; ++i, ++stage) {
      const int slot = stage % NST;
      const int tok0 = p.b0 * B + i * C::TS;
      const int nvalid = p.tok_end - tok0 < C::TS ? p.tok_end - tok0 : C::TS;
      const bool valid = t < nvalid;
      if constexpr (!F8) wait(&full[slot], (stage / NST) & 1);  // (rows zeroed below)
      wait(&s_full[stage & 1], (stage >> 1) & 1);
      __syncwarp();
      tc_fence_after();
      uint32_t sr[NCP];
      tmem_ld<NCP>(tmem + C::TM_S + (stage & 1) * 32 + tl, sr);
      float x[NCP];
      bool exceed = false;
#pragma unroll
      for (int c = 0; c < NCP; ++c) {
        x[c] = fmaf(__uint_as_float(sr[c]), qs, -m_ref[c]);
        exceed |= x[c] > C::TAU;
      }
      if (bar_or_sync(1, 128, valid && exceed)) {
        // ---- the reference moves: exact column maxima of this stage
        float v[NCP];
#pragma unroll
        for (int c = 0; c < NCP; ++c) v[c] = valid ? __uint_as_float(sr[c]) * qs : -INFINITY;
        const float wm = warp_column_reduce<NCP, true>(v);
        if (lane < NCP) red[warp * 32 + lane] = wm;
        named_bar_sync(1, 128);
        float cm = -INFINITY;
        if (lane < NCP) {
#pragma unroll
          for (int w = 0; w < 4; ++w) cm = fmaxf(cm, red[w * 32 + lane]);
        }
        cmx[warp * 32 + lane] = cm;
        __syncwarp();
        float al[NCP];
#pragma unroll
        for (int c = 0; c < NCP; ++c) {
          const float mn = fmaxf(m_ref[c], cmx[warp * 32 + c]);
          al[c] = exp2_approx(m_ref[c] - mn);
          m_ref[c] = mn;
          l_part[c] *= al[c];
          x[c] = fmaf(__uint_as_float(sr[c]), qs, -mn);
        }
        if (i > 0) {
          // rescale O^T once the previous stage's MMAs are done with it
          // (the stage's empty barrier completes with them; its phases are
          // NST stages apart, so the parity cannot alias)
          wait(&empty[(stage - 1) % NST], ((stage - 1) / NST) & 1);
          __syncwarp();
          tc_fence_after();
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            uint32_t o[NCP];
            tmem_ld<NCP>(tmem + C::TM_O + part * 32 + tl, o);
#pragma unroll
            for (int c = 0; c < NCP; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * al[c]);
            tmem_st<NCP>(tmem + C::TM_O + part * 32 + tl, o);
          }
        }
      }
      // ---- weights: bf16 (F8: fp16) high part (chunks 0-3) and remainder
      // (chunks 4-7) of row t of P (N-major, 128-byte swizzle: chunk c at
      // c ^ (t & 7))
      const uint32_t pb = smem_u32(k_st + slot * tc_k_stage_bytes<F8>());
#pragma unroll
      for (int c8 = 0; c8 < NCP / 8; ++c8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = c8 * 8 + 2 * k;
          const float p0 = valid ? exp2_approx(x[c]) : 0.f;
          const float p1 = valid ? exp2_approx(x[c + 1]) : 0.f;
          l_part[c] += p0;
          l_part[c + 1] += p1;
          if constexpr (F8) {
            hi[k] = pack_f16(p0, p1);
            lo[k] = pack_f16(p0 - half_lo(hi[k]), p1 - half_hi(hi[k]));
          } else {
            hi[k] = pack_bf16(p0, p1);
            lo[k] = pack_bf16(p0 - __uint_as_float(hi[k] << 16),
                              p1 - __uint_as_float(hi[k] & 0xffff0000u));
          }
        }
        sts128(pb + t * 128 + ((c8 ^ (t & 7)) << 4), hi[0], hi[1], hi[2], hi[3]);
        sts128(pb + t * 128 + (((4 + c8) ^ (t & 7)) << 4), lo[0], lo[1], lo[2], lo[3]);
      }
      // rows past the context inside the last 16-row MMA step: V must be
      // finite there (unused slots may hold anything), so it is zeroed (FP8:
      // by the converters)
      if (!F8 && !valid && t < ((nvalid + 15) & ~15)) {
        const uint32_t vb = smem_u32(v_st + slot * C::STAGE) + t * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int k = 0; k < 8; ++k) sts128(vb + h * C::HALF + k * 16, 0u, 0u, 0u, 0u);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[stage % NST]);
    }

    // ---- end of the piece: O^T from TMEM once the last stage's MMAs are
    // done, l reduced over the 128 rows
    wait(&empty[(stage - 1) % NST], ((stage - 1) / NST) & 1);
    __syncwarp();
    tc_fence_after();
    const long long slot_id = (long long)blockIdx.x + p.seg;
#pragma unroll
    for (int c0 = 0; c0 < NCP; c0 += 8) {
      uint32_t oh[8], ol[8];
      tmem_ld8(tmem + C::TM_O + c0 + tl, oh);
      tmem_ld8(tmem + C::TM_O + 32 + c0 + tl, ol);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c0 + c < ncols) {
          float o = __uint_as_float(oh[c]) + __uint_as_float(ol[c]);
          if constexpr (F8) o *= a->vscale;
          a->ws_o[(slot_id * cstride + c0 + c) * C::D + t] = o;
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(o_free);
    const float ls = warp_column_reduce<NCP, false>(l_part);
    if (lane < NCP) lsum[warp * 32 + lane] = ls;
    named_bar_sync(1, 128);
    if (warp == 0 && lane < ncols) {
      float mc = m_ref[0];
#pragma unroll
      for (int c = 1; c < NCP; ++c) mc = lane == c ? m_ref[c] : mc;
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) L += lsum[w * 32 + lane];
      a->ws_ml[(slot_id * cstride + lane) * 2] = mc;
      a->ws_ml[(slot_id * cstride + lane) * 2 + 1] = L;
    }
  }
};

template <bool PLAN, bool F8 = false>
__global__ void __launch_bounds__(tc_threads<F8>(), 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
  using C = TcCfg;
  constexpr int NST = tc_stages<F8>();
  constexpr int KSTAGE = tc_k_stage_bytes<F8>();  // FP8: the K codes, later P
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* k_st = smem;
  unsigned char* v_st = k_st + NST * KSTAGE;
  unsigned char* q_s = v_st + NST * C::STAGE;  // QBUF Q tiles
  float* red = reinterpret_cast<float*>(q_s + C::QBUF * C::QTILE);
  float* cmx = red + 128;
  float* lsum = cmx + 128;
  uint64_t* full = reinterpret_cast<uint64_t*>(lsum + 128);
  uint64_t* empty = full + NST;
  uint64_t* s_full = empty + NST;  // [2]
  uint64_t* p_full = s_full + 2;   // [NST] by ring slot
  uint64_t* q_full = p_full + NST;         // [QBUF]
  uint64_t* q_empty = q_full + C::QBUF;    // [QBUF]
  uint64_t* o_free = q_empty + C::QBUF;
  uint64_t* fin = o_free + 1;
  uint64_t* full_v = fin + 1;     // [NST] F8: the V copies (full: the K copies)
  uint64_t* cvt_k = full_v + NST;  // [NST] F8: K rows in TMEM
  uint64_t* cvt_v = cvt_k + NST;   // [NST] F8: V rows converted in shared memory
  long long* walk = reinterpret_cast<long long*>(full + C::NBARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(walk + 4);
  int32_t* tcache = reinterpret_cast<int32_t*>(tmem_slot + 4);
  PlanStart* rec_s = reinterpret_cast<PlanStart*>(tcache + 2 * kTableCache);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int H = a.n_kv_heads;
  const int G = a.n_q_heads / H;
  // rows per TMA box (a multiple of 8 dividing B and 128); FP8: the code
  // tensor map's box, one 128-byte row of codes wide
  const int UR = F8 ? mma_box_rows(B, C::TS) : (B < 64 ? B : 64);

  // self-check: swizzled buffers must sit on 1 KiB boundaries
  if ((smem_u32(k_st) & 1023u) != 0u) {
    if (threadIdx.x == 0) record_status(a.status, 32);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], F8 ? 1 : 2);  // the K and the V producer (F8: K only)
      mbar_init(&empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    for (int i = 0; i < NST; ++i) mbar_init(&p_full[i], 4);
    for (int i = 0; i < C::QBUF; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(o_free, 4);
    mbar_init(fin, 2);  // both MMA issuers
    if constexpr (F8) {
      for (int i = 0; i < NST; ++i) {
        mbar_init(&full_v[i], 1);
        mbar_init(&cvt_k[i], kTcCvtWarps);
        mbar_init(&cvt_v[i], kTcCvtWarps);
      }
    }
    fence_barrier_init();
  }
  constexpr uint32_t kTmCols = F8 ? C::TM_COLS_F8 : C::TM_COLS;
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmCols);
    tmem_relinquish();
  }
  // The walk start and the producers' first block-table entries read only
  // host-written metadata (plan, context lengths, tables), complete before the
  // first kernel of the stream's programmatic chain started, so they are
  // read before waiting for the previous grid; the pool, q and the workspace
  // only after it.
  // a plan with start records for this grid: the CTA's first piece and its
  // first blocks' ids come with one 128-byte read (no search, no table read)
  const bool use_rec = PLAN && a.starts != nullptr && a.start_grid == a.grid;
  if (warp == 4) {
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

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
  // the first piece of this CTA, without advancing the walk
  auto peek_first = [&](Piece& p0) -> bool {
    const PieceWalker pw_s = pw;
    const PlanWalker plw_s = plw;
    const bool rf = rec_first;
    const bool ok = next_piece(p0);
    pw = pw_s;
    plw = plw_s;
    rec_first = rf;
    return ok;
  };
  auto wait_previous_grid = [&]() {
    griddep_wait();
    griddep_launch_dependents();
    if constexpr (!PLAN) {
      if (blockIdx.x == 0 && warp == 4)
        write_prefix(a.ctx, a.n_seq, B, H, a.max_blocks, a.ws_pre);
    }
  };
  auto stages_of = [&](const Piece& p) -> int {
    const int n = p.tok_end - p.b0 * B;
    return n > 0 ? (n + C::TS - 1) / C::TS : 0;
  };

  if (warp == 4 || warp == 5) {
    // ----------------------------------------------- producers (K, V)
    if constexpr (F8) tc_regs_f8<kTcRegsHelper>();
    const bool kp = warp == 4;  // K producer, also stages Q
    const CUtensorMap* tmap = kp ? &tmap_k : &tmap_v;
    unsigned char* dst_st = kp ? k_st : v_st;
    if (lane == 0) prefetch_tmap(tmap);
    bool alive = true;
    int stage = 0, npiece = 0;
    TableCache tc;
    tc.ent = tcache + (warp - 4) * kTableCache;
    if (!use_rec) {
      Piece p0;
      if (peek_first(p0)) tc.ensure(a.table, a.max_blocks, p0.rep, p0.b0, p0.b0, lane);
    }
    wait_previous_grid();
    // Q tile of a piece: row c = query column c (zero past the piece's
    // columns), 128 dims, K-major, 128-byte swizzle.  Lane l holds the
    // 16-byte chunks l, l + 32, ... of the tile; the loads for the next piece
    // are issued before the current piece's copies, so their latency is
    // hidden behind them.
    uint4 qv[16];
    auto load_q = [&](const Piece& x) {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int idx = k * 32 + lane;
        const int col = idx >> 4, cg = idx & 15;
        qv[k] = make_uint4(0, 0, 0, 0);
        if (col < x.ncols) {
          int seqm = x.rep, gi = col;
          if constexpr (PLAN) {
            const int mi = col / G;
            gi = col - mi * G;
            seqm = a.members[x.mem + mi];
          }
          qv[k] = *reinterpret_cast<const uint4*>(
              reinterpret_cast<const unsigned char*>(a.q) +
              (((long long)seqm * a.n_q_heads + (long long)x.head * G + gi) * C::D + cg * 8) * 2);
        }
      }
    };
    auto next_nonempty = [&](Piece& x) {
      while (next_piece(x))
        if (stages_of(x) > 0) return true;
      return false;
    };
    // Q tile of piece number np into its buffer, once the S MMAs of the
    // piece QBUF before are done with that buffer
    auto stage_q = [&](int np) {
      const int qb = np % C::QBUF;
      if (kp && np >= C::QBUF && alive) {
        if (!mbar_wait_bounded(&q_empty[qb], ((np / C::QBUF) - 1) & 1, kWaitLimitNs)) {
          alive = false;
          if (lane == 0) record_status(a.status, 8);
        }
      }
      alive = __all_sync(0xffffffffu, alive);
      if (kp && alive) {
        const uint32_t qs = smem_u32(q_s + qb * C::QTILE);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int idx = k * 32 + lane;
          const int col = idx >> 4, cg = idx & 15;
          const int h = cg >> 3, c = cg & 7;
          uint4 w = qv[k];
          if constexpr (F8) {  // bf16 -> fp16 pairs
            w.x = pack_f16(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
            w.y = pack_f16(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
            w.z = pack_f16(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
            w.w = pack_f16(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
          }
          sts128(qs + h * C::QHALF + col * 128 + ((c ^ (col & 7)) << 4), w.x, w.y, w.z, w.w);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[qb]);
      }
    };
    Piece p, pn;
    bool have = next_nonempty(p);
    if (have && kp) load_q(p);
    while (have) {
      const int n_st = stages_of(p);
      bool have_next = false;
      for (int i = 0; i < n_st; ++i, ++stage) {
        const int slot = stage % NST;
        if (stage >= NST && alive) {
          if (!mbar_wait_bounded(&empty[slot], ((stage / NST) & 1) ^ 1, kWaitLimitNs)) {
            alive = false;
            if (lane == 0) record_status(a.status, 8);
          }
        }
        alive = __all_sync(0xffffffffu, alive);
        if (!alive) continue;
        const int tok0 = p.b0 * B + i * C::TS;
        const int nvalid = p.tok_end - tok0 < C::TS ? p.tok_end - tok0 : C::TS;
        const int nunits = (nvalid + UR - 1) / UR;
        const int jl = (tok0 + (nunits - 1) * UR) / B;
        // the first stage of the record's piece takes the record's block ids
        const bool from_rec = use_rec && stage == 0 && p.seg == rec_s->seg &&
                              tok0 / B >= rec_s->b0 && jl - rec_s->b0 < rec_s->n_pid;
        if (!from_rec) tc.ensure(a.table, a.max_blocks, p.rep, tok0 / B, jl, lane);
        if constexpr (PLAN) {
          // fused slot write: the stage holding a private segment's last
          // token (the sequence's newest) writes that row first, K by the K
          // producer and V by the V producer
          if (a.k_new != nullptr && p.last && p.ncols == G && tok0 + C::TS >= p.tok_end) {
            const int t = p.tok_end - 1;
            const int j = t / B;
            const int pid = from_rec ? rec_s->pid[j - rec_s->b0] : tc.ent[j - tc.base];
            if (pid >= 0 && pid < a.n_blocks)
              write_new_row<C::D, F8>(a, p.rep, p.head, pid, t - j * B, kp, !kp, lane);
          }
        }
        uint64_t* landed = F8 && !kp ? &full_v[slot] : &full[slot];
        if (lane == 0) mbar_arrive_expect_tx(landed, 1u * nunits * UR * C::D * (F8 ? 1 : 2));
        __syncwarp();
        for (int u = lane; u < nunits; u += 32) {
          const int tk = tok0 + u * UR;
          const int j = tk / B;
          const int row = tk - j * B;
          int pid = from_rec ? rec_s->pid[j - rec_s->b0] : tc.ent[j - tc.base];
          if (pid < 0 || pid >= a.n_blocks) {
            record_status(a.status, 1);
            pid = 0;  // stay in bounds; the result is flagged as invalid
          }
          const int y = (a.layer * a.n_blocks + pid) * B + row;
          if constexpr (F8) {
            // the codes of UR rows: K at the start of its 16 KiB buffer, V
            // into the upper half of its fp16 buffer
            tma_load_2d(dst_st + slot * (kp ? KSTAGE : C::STAGE) + (kp ? 0 : C::HALF) + u * UR * 128,
                        tmap, p.head * C::D, y, landed);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int x = p.head * C::D + h * 64;
              const int off = slot * C::STAGE + h * C::HALF + u * UR * 128;
              tma_load_2d(dst_st + off, tmap, x, y, &full[slot]);
            }
          }
        }
        if (i == 0) {
          // the piece's Q goes in behind its first copies (their latency
          // covers it), then the next piece's Q loads are issued
          stage_q(npiece);
          have_next = next_nonempty(pn);
          if (have_next && kp) load_q(pn);
        }
      }
      ++npiece;  // (after a failed wait the walk stops here: have_next stays false)
      p = pn;
      have = have_next;
    }
    // copies still in flight land before the CTA may exit
    const int first = stage > NST ? stage - NST : 0;
    uint64_t* landed = F8 && !kp ? full_v : full;
    for (int k = first; k < stage && alive; ++k)
      alive = mbar_wait_bounded(&landed[k % NST], (k / NST) & 1, kWaitLimitNs);
  } else if (warp == 6 || warp == 7) {
    // ------------------------------------- MMA issuers: 6 for S, 7 for P.V
    if constexpr (F8) tc_regs_f8<kTcRegsHelper>();
    wait_previous_grid();
    if (lane == 0) {
      const uint32_t kb = smem_u32(k_st), vb = smem_u32(v_st), qb = smem_u32(q_s);
      bool alive = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (alive && !mbar_wait_bounded(bar, parity, kWaitLimitNs)) {
          alive = false;
          record_status(a.status, 8);
        }
        return alive;
      };
      int stage = 0, npiece = 0;
      Piece p;
      if (warp == 6) {
        // S^T of each stage as soon as its K is in and its TMEM buffer has
        // been read (P of the stage two before is written)
        constexpr uint32_t idS16 =
            F8 ? idesc_f16(128, 16, false, false) : idesc_bf16(128, 16, false, false);
        constexpr uint32_t idS32 =
            F8 ? idesc_f16(128, 32, false, false) : idesc_bf16(128, 32, false, false);
        uint64_t* ready = F8 ? cvt_k : full;  // a stage's K is in shared memory (F8: TMEM)
        while (next_piece(p)) {
          const int n_st = stages_of(p);
          if (n_st == 0) continue;
          const uint32_t idS = p.ncols <= 16 ? idS16 : idS32;
          const int qbi = npiece % C::QBUF;
          const uint32_t qbase = qb + qbi * C::QTILE;
          wait(&q_full[qbi], (npiece / C::QBUF) & 1);
          for (int i = 0; i < n_st; ++i) {
            const int st = stage + i;
            if (st >= 2) wait(&p_full[(st - 2) % NST], ((st - 2) / NST) & 1);
            wait(&ready[st % NST], (st / NST) & 1);
            if (!alive) continue;
            tc_fence_after();
            const uint32_t ks = kb + (st % NST) * KSTAGE;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t off = (k >> 2) * C::HALF + (k & 3) * 32;
              const uint32_t qoff = (k >> 2) * C::QHALF + (k & 3) * 32;
              const uint64_t qd = smem_desc(qbase + qoff, 16, 1024, kSwizzle128);
              if constexpr (F8)  // K rows in TMEM: 8 columns (16 fp16) a k-step
                tc_mma_ts(tmem + C::TM_S + (st & 1) * 32, tmem + C::TM_K + (st % NST) * 64 + k * 8,
                          qd, idS, k > 0);
              else
                tc_mma(tmem + C::TM_S + (st & 1) * 32, smem_desc(ks + off, 16, 1024, kSwizzle128),
                       qd, idS, k > 0);
            }
            tc_commit(&s_full[st & 1]);
          }
          tc_commit(&q_empty[qbi]);  // the Q tile is free once these are done
          stage += n_st;
          ++npiece;
        }
      } else {
        // O^T += V^T . [P_hi | P_lo]^T of each stage once P is written (F8:
        // and its V rows converted); a piece's first stage starts O^T anew
        // once the previous piece's O^T has been read out
        constexpr uint32_t idPV =
            F8 ? idesc_f16(128, 64, true, true) : idesc_bf16(128, 64, true, true);
        while (next_piece(p)) {
          const int n_st = stages_of(p);
          if (n_st == 0) continue;
          if (npiece > 0) wait(o_free, (npiece - 1) & 1);
          for (int i = 0; i < n_st; ++i) {
            const int cur = stage + i;
            wait(&p_full[cur % NST], (cur / NST) & 1);
            if constexpr (F8) wait(&cvt_v[cur % NST], (cur / NST) & 1);
            if (!alive) continue;
            tc_fence_after();
            const int tok0 = p.b0 * B + i * C::TS;
            const int nvalid = p.tok_end - tok0 < C::TS ? p.tok_end - tok0 : C::TS;
            const int nk = (nvalid + 15) >> 4;
            const uint32_t vs = vb + (cur % NST) * C::STAGE;
            const uint32_t ps = kb + (cur % NST) * KSTAGE;
            for (int k = 0; k < nk; ++k)
              tc_mma(tmem + C::TM_O, smem_desc(vs + k * 2048, C::HALF, 1024, kSwizzle128),
                     smem_desc(ps + k * 2048, C::HALF, 1024, kSwizzle128), idPV,
                     (i > 0 || k > 0) ? 1u : 0u);
            tc_commit(&empty[cur % NST]);
          }
          stage += n_st;
          ++npiece;
        }
      }
      // every MMA either thread issued has completed before TMEM is released
      tc_commit(fin);
      mbar_wait_bounded(fin, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp >= kTcCvtWarp0) {
    // ------------------------------------------------ FP8 converters (8-11)
    if constexpr (F8) {
      tc_regs_f8<kTcRegsCvt>();
      wait_previous_grid();
      const int r = threadIdx.x - kTcCvtWarp0 * 32;  // token row of a stage
      bool alive = true;
      int stage = 0;
      // row r of a stage's V: its 128 codes (upper half, 128-byte swizzle)
      // read whole, then written as 128 fp16 values over both halves
      auto convert_v = [&](unsigned char* st, bool valid) {
        const uint32_t b = smem_u32(st);
        uint32_t w[8][4];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          w[c][0] = w[c][1] = w[c][2] = w[c][3] = 0u;
          if (valid)
            lds128(b + C::HALF + r * 128 + ((c ^ (r & 7)) << 4), w[c][0], w[c][1], w[c][2],
                   w[c][3]);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t h[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) e4m3x4_to_f16(w[c][k], h[2 * k], h[2 * k + 1]);
          // codes 16c .. 16c + 15: half c / 4, 16-byte chunks 2 (c % 4) and + 1
          const uint32_t row = b + (c >> 2) * C::HALF + r * 128;
          const int cc = (c & 3) * 2;
          sts128(row + ((cc ^ (r & 7)) << 4), h[0], h[1], h[2], h[3]);
          sts128(row + (((cc + 1) ^ (r & 7)) << 4), h[4], h[5], h[6], h[7]);
        }
      };
      // row r of a stage's K: its codes (128-byte swizzle) as 64 fp16 pairs
      // into TMEM lane r, dimensions 2j and 2j + 1 in column j
      const uint32_t tl = static_cast<uint32_t>((warp & 3) * 32) << 16;
      auto convert_k = [&](unsigned char* st, uint32_t tcol, bool valid) {
        const uint32_t b = smem_u32(st);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t w[4][4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            w[c][0] = w[c][1] = w[c][2] = w[c][3] = 0u;
            if (valid)
              lds128(b + r * 128 + (((4 * hf + c) ^ (r & 7)) << 4), w[c][0], w[c][1], w[c][2],
                     w[c][3]);
          }
          uint32_t h[32];
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              e4m3x4_to_f16(w[c][k], h[8 * c + 2 * k], h[8 * c + 2 * k + 1]);
          __syncwarp();
          tmem_st32(tmem + tl + tcol + hf * 32, h);
        }
      };
      Piece p;
      while (next_piece(p)) {
        const int n_st = stages_of(p);
        for (int i = 0; i < n_st; ++i, ++stage) {
          const int slot = stage % NST;
          const uint32_t par = (stage / NST) & 1;
          if (alive && !mbar_wait_bounded(&full[slot], par, kWaitLimitNs)) {
            alive = false;
            record_status(a.status, 8);
          }
          alive = __all_sync(0xffffffffu, alive);
          if (!alive) continue;
          const int tok0 = p.b0 * B + i * C::TS;
          const bool valid = r < p.tok_end - tok0;
          convert_k(k_st + slot * KSTAGE, C::TM_K + slot * 64, valid);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&cvt_k[slot]);
          if (alive && !mbar_wait_bounded(&full_v[slot], par, kWaitLimitNs)) {
            alive = false;
            record_status(a.status, 8);
          }
          alive = __all_sync(0xffffffffu, alive);
          if (!alive) continue;
          convert_v(v_st + slot * C::STAGE, valid);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&cvt_v[slot]);
        }
      }
    }
  } else {
    // ----------------------------------------------------- softmax warps
    if constexpr (F8) tc_regs_f8<kTcRegsSoftmax>();
    wait_previous_grid();
    TcSoftmax sm;
    sm.a = &a;
    sm.k_st = k_st;
    sm.v_st = v_st;
    sm.red = red;
    sm.cmx = cmx;
    sm.lsum = lsum;
    sm.full = full;
    sm.s_full = s_full;
    sm.p_full = p_full;
    sm.empty = empty;
    sm.o_free = o_free;
    sm.tmem = tmem;
    sm.B = B;
    sm.cstride = PLAN ? a.c_max : G;
    sm.alive = true;
    sm.stage = 0;
    Piece p;
    while (next_piece(p)) {
      const int n_st = stages_of(p);
      if (n_st == 0) {
        // no block of this piece: an empty partial that the merge skips
        const long long slot_id = (long long)blockIdx.x + p.seg;
        for (int c = 0; c < p.ncols; ++c)
          a.ws_o[(slot_id * sm.cstride + c) * C::D + threadIdx.x] = 0.f;
        if (threadIdx.x < p.ncols) {
          a.ws_ml[(slot_id * sm.cstride + threadIdx.x) * 2] = -INFINITY;
          a.ws_ml[(slot_id * sm.cstride + threadIdx.x) * 2 + 1] = 0.f;
        }
        continue;
      }
      if (p.ncols <= 8)
        sm.template run<8, F8>(p, n_st);
      else if (p.ncols <= 16)
        sm.template run<16, F8>(p, n_st);
      else
        sm.template run<32, F8>(p, n_st);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
}

// Launch of the tcgen05 split pass, one CTA per SM (capped at max_grid) on
// the first call for a pool (*grid_io <= 0), the same count afterwards.
template <bool F8>
cudaError_t launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a_in,
                      int sm_count, int max_grid, int* grid_io, cudaStream_t st, bool pdl) {
  constexpr int smem = decode_tc_smem_bytes<F8>();
  auto k_plain = decode_tc_kernel<false, F8>;
  auto k_plan = decode_tc_kernel<true, F8>;
  // the dynamic shared-memory limit is a per-function, per-device attribute
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
    if constexpr (F8) {
      // the warpgroups' register split assumes this launch count
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, v ? k_plan : k_plain);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kTcRegsLaunchF8) return cudaErrorInvalidConfiguration;
    }
    attr_set[v][dev] = true;
  }
  if (*grid_io <= 0) *grid_io = sm_count < max_grid ? sm_count : max_grid;
  DecodeArgs a = a_in;
  a.grid = *grid_io;
  return launch_kernel(pdl, v ? k_plan : k_plain, dim3(a.grid), dim3(tc_threads<F8>()), smem, st,
                       tk, tv, a);
}

}  // namespace pkv
