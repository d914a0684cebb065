// Split-K paged decode attention, partial pass, on the fifth-generation
// tensor cores (tcgen05) with accumulators in tensor memory (TMEM).
//
// Same contract, work split, pieces and workspace as decode_mma.cuh: per
// piece (a block range of one segment) it writes the base-2 online-softmax
// statistics m, l and the unnormalised O of each of the segment's query
// columns ("PagedAttention 的块表与碎片控制" §07 for the attention, "KV 缓存管理"
// chunked-prefill section for the split and merge rule).  bfloat16 K/V,
// D_h = 128, B a multiple of 8 with whole 64-row boxes per block.
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
// the next pieces' S can start while the current one finishes), and lane 0 of
// warp 6 issues the MMAs, starting the next stage's S first when its data
// has already landed.
// Softmax is
// lazy: the reference max m of a column only moves when a new score exceeds
// it by more than 2^8 (TAU = 8 in base-2 units), so in the steady state a
// stage costs one barrier-reduction to confirm that nothing moved, and the
// weights stay below 2^8.  When m moves, the column maxima of the stage are
// reduced exactly, l is rescaled, and O^T is rescaled in TMEM once the
// previous stage's MMAs have completed.
//
// A parity wait is exact only while the waiter is never two phases ahead of
// the barrier: each role waits every phase of full, s_full, p_full, q_full,
// q_empty and o_free in order, and the MMAs of a stage are awaited through that
// stage's empty barrier, whose phases are NST stages apart.
//
// Every mbarrier wait is bounded; a wait that gives up records
// KV_DEV_WAIT_TIMEOUT and the role runs the rest of its loops without waiting
// or issuing, so that every named barrier is still reached and the CTA frees
// its TMEM and exits.
#pragma once

#include "decode_mma.cuh"
#include "tc.cuh"

namespace pkv {

constexpr int kTcWarps = 7;
constexpr int kTcThreads = kTcWarps * 32;

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
};

constexpr int decode_tc_smem_bytes() {
  return 2 * TcCfg::NST * TcCfg::STAGE  // K, V stages
         + TcCfg::QBUF * TcCfg::QTILE   // Q tiles
         + 3 * 4 * 32 * 4               // column maxima, per-warp broadcast, l sums
         + 20 * 8                       // mbarriers
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
  template <int NCP>
  __device__ void run(const Piece& p, int n_st) {
    using C = TcCfg;
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
      const int slot = stage % C::NST;
      const int tok0 = p.b0 * B + i * C::TS;
      const int nvalid = p.tok_end - tok0 < C::TS ? p.tok_end - tok0 : C::TS;
      const bool valid = t < nvalid;
      wait(&full[slot], (stage / C::NST) & 1);
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
          wait(&empty[(stage - 1) % C::NST], ((stage - 1) / C::NST) & 1);
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
      // ---- weights: bf16 high part (chunks 0-3) and remainder (chunks 4-7)
      // of row t of P (N-major, 128-byte swizzle: chunk c at c ^ (t & 7))
      const uint32_t pb = smem_u32(k_st + slot * C::STAGE);
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
          hi[k] = pack_bf16(p0, p1);
          lo[k] = pack_bf16(p0 - __uint_as_float(hi[k] << 16),
                            p1 - __uint_as_float(hi[k] & 0xffff0000u));
        }
        sts128(pb + t * 128 + ((c8 ^ (t & 7)) << 4), hi[0], hi[1], hi[2], hi[3]);
        sts128(pb + t * 128 + (((4 + c8) ^ (t & 7)) << 4), lo[0], lo[1], lo[2], lo[3]);
      }
      // rows past the context inside the last 16-row MMA step: V must be
      // finite there (unused slots may hold anything), so it is zeroed
      if (!valid && t < ((nvalid + 15) & ~15)) {
        const uint32_t vb = smem_u32(v_st + slot * C::STAGE) + t * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int k = 0; k < 8; ++k) sts128(vb + h * C::HALF + k * 16, 0u, 0u, 0u, 0u);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[stage & 1]);
    }

    // ---- end of the piece: O^T from TMEM once the last stage's MMAs are
    // done, l reduced over the 128 rows
    wait(&empty[(stage - 1) % C::NST], ((stage - 1) / C::NST) & 1);
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
        if (c0 + c < ncols)
          a->ws_o[(slot_id * cstride + c0 + c) * C::D + t] =
              __uint_as_float(oh[c]) + __uint_as_float(ol[c]);
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

template <bool PLAN>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
  using C = TcCfg;
  constexpr int NST = C::NST;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* k_st = smem;
  unsigned char* v_st = k_st + NST * C::STAGE;
  unsigned char* q_s = v_st + NST * C::STAGE;  // QBUF Q tiles
  float* red = reinterpret_cast<float*>(q_s + C::QBUF * C::QTILE);
  float* cmx = red + 128;
  float* lsum = cmx + 128;
  uint64_t* full = reinterpret_cast<uint64_t*>(lsum + 128);
  uint64_t* empty = full + NST;
  uint64_t* s_full = empty + NST;  // [2]
  uint64_t* p_full = s_full + 2;   // [2]
  uint64_t* q_full = p_full + 2;           // [QBUF]
  uint64_t* q_empty = q_full + C::QBUF;    // [QBUF]
  uint64_t* o_free = q_empty + C::QBUF;
  uint64_t* fin = o_free + 1;
  long long* walk = reinterpret_cast<long long*>(full + 20);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(walk + 4);
  int32_t* tcache = reinterpret_cast<int32_t*>(tmem_slot + 4);
  PlanStart* rec_s = reinterpret_cast<PlanStart*>(tcache + 2 * kTableCache);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int H = a.n_kv_heads;
  const int G = a.n_q_heads / H;
  const int UR = B < 64 ? B : 64;  // rows per TMA box (a multiple of 8 dividing B and 128)

  // self-check: swizzled buffers must sit on 1 KiB boundaries
  if ((smem_u32(k_st) & 1023u) != 0u) {
    if (threadIdx.x == 0) record_status(a.status, 32);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 2);  // the K and the V producer
      mbar_init(&empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full[0], 4);
    mbar_init(&p_full[1], 4);
    for (int i = 0; i < C::QBUF; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(o_free, 4);
    mbar_init(fin, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TM_COLS);
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
          sts128(qs + h * C::QHALF + col * 128 + ((c ^ (col & 7)) << 4), qv[k].x, qv[k].y,
                 qv[k].z, qv[k].w);
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
              write_new_row<C::D, false>(a, p.rep, p.head, pid, t - j * B, kp, !kp, lane);
          }
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], 1u * nunits * UR * C::D * 2);
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
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int x = p.head * C::D + h * 64;
            const int off = slot * C::STAGE + h * C::HALF + u * UR * 128;
            tma_load_2d(dst_st + off, tmap, x, y, &full[slot]);
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
    for (int k = first; k < stage && alive; ++k)
      alive = mbar_wait_bounded(&full[k % NST], (k / NST) & 1, kWaitLimitNs);
  } else if (warp == 6) {
    // -------------------------------------------------------- MMA issuer
    wait_previous_grid();
    if (lane == 0) {
      const uint32_t kb = smem_u32(k_st), vb = smem_u32(v_st), qb = smem_u32(q_s);
      constexpr uint32_t idS16 = idesc_bf16(128, 16, false, false);
      constexpr uint32_t idS32 = idesc_bf16(128, 32, false, false);
      constexpr uint32_t idPV = idesc_bf16(128, 64, true, true);
      bool alive = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (alive && !mbar_wait_bounded(bar, parity, kWaitLimitNs)) {
          alive = false;
          record_status(a.status, 8);
        }
        return alive;
      };
      auto issue_s = [&](int st, uint32_t idS, uint32_t qbase) {
        const uint32_t ks = kb + (st % NST) * C::STAGE;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * C::HALF + (k & 3) * 32;
          const uint32_t qoff = (k >> 2) * C::QHALF + (k & 3) * 32;
          tc_mma(tmem + C::TM_S + (st & 1) * 32, smem_desc(ks + off, 16, 1024, kSwizzle128),
                 smem_desc(qbase + qoff, 16, 1024, kSwizzle128), idS, k > 0);
        }
        tc_commit(&s_full[st & 1]);
      };
      int stage = 0, npiece = 0;
      Piece p;
      while (next_piece(p)) {
        const int n_st = stages_of(p);
        if (n_st == 0) continue;
        const uint32_t idS = p.ncols <= 16 ? idS16 : idS32;
        const int qbi = npiece % C::QBUF;
        const uint32_t qbase = qb + qbi * C::QTILE;
        wait(&q_full[qbi], (npiece / C::QBUF) & 1);
        if (npiece > 0) wait(o_free, (npiece - 1) & 1);
        int issued = 0;  // S issued for stages stage .. stage + issued - 1
        // S of the next stage; blocking, or only when its data is already in
        auto issue_next = [&](bool block) {
          const int st = stage + issued;
          const bool ok = block ? wait(&full[st % NST], (st / NST) & 1)
                                : alive && mbar_test_wait(&full[st % NST], (st / NST) & 1);
          if (!ok) return;
          tc_fence_after();
          issue_s(st, idS, qbase);
          if (++issued == n_st) tc_commit(&q_empty[qbi]);  // Q tile free once these are done
        };
        issue_next(true);
        for (int i = 0; i < n_st; ++i) {
          const int cur = stage + i;
          // the next stage's S goes first when its data is already in (its S
          // buffer was released with P of the stage before); the wait for P
          // suspends the thread rather than spinning, since this lane shares
          // a scheduler with a softmax warp
          if (issued == i + 1 && issued < n_st) issue_next(false);
          wait(&p_full[cur & 1], (cur >> 1) & 1);
          if (alive) {
            tc_fence_after();
            const int tok0 = p.b0 * B + i * C::TS;
            const int nvalid = p.tok_end - tok0 < C::TS ? p.tok_end - tok0 : C::TS;
            const int nk = (nvalid + 15) >> 4;
            const uint32_t vs = vb + (cur % NST) * C::STAGE;
            const uint32_t ps = kb + (cur % NST) * C::STAGE;
            for (int k = 0; k < nk; ++k)
              tc_mma(tmem + C::TM_O, smem_desc(vs + k * 2048, C::HALF, 1024, kSwizzle128),
                     smem_desc(ps + k * 2048, C::HALF, 1024, kSwizzle128), idPV,
                     (i > 0 || k > 0) ? 1u : 0u);
            tc_commit(&empty[cur % NST]);
          }
          if (issued == i + 1 && issued < n_st) issue_next(true);
        }
        stage += n_st;
        ++npiece;
      }
      // every MMA issued has completed before TMEM is released
      tc_commit(fin);
      mbar_wait_bounded(fin, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------- softmax warps
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
        sm.run<8>(p, n_st);
      else if (p.ncols <= 16)
        sm.run<16>(p, n_st);
      else
        sm.run<32>(p, n_st);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

}  // namespace pkv
