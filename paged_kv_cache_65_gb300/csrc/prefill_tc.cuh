// Chunked-prefill attention over the paged cache on tcgen05 ("KV 缓存管理",
// chunked-prefill section; "第 8 章 推理优化" §8.2.3).
//
// Sequence s has a chunk of c new tokens (rows chunk_start[s] ..
// chunk_start[s + 1] - 1 of q) whose keys and values are already in the pool:
// they are the last c of context_lens[s] = h + c positions.  The chunk's
// token i (position h + i) attends to every position 0 .. h + i: the whole
// history and the chunk's tokens up to its own.
//
// One CTA per (sequence, K/V head, tile of 128 query rows).  A tile row is
// (token, query head of the K/V head): row r = t * G + g, so a tile holds
// 128 / G tokens.  Per block of 128 keys (keys in FlashAttention orientation,
// both accumulators in TMEM):
//     S [128 rows x 128 keys] = Q [128 x 128] . K^T            (8 MMAs, K = 16)
//     O [128 rows x 128 dims] += P_hi . V + P_lo . V           (16 MMAs)
// Q and the K block are K-major in shared memory, V is N-major, all with the
// 128-byte swizzle (K and V written by TMA from the pool's block rows).  P,
// the weights as a bf16 high part and a bf16 remainder (~16 mantissa bits),
// is written by the softmax threads over the block's own S columns in TMEM
// and read from there as the A operand of the P.V MMAs; three S/P buffers
// and O fill the 512 TMEM columns.  K and V have their own three-deep
// stages: a K slot is free once its S MMAs are done, a V slot once its P.V
// MMAs are.
//
// Warps 0-7: softmax, two warpgroups on the same rows: thread r of group h
// owns row r (TMEM lane r) and the keys 64 h .. 64 h + 63 of every block (and
// O's columns 64 h ..).  The two halves of a row exchange their maxima
// through shared memory (truncated to bf16, so both compute the same
// reference) and add their sums at the end.  The reference maximum of a row
// is lazy: it moves only when a score exceeds it by more than 2^8 (then l
// and the row of O are rescaled, after the previous block's MMAs have
// completed).  Warps 8-11 issue the TMA loads of K and V (one 64-column half
// each, so that box issue keeps up with 16-token pages); lane 0 of warp 12
// issues the S MMAs, running ahead as far as K blocks and free S/P buffers
// allow, and lane 0 of warp 13 the P.V MMAs (one thread issuing both kinds
// could not keep the tensor core busy: a single thread issues an MMA every
// ~60 cycles, about the tensor core's time for one 128 x 128 x 16 step).
// Every mbarrier wait is bounded; parity waits are exact because no waiter
// runs two phases ahead.
#pragma once

#include <cuda_bf16.h>

#include "decode_tc.cuh"
#include "prefill.h"

namespace pkv {

struct PfCfg {
  static constexpr int D = 128;
  static constexpr int KB = 128;          // keys per block
  static constexpr int HALF = KB * 128;   // one 64-element half of a K or V block: 16 KiB
  static constexpr int STAGE = 2 * HALF;  // K (or V) of one block: 32 KiB
  static constexpr int NST = 3;           // K and V stages
  static constexpr int QT = 2 * 128 * 128;  // Q tile, 128 rows x 128 dims: 32 KiB
  static constexpr int NSB = 3;             // S/P buffers in TMEM, 128 columns each
  static constexpr int TM_O = NSB * 128;    // O after them
  static constexpr int TM_COLS = 512;
  static constexpr float TAU = 8.f;
};
static_assert(PfCfg::TM_O + PfCfg::D <= PfCfg::TM_COLS, "TMEM columns");

// warpgroups 0 and 1 (warps 0-7): softmax, keys 0-63 and 64-127 of a block;
// warpgroup 2: K producers 8 (columns 0-63) and 10 (64-127), V producers 9
// and 11; warpgroup 3: MMA issuers 12 (S) and 13 (P.V), 14 and 15 idle.
// Every SM sub-partition (warp % 4) holds one warp of each group.  Launched
// at 128 registers a thread (512 threads), the groups move to 192 / 192 /
// 64 / 64: 128 x (2 x 192 + 2 x 64) = 65536.
constexpr int kPfWarps = 16;
constexpr int kPfRegsSoftmax = 192, kPfRegsHelper = 64;
static_assert(128 * (2 * kPfRegsSoftmax + 2 * kPfRegsHelper) <= 65536, "register split");
constexpr int kPfTableCache = 32;  // block-table entries per producer
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kPfBarriers = 4 * PfCfg::NST + 2 * PfCfg::NSB + 2;

constexpr int prefill_tc_smem_bytes() {
  return PfCfg::QT + 2 * PfCfg::NST * PfCfg::STAGE  // Q, K and V blocks
         + kPfBarriers * 8 + 16                     // mbarriers, TMEM address
         + 4 * kPfTableCache * 4                    // producer table caches
         + 2 * 2 * 128 * 2                          // row-maximum exchange (bf16)
         + 1024;                                    // alignment
}

// Paired fp32 arithmetic (two lanes of fp32 in one 64-bit register, one
// instruction for both) and the three-input maximum.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// swizzled 16-byte chunk ch (0..15 over 128 elements) of row r in a K-major
// tile of two 64-element halves
__device__ __forceinline__ uint32_t kmajor_chunk(uint32_t base, int r, int ch) {
  return base + (ch >> 3) * (128 * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
  using C = PfCfg;
  constexpr int NST = C::NST;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.n_kv_heads, G = a.n_q_heads / H, B = a.block_size;
  const int T = 128 / G;  // tokens per tile
  // the work item: (sequence, tile) from the grid, or from a host-built
  // heaviest-first order (host-written metadata, like the chunk geometry:
  // read before waiting on the previous grid)
  int s, head, tile, planned_c = -1;
  if (a.sched) {
    const int item = static_cast<int>(blockIdx.x) / H;
    head = static_cast<int>(blockIdx.x) - item * H;
    const int4 w = a.sched[item];
    s = w.x;
    tile = w.y;
    planned_c = w.z;
    if (s < 0 || s >= a.n_seq || tile < 0) {
      if (threadIdx.x == 0) record_status(a.status, 16);
      return;
    }
  } else {
    s = blockIdx.z;
    head = blockIdx.y;
    tile = blockIdx.x;
  }
  const int row0 = a.chunk_start[s];
  const int c = a.chunk_start[s + 1] - row0;
  const int ctx = a.ctx[s];
  const bool sized = a.sched ? c == planned_c : c <= static_cast<int>(gridDim.x) * T;
  if (c < 0 || ctx < c || ctx > a.max_blocks * B || !sized) {
    // inconsistent metadata, a chunk longer than the grid was sized for, or
    // one whose length is not the one the work order was built for
    if (threadIdx.x == 0 && (a.sched ? head == 0 : blockIdx.x == 0 && blockIdx.y == 0))
      record_status(a.status, 16);
    return;
  }
  const int tok0 = tile * T;
  if (tok0 >= c) return;  // past this sequence's chunk
  const int h = ctx - c;                               // history length
  const int ntok = c - tok0 < T ? c - tok0 : T;        // tokens of this tile
  const int n_keys = h + tok0 + ntok;                  // keys up to the tile's last token
  const int n_kb = (n_keys + C::KB - 1) / C::KB;
  const int UR = B < 64 ? B : 64;                      // rows per TMA box

  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* q_s = smem;
  unsigned char* k_st = q_s + C::QT;
  unsigned char* v_st = k_st + NST * C::STAGE;
  uint64_t* k_full = reinterpret_cast<uint64_t*>(v_st + NST * C::STAGE);
  uint64_t* k_empty = k_full + NST;  // S MMAs of the block done
  uint64_t* v_full = k_empty + NST;
  uint64_t* v_empty = v_full + NST;  // P.V MMAs of the block done
  uint64_t* s_full = v_empty + NST;  // [NSB]
  uint64_t* p_full = s_full + C::NSB;  // [NSB]
  uint64_t* q_full = p_full + C::NSB;
  uint64_t* fin = q_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  int32_t* tcache = reinterpret_cast<int32_t*>(tmem_slot + 4);
  // [2 parities][2 halves][128 rows] bf16 maxima; at the end each row's
  // two half sums, split over its slots of both parities
  uint16_t* xmax = reinterpret_cast<uint16_t*>(tcache + 4 * kPfTableCache);

  if ((smem_u32(q_s) & 1023u) != 0u) {
    if (threadIdx.x == 0) record_status(a.status, 32);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&k_full[i], 2);  // the producers of the two halves
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 2);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < C::NSB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);  // both softmax warpgroups
    }
    mbar_init(q_full, 8);
    mbar_init(fin, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8 && warp < 12) {
    // ------------------------------------ producers (K or V, one half each)
    reg_dealloc<kPfRegsHelper>();
    const bool kp = (warp & 1) == 0;
    const int hf = (warp - 8) >> 1;  // 64-column half of the rows
    const CUtensorMap* tmap = kp ? &tmap_k : &tmap_v;
    unsigned char* dst_st = kp ? k_st : v_st;
    uint64_t* full = kp ? k_full : v_full;
    uint64_t* empty = kp ? k_empty : v_empty;
    if (lane == 0) prefetch_tmap(tmap);
    TableCacheN<kPfTableCache> tc;
    tc.ent = tcache + (warp - 8) * kPfTableCache;
    tc.ensure(a.table, a.max_blocks, s, 0, 0, lane);  // host-written: before the wait
    griddep_wait();
    griddep_launch_dependents();
    bool alive = true;
    for (int j = 0; j < n_kb; ++j) {
      const int slot = j % NST;
      if (j >= NST && alive) {
        if (!mbar_wait_bounded(&empty[slot], ((j / NST) & 1) ^ 1, kWaitLimitNs)) {
          alive = false;
          if (lane == 0) record_status(a.status, 8);
        }
      }
      alive = __all_sync(0xffffffffu, alive);
      if (!alive) break;
      const int k0 = j * C::KB;
      const int nvalid = n_keys - k0 < C::KB ? n_keys - k0 : C::KB;
      const int nunits = (nvalid + UR - 1) / UR;
      tc.ensure(a.table, a.max_blocks, s, k0 / B, (k0 + (nunits - 1) * UR) / B, lane);
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], 1u * nunits * UR * 64 * 2);
      __syncwarp();
      for (int u = lane; u < nunits; u += 32) {
        const int tk = k0 + u * UR;
        const int jb = tk / B;
        const int row = tk - jb * B;
        int pid = tc.ent[jb - tc.base];
        if (pid < 0 || pid >= a.n_blocks) {
          record_status(a.status, 1);
          pid = 0;  // stay in bounds; the result is flagged as invalid
        }
        const int y = (a.layer * a.n_blocks + pid) * B + row;
        tma_load_2d(dst_st + slot * C::STAGE + hf * C::HALF + u * UR * 128, tmap,
                    head * C::D + hf * 64, y, &full[slot]);
      }
    }
    // copies still in flight land before the CTA may exit
    const int first = n_kb > NST ? n_kb - NST : 0;
    for (int j = first; j < n_kb && alive; ++j)
      alive = mbar_wait_bounded(&full[j % NST], (j / NST) & 1, kWaitLimitNs);
  } else if (warp >= 12) {
    // ------------------------------ MMA issuers (12: S, 13: P.V); 14, 15 idle
    reg_dealloc<kPfRegsHelper>();
    griddep_wait();
    griddep_launch_dependents();
    if (warp < 14 && lane == 0) {
      bool alive = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (alive && !mbar_wait_bounded(bar, parity, kWaitLimitNs)) {
          alive = false;
          record_status(a.status, 8);
        }
        return alive;
      };
      if (warp == 12) {
        // S of block j into S/P buffer j % NSB, once K has landed and the
        // P.V that last read the buffer (block j - NSB) is done
        const uint32_t qb = smem_u32(q_s), kb = smem_u32(k_st);
        constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
        wait(q_full, 0);
        for (int j = 0; j < n_kb && alive; ++j) {
          if (!wait(&k_full[j % NST], (j / NST) & 1)) break;
          if (j >= C::NSB && !wait(&v_empty[(j - C::NSB) % NST], ((j - C::NSB) / NST) & 1)) break;
          tc_fence_after();
          const uint32_t ks = kb + (j % NST) * C::STAGE;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * C::HALF + (k & 3) * 32;
            tc_mma(tmem + (j % C::NSB) * 128, smem_desc(qb + off, 16, 1024, kSwizzle128),
                   smem_desc(ks + off, 16, 1024, kSwizzle128), idS, k > 0);
          }
          tc_commit(&k_empty[j % NST]);
          tc_commit(&s_full[j % C::NSB]);
        }
      } else {
        const uint32_t vb = smem_u32(v_st);
        constexpr uint32_t idPV = idesc_bf16(128, 128, false, true);
        for (int j = 0; j < n_kb && alive; ++j) {
          wait(&p_full[j % C::NSB], (j / C::NSB) & 1);
          wait(&v_full[j % NST], (j / NST) & 1);
          if (!alive) break;
          tc_fence_after();
          const int nvalid = n_keys - j * C::KB < C::KB ? n_keys - j * C::KB : C::KB;
          const int nk = (nvalid + 15) >> 4;
          const uint32_t vs = vb + (j % NST) * C::STAGE;
          const uint32_t pt = tmem + (j % C::NSB) * 128;  // P high part; remainder at +64
          for (int k = 0; k < nk; ++k) {
            const uint64_t dv = smem_desc(vs + k * 2048, C::HALF, 1024, kSwizzle128);
            tc_mma_ts(tmem + C::TM_O, pt + k * 8, dv, idPV, (j > 0 || k > 0) ? 1u : 0u);
            tc_mma_ts(tmem + C::TM_O, pt + 64 + k * 8, dv, idPV, 1u);
          }
          tc_commit(&v_empty[j % NST]);
        }
        tc_commit(fin);
        mbar_wait_bounded(fin, 0, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- softmax rows
    reg_alloc<kPfRegsSoftmax>();
    const int hh = warp >> 2;              // half: keys 64 hh .. 64 hh + 63 of a block
    const int qd = warp & 3;               // TMEM lane quadrant
    const int r = qd * 32 + lane;          // tile row = TMEM lane
    const int tl = r / G, g = r - tl * G;  // token of the tile, query head of the K/V head
    const bool row_ok = tl < ntok;
    const int pos = h + tok0 + tl;         // the token's position: keys 0 .. pos
    const uint32_t lanes = static_cast<uint32_t>(qd * 32) << 16;
    const int xbar = 1 + qd;               // named barrier of the row quadrant's two warps
    griddep_wait();
    griddep_launch_dependents();
    bool alive = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (alive && !mbar_wait_bounded(bar, parity, kWaitLimitNs)) {
        alive = false;
        record_status(a.status, 8);
      }
      return alive;
    };
    // ---- Q tile: row r, K-major, 128-byte swizzle (zero past the chunk);
    // each half stages its 64 dimensions
    {
      const uint32_t qbase = smem_u32(q_s);
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const unsigned char*>(a.q) +
          ((static_cast<long long>(row0 + tok0 + tl) * a.n_q_heads + head * G + g) * C::D) * 2);
#pragma unroll 4
      for (int c = 0; c < 8; ++c) {
        const int ch = 8 * hh + c;
        const uint4 v = row_ok ? src[ch] : make_uint4(0, 0, 0, 0);
        sts128(kmajor_chunk(qbase, r, ch), v.x, v.y, v.z, v.w);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    const float qs = a.qscale;
    float m_ref = -INFINITY, l = 0.f;  // l: this half's sum
    for (int j = 0; j < n_kb; ++j) {
      const int slot = j % NST;
      const int k0 = j * C::KB;
      const int nvalid = n_keys - k0 < C::KB ? n_keys - k0 : C::KB;
      wait(&s_full[j % C::NSB], (j / C::NSB) & 1);
      __syncwarp();
      tc_fence_after();
      const uint32_t sb = tmem + (j % C::NSB) * 128 + lanes;
      // this half of the row of S: two loads, one wait
      uint32_t sr[2][32];
      tmem_ld32_nowait(sb + 64 * hh, sr[0]);
      tmem_ld32_nowait(sb + 64 * hh + 32, sr[1]);
      tmem_wait_ld32(sr[0]);
      tmem_wait_ld32(sr[1]);
      // keys this row may not see (past its position; every key for a row
      // past the chunk) become -inf, whatever the slot held; blocks with no
      // such key in the whole warp skip this
      const int lim = (row_ok ? pos - k0 : -1) - 64 * hh;  // key 64 hh + i admitted iff i <= lim
      if (__any_sync(0xffffffffu, lim < 63)) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i) sr[q][i] = q * 32 + i > lim ? 0xff800000u : sr[q][i];
      }
      // pass 1: this half's maximum (four chains of three-input maxima),
      // then the row's: both halves take the larger of the two truncated to
      // bf16, so they agree on the reference exactly
      float mm[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mm[i] = -INFINITY;
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          mm[(i >> 1) & 3] = fmax3(mm[(i >> 1) & 3], __uint_as_float(sr[q][i]),
                                   __uint_as_float(sr[q][i + 1]));
      const float mh = fmaxf(fmaxf(mm[0], mm[1]), fmaxf(mm[2], mm[3])) * qs;
      uint16_t* xm = xmax + (j & 1) * 256;
      const uint16_t mine = static_cast<uint16_t>(__float_as_uint(mh) >> 16);
      xm[hh * 128 + r] = mine;
      named_bar_sync(xbar, 64);
      const uint16_t other = xm[(1 - hh) * 128 + r];
      const float mx = fmaxf(__uint_as_float(static_cast<uint32_t>(mine) << 16),
                             __uint_as_float(static_cast<uint32_t>(other) << 16));
      // the reference moves when the maximum exceeds it by more than 2^8: l
      // and, after the previous block's MMAs, this half of O's row are
      // rescaled (the TMEM accesses are warp-wide: lanes whose reference
      // stays scale by 1)
      const bool upd = mx > m_ref + C::TAU;
      float al = 1.f;
      if (upd) {
        al = exp2_approx(m_ref - mx);
        l *= al;
        m_ref = mx;
      }
      if (__any_sync(0xffffffffu, upd)) {
        if (j > 0) {
          wait(&v_empty[(j - 1) % NST], ((j - 1) / NST) & 1);
          __syncwarp();
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 64 * hh; c0 < 64 * hh + 64; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + C::TM_O + c0 + lanes, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al);
            tmem_st32(tmem + C::TM_O + c0 + lanes, o);
          }
        }
      }
      // pass 2: p = 2^(s * qs - m), a -inf score giving 0 (a row with no
      // admitted key so far has m = -inf and uses 0 instead, all its scores
      // being -inf).  The high part is p's upper 16 bits, the remainder
      // p - hi (exact in fp32, below 2^-7 p) likewise truncated to its upper
      // 16 bits, so hi + lo is within 2^-15 of p with no conversion
      // instruction.  Both go over the block's S columns (high parts of keys
      // 64 hh .. in columns 32 hh .., remainders in 64 + 32 hh ..; S is in
      // registers by now).  l sums p in paired partial sums.
      const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
      const uint64_t qs2 = f2_pack(qs, qs), nm2 = f2_pack(nm, nm), neg2 = f2_pack(-1.f, -1.f);
      uint64_t lp2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
      {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int q = k >> 4, i = 2 * (k & 15);
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[q][i]), __uint_as_float(sr[q][i + 1])), qs2,
                           nm2),
                    x0, x1);
          const float p0 = exp2_approx(x0), p1 = exp2_approx(x1);
          const uint64_t pp = f2_pack(p0, p1);
          lp2[k & 1] = f2_add(lp2[k & 1], pp);
          const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
          hi[k] = __byte_perm(b0, b1, 0x7632);
          float r0, r1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(b0 & 0xffff0000u),
                                   __uint_as_float(b1 & 0xffff0000u)),
                           neg2, pp),
                    r0, r1);
          lo[k] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
        }
        tmem_st32_nowait(sb + 32 * hh, hi);
        tmem_st32_nowait(sb + 64 + 32 * hh, lo);
      }
      {
        float a0, a1, b0, b1;
        f2_unpack(lp2[0], a0, a1);
        f2_unpack(lp2[1], b0, b1);
        l += (a0 + a1) + (b0 + b1);
      }
      tmem_wait_st();
      // keys past the context inside the last 16-key step: V must be finite
      // there (unused slots may hold anything), so its rows are zeroed (each
      // half zeroes its 64 dimensions)
      if (r >= nvalid && r < ((nvalid + 15) & ~15)) {
        wait(&v_full[slot], (j / NST) & 1);
        const uint32_t vb = smem_u32(v_st + slot * C::STAGE) + hh * C::HALF + r * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) sts128(vb + k * 16, 0u, 0u, 0u, 0u);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j % C::NSB]);
    }
    // ---- O row: the two halves' sums, then the last block's MMAs,
    // normalise, store this half's 64 dimensions.  A sum crosses in the
    // row's own two exchange slots of this half (16 bits in each parity's
    // slot): other row quadrants may still be in their loop, reading and
    // writing their own rows' slots, so nothing here may touch another
    // row's bytes; both parities of this row are free once the two halves
    // are past their last maximum read.
    named_bar_sync(xbar, 64);
    {
      const uint32_t lb = __float_as_uint(l);
      xmax[hh * 128 + r] = static_cast<uint16_t>(lb & 0xffffu);
      xmax[256 + hh * 128 + r] = static_cast<uint16_t>(lb >> 16);
    }
    named_bar_sync(xbar, 64);
    const float l0 = __uint_as_float(static_cast<uint32_t>(xmax[r]) |
                                     (static_cast<uint32_t>(xmax[256 + r]) << 16));
    const float l1 = __uint_as_float(static_cast<uint32_t>(xmax[128 + r]) |
                                     (static_cast<uint32_t>(xmax[256 + 128 + r]) << 16));
    const float lt = l0 + l1;
    wait(&v_empty[(n_kb - 1) % NST], ((n_kb - 1) / NST) & 1);
    __syncwarp();
    tc_fence_after();
    const float inv = lt > 0.f ? a.vscale / lt : 0.f;
    const long long orow = (static_cast<long long>(row0 + tok0 + tl) * a.n_q_heads + head * G + g);
#pragma unroll 1
    for (int c0 = 64 * hh; c0 < 64 * hh + 64; c0 += 32) {
      uint32_t o[32];
      tmem_ld32(tmem + C::TM_O + c0 + lanes, o);
      if (row_ok) {
        if (a.out_f32) {
          float4* dst = reinterpret_cast<float4*>(a.out_f32 + orow * C::D + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                 __uint_as_float(o[4 * i + 2]) * inv,
                                 __uint_as_float(o[4 * i + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(a.out_bf16 + orow * C::D + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16(__uint_as_float(o[8 * i]) * inv, __uint_as_float(o[8 * i + 1]) * inv),
                                pack_bf16(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv),
                                pack_bf16(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv),
                                pack_bf16(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv));
        }
      }
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
