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
// Q and the K block are K-major, V is N-major, all with the 128-byte swizzle
// (K and V written by TMA from the pool's block rows); P, the weights as a
// bf16 high part and a bf16 remainder (~16 mantissa bits), is written by the
// softmax threads K-major: the high part into the K area of the block (the S
// MMA is done with it), the remainder into its own buffer.
//
// Warps 0-3: softmax, thread r owns row r (TMEM lane r) of S and O, so row
// maxima and sums need no exchange.  The reference maximum of a row is lazy:
// it moves only when a score exceeds it by more than 2^8 (then l and the
// thread's O row are rescaled, after the previous block's MMAs have
// completed).  Warps 4 and 5 issue the TMA loads of K and V, lane 0 of warp
// 6 the MMAs (the next block's S goes ahead of this block's P.V when its
// data has landed).  Every mbarrier wait is bounded; parity waits are exact
// because no waiter runs two phases ahead (block MMAs are awaited through the
// block's empty barrier, whose phases are NST blocks apart).
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
  static constexpr int NST = 2;           // key blocks in flight
  static constexpr int QT = 2 * 128 * 128;  // Q tile, 128 rows x 128 dims: 32 KiB
  static constexpr int PT = 2 * 128 * 128;  // one part of P, 128 rows x 128 keys: 32 KiB
  static constexpr int TM_S = 0;            // TMEM columns: S buffers at 0 and 128,
  static constexpr int TM_O = 256;          // O at 256
  static constexpr int TM_COLS = 512;
  static constexpr float TAU = 8.f;
};

constexpr int kPfWarps = 7;
constexpr int kPfTableCache = 128;  // block-table entries per producer
constexpr int kPfThreads = kPfWarps * 32;

constexpr int prefill_tc_smem_bytes() {
  return PfCfg::QT + 2 * PfCfg::NST * PfCfg::STAGE  // Q, K and V blocks
         + PfCfg::NST * PfCfg::PT                   // P remainders
         + 16 * 8 + 16                              // mbarriers, TMEM address
         + 2 * kPfTableCache * 4                    // producer table caches
         + 1024;                                    // alignment
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
  const int s = blockIdx.z, head = blockIdx.y;
  const int H = a.n_kv_heads, G = a.n_q_heads / H, B = a.block_size;
  const int T = 128 / G;  // tokens per tile
  // tile geometry (host-written metadata: read before waiting on the
  // previous grid)
  const int row0 = a.chunk_start[s];
  const int c = a.chunk_start[s + 1] - row0;
  const int ctx = a.ctx[s];
  if (c < 0 || ctx < c || ctx > a.max_blocks * B || c > static_cast<int>(gridDim.x) * T) {
    // inconsistent metadata, or a chunk longer than the grid was sized for
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) record_status(a.status, 16);
    return;
  }
  const int tok0 = blockIdx.x * T;
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
  unsigned char* plo = v_st + NST * C::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(plo + NST * C::PT);
  uint64_t* empty = full + NST;
  uint64_t* s_full = empty + NST;  // [2]
  uint64_t* p_full = s_full + 2;   // [2]
  uint64_t* q_full = p_full + 2;
  uint64_t* fin = q_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 16);
  int32_t* tcache = reinterpret_cast<int32_t*>(tmem_slot + 4);

  if ((smem_u32(q_s) & 1023u) != 0u) {
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
    mbar_init(q_full, 4);
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

  if (warp == 4 || warp == 5) {
    // ------------------------------------------------ producers (K, V)
    const bool kp = warp == 4;
    const CUtensorMap* tmap = kp ? &tmap_k : &tmap_v;
    unsigned char* dst_st = kp ? k_st : v_st;
    if (lane == 0) prefetch_tmap(tmap);
    TableCacheN<kPfTableCache> tc;
    tc.ent = tcache + (warp - 4) * kPfTableCache;
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
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], 1u * nunits * UR * C::D * 2);
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
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(dst_st + slot * C::STAGE + hf * C::HALF + u * UR * 128, tmap,
                      head * C::D + hf * 64, y, &full[slot]);
      }
    }
    // copies still in flight land before the CTA may exit
    const int first = n_kb > NST ? n_kb - NST : 0;
    for (int j = first; j < n_kb && alive; ++j)
      alive = mbar_wait_bounded(&full[j % NST], (j / NST) & 1, kWaitLimitNs);
  } else if (warp == 6) {
    // ---------------------------------------------------------- MMA issuer
    griddep_wait();
    griddep_launch_dependents();
    if (lane == 0) {
      const uint32_t qb = smem_u32(q_s), kb = smem_u32(k_st), vb = smem_u32(v_st),
                     pl = smem_u32(plo);
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16(128, 128, false, true);
      bool alive = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (alive && !mbar_wait_bounded(bar, parity, kWaitLimitNs)) {
          alive = false;
          record_status(a.status, 8);
        }
        return alive;
      };
      int issued = 0;  // S issued for blocks 0 .. issued - 1
      auto issue_s = [&](bool block) {
        const int j = issued;
        const bool ok = block ? wait(&full[j % NST], (j / NST) & 1)
                              : alive && mbar_test_wait(&full[j % NST], (j / NST) & 1);
        if (!ok) return;
        tc_fence_after();
        const uint32_t ks = kb + (j % NST) * C::STAGE;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * C::HALF + (k & 3) * 32;
          tc_mma(tmem + C::TM_S + (j & 1) * 128, smem_desc(qb + off, 16, 1024, kSwizzle128),
                 smem_desc(ks + off, 16, 1024, kSwizzle128), idS, k > 0);
        }
        tc_commit(&s_full[j & 1]);
        ++issued;
      };
      wait(q_full, 0);
      issue_s(true);
      for (int j = 0; j < n_kb && alive; ++j) {
        if (issued == j + 1 && issued < n_kb) issue_s(false);
        wait(&p_full[j & 1], (j >> 1) & 1);
        if (alive) {
          tc_fence_after();
          const int nvalid = n_keys - j * C::KB < C::KB ? n_keys - j * C::KB : C::KB;
          const int nk = (nvalid + 15) >> 4;
          const uint32_t vs = vb + (j % NST) * C::STAGE;
          const uint32_t ph = kb + (j % NST) * C::STAGE;  // P high part in the K area
          const uint32_t pr = pl + (j % NST) * C::PT;
          for (int k = 0; k < nk; ++k) {
            const uint32_t poff = (k >> 2) * C::HALF + (k & 3) * 32;
            const uint64_t dv = smem_desc(vs + k * 2048, C::HALF, 1024, kSwizzle128);
            tc_mma(tmem + C::TM_O, smem_desc(ph + poff, 16, 1024, kSwizzle128), dv, idPV,
                   (j > 0 || k > 0) ? 1u : 0u);
            tc_mma(tmem + C::TM_O, smem_desc(pr + poff, 16, 1024, kSwizzle128), dv, idPV, 1u);
          }
          tc_commit(&empty[j % NST]);
        }
        if (issued == j + 1 && issued < n_kb) issue_s(true);
      }
      tc_commit(fin);
      mbar_wait_bounded(fin, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- softmax rows
    const int r = threadIdx.x;             // tile row = TMEM lane
    const int tl = r / G, g = r - tl * G;  // token of the tile, query head of the K/V head
    const bool row_ok = tl < ntok;
    const int pos = h + tok0 + tl;         // the token's position: keys 0 .. pos
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
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
    // ---- Q tile: row r, K-major, 128-byte swizzle (zero past the chunk)
    {
      const uint32_t qbase = smem_u32(q_s);
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const unsigned char*>(a.q) +
          ((static_cast<long long>(row0 + tok0 + tl) * a.n_q_heads + head * G + g) * C::D) * 2);
#pragma unroll 4
      for (int ch = 0; ch < 16; ++ch) {
        const uint4 v = row_ok ? src[ch] : make_uint4(0, 0, 0, 0);
        sts128(kmajor_chunk(qbase, r, ch), v.x, v.y, v.z, v.w);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    const float qs = a.qscale;
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < n_kb; ++j) {
      const int slot = j % NST;
      const int k0 = j * C::KB;
      const int nvalid = n_keys - k0 < C::KB ? n_keys - k0 : C::KB;
      wait(&full[slot], (j / NST) & 1);
      wait(&s_full[j & 1], (j >> 1) & 1);
      __syncwarp();
      tc_fence_after();
      const uint32_t sb = tmem + C::TM_S + (j & 1) * 128 + lanes;
      const bool masked = k0 + C::KB - 1 > pos;  // some key of the block is past pos
      // pass 1: the row maximum of the admitted scores
      float mx = -INFINITY;
#pragma unroll 1
      for (int c0 = 0; c0 < C::KB; c0 += 32) {
        uint32_t sr[32];
        tmem_ld32(sb + c0, sr);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const bool ok = !masked || k0 + c0 + i <= pos;
          mx = ok ? fmaxf(mx, __uint_as_float(sr[i])) : mx;
        }
      }
      mx = row_ok ? mx * qs : -INFINITY;
      // the reference moves when a score exceeds it by more than 2^8: l and,
      // after the previous block's MMAs, this row of O are rescaled (the
      // TMEM accesses are warp-wide: lanes whose reference stays scale by 1)
      const bool upd = mx > m_ref + C::TAU;
      float al = 1.f;
      if (upd) {
        al = exp2_approx(m_ref - mx);
        l *= al;
        m_ref = mx;
      }
      if (__any_sync(0xffffffffu, upd)) {
        if (j > 0) {
          wait(&empty[(j - 1) % NST], ((j - 1) / NST) & 1);
          __syncwarp();
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < C::D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + C::TM_O + c0 + lanes, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al);
            tmem_st32(tmem + C::TM_O + c0 + lanes, o);
          }
        }
      }
      // pass 2: weights, high part into the K area, remainder into its buffer
      const uint32_t ph = smem_u32(k_st + slot * C::STAGE);
      const uint32_t pr = smem_u32(plo + slot * C::PT);
#pragma unroll 1
      for (int c0 = 0; c0 < C::KB; c0 += 32) {
        uint32_t sr[32];
        tmem_ld32(sb + c0, sr);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = c8 * 8 + 2 * k;
            const bool ok0 = row_ok && (!masked || k0 + c0 + i <= pos);
            const bool ok1 = row_ok && (!masked || k0 + c0 + i + 1 <= pos);
            const float p0 = ok0 ? exp2_approx(fmaf(__uint_as_float(sr[i]), qs, -m_ref)) : 0.f;
            const float p1 =
                ok1 ? exp2_approx(fmaf(__uint_as_float(sr[i + 1]), qs, -m_ref)) : 0.f;
            l += p0 + p1;
            hi[k] = pack_bf16(p0, p1);
            lo[k] = pack_bf16(p0 - __uint_as_float(hi[k] << 16),
                              p1 - __uint_as_float(hi[k] & 0xffff0000u));
          }
          const int ch = (c0 >> 3) + c8;
          sts128(kmajor_chunk(ph, r, ch), hi[0], hi[1], hi[2], hi[3]);
          sts128(kmajor_chunk(pr, r, ch), lo[0], lo[1], lo[2], lo[3]);
        }
      }
      // keys past the context inside the last 16-key step: V must be finite
      // there (unused slots may hold anything), so its rows are zeroed
      if (r >= nvalid && r < ((nvalid + 15) & ~15)) {
        const uint32_t vb = smem_u32(v_st + slot * C::STAGE) + r * 128;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int k = 0; k < 8; ++k) sts128(vb + hf * C::HALF + k * 16, 0u, 0u, 0u, 0u);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j & 1]);
    }
    // ---- O row: wait for the last block's MMAs, normalise, store
    wait(&empty[(n_kb - 1) % NST], ((n_kb - 1) / NST) & 1);
    __syncwarp();
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const long long orow = (static_cast<long long>(row0 + tok0 + tl) * a.n_q_heads + head * G + g);
#pragma unroll 1
    for (int c0 = 0; c0 < C::D; c0 += 32) {
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
