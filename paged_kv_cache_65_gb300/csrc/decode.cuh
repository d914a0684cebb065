// Split-K paged decode attention, partial pass.
//
// What it computes ("PagedAttention 的块表与碎片控制" §07, "KV 缓存管理"
// chunked-prefill section): for a sequence s, K/V head h and a contiguous
// range of its logical blocks, the online-softmax statistics of every query
// head g of h's group:
//     m = max_t s_t,  l = sum_t 2^(s_t - m),  O = sum_t 2^(s_t - m) v_t,
// with s_t = (q . k_t) * scale * log2(e)  (base-2 scores; 2^(x log2 e) = e^x).
// Token t of s is read through block_table[s][t / B], slot t % B (§03, §06).
//
// Work split.  All (sequence, K/V head) segments are laid end to end in
// block units (sequence-major, then head); the W blocks are cut into
// `grid` equal chunks, one per CTA (a stream-K style split, so every CTA gets
// the same number of blocks whatever the length mix).  A CTA's chunk may
// cover the tail of one segment and the head of the next; it emits one
// partial per segment piece into workspace slot (cta + segment index), which
// is unique because segments and CTAs advance together.
//
// CTA layout.  4 consumer warps + 1 producer warp.  The producer streams the
// piece's blocks through NST shared-memory stages with TMA tensor loads (box
// = [D_h elements] x [min(B, TS) tokens] of one K/V head: D_h * esize bytes
// per token row, H_kv * D_h * esize bytes apart), completing on an mbarrier
// per stage.  Consumers split each stage into rounds of RT tokens; in a
// round, TG lanes share one token (each lane owns 16 bytes = VEC elements of
// D_h), partial dot products for S steps x G heads are reduced across the TG
// lanes with a transpose-reduce (about one shuffle per score), the round max
// updates the running max, and P.V accumulates in float32 with packed
// f32x2 FMAs.  Each K/V byte is read from HBM once per CTA for all G query
// heads.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"
#include "ptx.cuh"

namespace pkv {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any real wait
constexpr int kTableCache = 256;  // block-table entries cached by the producer

struct DecodeArgs {
  const void* q;
  const int32_t* table;
  const int32_t* ctx;
  long long* ws_pre;  // [n_seq + 1]: blocks (all heads) before each sequence
  float* ws_ml;  // [n_slots][columns][2]: (m in base-2 units, l)
  float* ws_o;   // [n_slots][columns][D]
  int32_t* status;
  int n_seq, max_blocks, layer, n_blocks, block_size, n_kv_heads, n_q_heads;
  float qscale;  // scale * log2(e) (times the K scale of an FP8 pool), folded into q
  float vscale;  // V scale of an FP8 pool (1 otherwise)
  int grid;
  // sharing-aware plan (tensor-core pass only); segs == nullptr: one segment
  // per (sequence, K/V head) taken from the context lengths
  const PlanSeg* segs;
  const int32_t* members;
  int n_segs;
  int c_max;
  long long plan_W;
  // per-CTA start records of the plan (null: none) and the CTA count they
  // were built for; used only when it equals `grid`
  const PlanStart* starts;
  int start_grid;
  // planned pass with the step's slot write fused in (k_new == null: none):
  // rows [plan row][H_kv][D_h] of this layer (bfloat16) of each listed
  // sequence's newest token, its last context position, written into the
  // pool (k_pool / v_pool, FP8 pools as codes of x / k_scale_w, v_scale_w)
  // by the CTA that reads the block holding it, before that read
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  void* k_pool = nullptr;
  void* v_pool = nullptr;
  float k_scale_w = 1.f, v_scale_w = 1.f;
  // q8_0 pools: the fp16 scales [L][N][H_kv][B][D / 32] of K and V
  const void* k_sc = nullptr;
  const void* v_sc = nullptr;
};

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Token rows per pipeline stage (and per TMA box when B is larger): 8 KiB of
// K (and of V) per stage, whatever the query group size.
constexpr int stage_tokens(int esize, int D) { return 8192 / (esize * D); }

template <int ESIZE, int D, int G>
struct DecodeCfg {
  static constexpr int VEC = 16 / ESIZE;             // elements per lane
  static constexpr int TG = D / VEC;                 // lanes per token
  static constexpr int LT = ilog2(TG);
  static constexpr int NG = 32 / TG;                 // tokens per step per warp
  static constexpr int S = G >= 8 ? 2 : 4;           // steps per round
  static constexpr int LS = ilog2(S);
  static constexpr int RT = NG * S;                  // tokens per round
  static constexpr int TS = stage_tokens(ESIZE, D);  // tokens per stage
  static constexpr int V = S * G;                    // scores per lane per round
  static constexpr int LV = ilog2(V);
  static constexpr int HV = V >= TG ? V / TG : 1;    // scores held after reduce
  static constexpr int STAGE_BYTES = TS * D * ESIZE; // one of K or V
  static_assert(TG >= 4 && TG <= 32 && LS <= LT, "lane-group size");
  static_assert((G & (G - 1)) == 0 && G <= 8, "G must be a power of two <= 8");
  static_assert(TS % RT == 0, "a stage holds whole rounds");
};

template <int ESIZE, int D, int G>
constexpr int decode_smem_bytes() {
  using C = DecodeCfg<ESIZE, D, G>;
  return 2 * kStages * C::STAGE_BYTES                    // K and V stages
         + kConsumerWarps * C::RT * G * 4                // p per warp
         + kConsumerWarps * G * D * 4                    // combine: O per warp
         + kConsumerWarps * G * 2 * 4                    // combine: m, l per warp
         + 2 * kStages * 8                               // mbarriers
         + kTableCache * 4                               // producer table cache
         + 64 + 128;                                     // walk state + alignment
}

// ---------------------------------------------------------------- helpers

// 16 bytes of bfloat16 -> 4 float2 (element 2j in .x, 2j+1 in .y)
__device__ __forceinline__ void cvt16(const uint4& w, float2 (&f)[4]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[j].x = __uint_as_float(ws[j] << 16);
    f[j].y = __uint_as_float(ws[j] & 0xffff0000u);
  }
}

// 16 bytes of float32 -> 2 float2
__device__ __forceinline__ void cvt16(const uint4& w, float2 (&f)[2]) {
  f[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
  f[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
}

// Transpose-reduce of N values across the lanes of a TG-lane group (masks
// M, M/2, ..., 1): while more than one value is left each level halves the
// set, a lane keeping the half selected by its mask bit.
template <int N, int M>
struct TReduce {
  static __device__ __forceinline__ void run(float* v, int li) {
    if constexpr (M == 0) {
      return;
    } else if constexpr (N > 1) {
      const bool upper = (li & M) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float keep = upper ? v[i + N / 2] : v[i];
        const float send = upper ? v[i] : v[i + N / 2];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
      TReduce<N / 2, M / 2>::run(v, li);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
      TReduce<1, M / 2>::run(v, li);
    }
  }
};

template <typename C>
__device__ __forceinline__ int held_index(int li, int k) {
  if constexpr (C::V >= C::TG)
    return li * (C::V / C::TG) + k;
  else
    return li >> (C::LT - C::LV);
}

// ------------------------------------------------------------ walk state

// Position of a CTA's chunk start within the segment list.
struct WalkStart {
  int s;        // sequence holding the chunk start (n_seq if none)
  long long pre;  // blocks before sequence s (all heads)
  long long W;    // total blocks
  long long chunk;
};

__device__ __forceinline__ int seq_blocks(const int32_t* ctx, int s, int B, int max_blocks,
                                          int32_t* status) {
  int c = ctx[s];
  if (c < 0 || c > max_blocks * B) {
    record_status(status, 16);
    c = c < 0 ? 0 : max_blocks * B;
  }
  return (c + B - 1) / B;
}

// One warp: total W, chunk, and the sequence containing block index r0.
__device__ inline WalkStart find_start(const int32_t* ctx, int n_seq, int B, int H, int max_blocks,
                                       int grid, int cta, int32_t* status) {
  const int lane = threadIdx.x & 31;
  long long run = 0;
  // pass 1: total
  for (int base = 0; base < n_seq; base += 32) {
    const int s = base + lane;
    long long nb = s < n_seq ? (long long)seq_blocks(ctx, s, B, max_blocks, nullptr) * H : 0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) nb += __shfl_xor_sync(0xffffffffu, nb, o);
    run += nb;
  }
  WalkStart w;
  w.W = run;
  w.chunk = (run + grid - 1) / grid;
  if (w.chunk == 0) w.chunk = 1;
  const long long r0 = (long long)cta * w.chunk;
  w.s = n_seq;
  w.pre = run;
  if (r0 >= run) return w;
  // pass 2: locate r0
  run = 0;
  for (int base = 0; base < n_seq; base += 32) {
    const int s = base + lane;
    long long nb = s < n_seq ? (long long)seq_blocks(ctx, s, B, max_blocks, status) * H : 0;
    long long incl = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, s < n_seq && r0 < run + incl);
    if (hit) {
      const int L = __ffs(hit) - 1;
      const long long excl = __shfl_sync(0xffffffffu, incl - nb, L);
      w.s = base + L;
      w.pre = run + excl;
      return w;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  return w;
}

// One warp of CTA 0: exclusive prefix of blocks (all heads) per sequence,
// plus the total at index n_seq, for the merge pass.
__device__ inline void write_prefix(const int32_t* ctx, int n_seq, int B, int H, int max_blocks,
                                    long long* pre) {
  const int lane = threadIdx.x & 31;
  long long run = 0;
  for (int base = 0; base < n_seq; base += 32) {
    const int s = base + lane;
    long long nb = s < n_seq ? (long long)seq_blocks(ctx, s, B, max_blocks, nullptr) * H : 0;
    long long incl = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (s < n_seq) pre[s] = run + incl - nb;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) pre[n_seq] = run;
}

// Producer-side cache of block-table entries in shared memory: the producer
// warp refills kTableCache consecutive entries of one sequence at a time
// (kTableCache / 32 independent loads per lane, one round trip) instead of
// paying a dependent global load before every TMA issue.

template <int N>
struct TableCacheN {
  static_assert(N % 32 == 0, "whole warps of entries");
  int32_t* ent;  // shared, N entries
  int seq = -1;
  int base = 0;

  // Make blocks [jf, jl] of `seq` available; whole warp calls.
  __device__ void ensure(const int32_t* table, int max_blocks, int s, int jf, int jl, int lane) {
    if (s == seq && jf >= base && jl < base + N) return;
    __syncwarp();
    seq = s;
    base = jf;
    const int32_t* row = table + (long long)s * max_blocks;
#pragma unroll
    for (int i = 0; i < N / 32; ++i) {
      const int j = base + i * 32 + lane;
      ent[i * 32 + lane] = j < max_blocks ? row[j] : 0;
    }
    __syncwarp();
  }
};
using TableCache = TableCacheN<kTableCache>;

// Iterates the pieces of [r0, r1) in segment order.
struct PieceWalker {
  const int32_t* ctx;
  int n_seq, B, H, max_blocks;
  int s;
  long long pre, r, r1;
  // current piece
  int seq, head, nb;          // nb: blocks of the sequence
  int ctx_len;
  int b0, b1;                 // block range inside the segment

  __device__ bool next() {
    while (r < r1 && s < n_seq) {
      int c = ctx[s];
      c = c < 0 ? 0 : (c > max_blocks * B ? max_blocks * B : c);
      const int nbs = (c + B - 1) / B;
      const long long seg_all = (long long)nbs * H;
      if (nbs == 0 || r >= pre + seg_all) {
        pre += seg_all;
        ++s;
        continue;
      }
      const long long off = r - pre;
      head = (int)(off / nbs);
      const long long seg_base = pre + (long long)head * nbs;
      seq = s;
      nb = nbs;
      ctx_len = c;
      b0 = (int)(r - seg_base);
      const long long end = r1 < seg_base + nbs ? r1 : seg_base + nbs;
      b1 = (int)(end - seg_base);
      r = end;
      return true;
    }
    return false;
  }
};

// ---------------------------------------------------------------- kernel

template <int ESIZE, int D, int G>
__global__ void __launch_bounds__(kThreads, (G <= 4 ? 3 : 2))
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
  using C = DecodeCfg<ESIZE, D, G>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  unsigned char* k_st = smem;
  unsigned char* v_st = k_st + kStages * C::STAGE_BYTES;
  float* p_s = reinterpret_cast<float*>(v_st + kStages * C::STAGE_BYTES);
  float* cmb_o = p_s + kConsumerWarps * C::RT * G;
  float* cmb_ml = cmb_o + kConsumerWarps * G * D;
  uint64_t* full = reinterpret_cast<uint64_t*>(cmb_ml + kConsumerWarps * G * 2);
  uint64_t* empty = full + kStages;
  long long* walk = reinterpret_cast<long long*>(empty + kStages);  // s, pre, W, chunk
  int32_t* tcache = reinterpret_cast<int32_t*>(walk + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int UR = B < C::TS ? B : C::TS;                  // rows per TMA box
  const int SB = B < C::TS ? C::TS / B : 1;              // boxes per stage
  const int STG = SB * UR;                               // tokens per stage
  const uint32_t box_bytes = (uint32_t)UR * D * ESIZE;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    fence_barrier_init();
  }
  // everything above touches only shared memory; global inputs (pool, q,
  // tables) may come from the previous grid in the stream
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 0) {
    WalkStart w = find_start(a.ctx, a.n_seq, B, a.n_kv_heads, a.max_blocks, a.grid, blockIdx.x,
                             a.status);
    if (blockIdx.x == 0) write_prefix(a.ctx, a.n_seq, B, a.n_kv_heads, a.max_blocks, a.ws_pre);
    if (lane == 0) {
      walk[0] = w.s;
      walk[1] = w.pre;
      walk[2] = w.W;
      walk[3] = w.chunk;
    }
  }
  __syncthreads();

  const long long W = walk[2], chunk = walk[3];
  PieceWalker pw;
  pw.ctx = a.ctx;
  pw.n_seq = a.n_seq;
  pw.B = B;
  pw.H = a.n_kv_heads;
  pw.max_blocks = a.max_blocks;
  pw.s = (int)walk[0];
  pw.pre = walk[1];
  pw.r = (long long)blockIdx.x * chunk;
  pw.r1 = pw.r + chunk < W ? pw.r + chunk : W;

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
    while (pw.next()) {
      const int tok_end = pw.b1 * B < pw.ctx_len ? pw.b1 * B : pw.ctx_len;
      for (int tok0 = pw.b0 * B; tok0 < tok_end; tok0 += STG) {
        const int slot = stage % kStages;
        if (stage >= kStages && alive) {
          if (!mbar_wait_bounded(&empty[slot], ((stage / kStages) & 1) ^ 1, kWaitLimitNs)) {
            alive = false;
            if (lane == 0) record_status(a.status, 8);
          }
        }
        const int nvalid = tok_end - tok0 < STG ? tok_end - tok0 : STG;
        const int nunits = (nvalid + UR - 1) / UR;
        tc.ensure(a.table, a.max_blocks, pw.seq, tok0 / B, (tok0 + (nunits - 1) * UR) / B, lane);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2u * nunits * box_bytes);
        __syncwarp();
        for (int u = lane; u < nunits; u += 32) {
          const int t = tok0 + u * UR;
          const int j = t / B;
          const int row = t - j * B;
          int pid = tc.ent[j - tc.base];
          if (pid < 0 || pid >= a.n_blocks) {
            record_status(a.status, 1);
            pid = 0;  // stay in bounds; the result is flagged as invalid
          }
          const int x = pw.head * D;
          const int y = (a.layer * a.n_blocks + pid) * B + row;
          tma_load_2d(k_st + slot * C::STAGE_BYTES + u * box_bytes, &tmap_k, x, y, &full[slot]);
          tma_load_2d(v_st + slot * C::STAGE_BYTES + u * box_bytes, &tmap_v, x, y, &full[slot]);
        }
        ++stage;
      }
    }
    // drain: do not leave while copies into this CTA's shared memory are in flight
    const int first = stage > kStages ? stage - kStages : 0;
    for (int k = first; k < stage; ++k)
      mbar_wait_bounded(&full[k % kStages], (k / kStages) & 1, kWaitLimitNs);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int grp = lane >> C::LT;              // token within a step
  const int li = lane & (C::TG - 1);          // lane within the token group
  const int ctid = threadIdx.x;               // 0 .. 127
  float* my_p = p_s + warp * C::RT * G;
  bool alive = true;
  int stage = 0;

  while (pw.next()) {
    // query heads h*G .. h*G+G-1 of this sequence, scaled, as float2 pairs
    float2 q2[G][C::VEC / 2];
    {
      const unsigned char* qb = reinterpret_cast<const unsigned char*>(a.q) +
                                ((long long)pw.seq * a.n_q_heads + (long long)pw.head * G) * D * ESIZE;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint4 w = *reinterpret_cast<const uint4*>(qb + (g * D + li * C::VEC) * ESIZE);
        cvt16(w, q2[g]);
#pragma unroll
        for (int j = 0; j < C::VEC / 2; ++j) {
          q2[g][j].x *= a.qscale;
          q2[g][j].y *= a.qscale;
        }
      }
    }
    float m_run[G], l_run[G];
    float2 o2[G][C::VEC / 2];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.f;
#pragma unroll
      for (int j = 0; j < C::VEC / 2; ++j) o2[g][j] = make_float2(0.f, 0.f);
    }

    const int tok_end = pw.b1 * B < pw.ctx_len ? pw.b1 * B : pw.ctx_len;
    for (int tok0 = pw.b0 * B; tok0 < tok_end; tok0 += STG) {
      const int slot = stage % kStages;
      if (alive && !mbar_wait_bounded(&full[slot], (stage / kStages) & 1, kWaitLimitNs)) {
        alive = false;
        if (lane == 0) record_status(a.status, 8);
      }
      alive = __all_sync(0xffffffffu, alive);  // reconverge after the poll loop
      const int nvalid = tok_end - tok0 < STG ? tok_end - tok0 : STG;
      const unsigned char* ks = k_st + slot * C::STAGE_BYTES;
      const unsigned char* vs = v_st + slot * C::STAGE_BYTES;
      const int nrounds = (nvalid + C::RT - 1) / C::RT;
      for (int rd = warp; rd < nrounds; rd += kConsumerWarps) {
        const int rbase = rd * C::RT;
        // ---- scores: 4 steps x G heads of partial dot products
        float acc[C::V];
#pragma unroll
        for (int st = 0; st < C::S; ++st) {
          const int row = rbase + st * C::NG + grp;
          const uint4 w = *reinterpret_cast<const uint4*>(ks + (row * D + li * C::VEC) * ESIZE);
          float2 kf[C::VEC / 2];
          cvt16(w, kf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < C::VEC / 2; ++j) s2 = __ffma2_rn(q2[g][j], kf[j], s2);
            acc[st * G + g] = s2.x + s2.y;
          }
        }
        TReduce<C::V, C::TG / 2>::run(acc, li);
        // ---- mask, round max per head
        float sc[C::HV], mx[C::HV];
#pragma unroll
        for (int k = 0; k < C::HV; ++k) {
          const int i = held_index<C>(li, k);
          const int row = rbase + (i / G) * C::NG + grp;
          sc[k] = row < nvalid ? acc[k] : -INFINITY;
          mx[k] = sc[k];
#pragma unroll
          for (int b = C::LT - C::LS; b < 5; ++b)
            mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 1 << b));
        }
        float alpha[G], mnew[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          int src, kk;
          if constexpr (C::V >= C::TG) {
            src = g / (C::V / C::TG);
            kk = g % (C::V / C::TG);
          } else {
            src = g << (C::LT - C::LV);
            kk = 0;
          }
          float rm = 0.f;
#pragma unroll
          for (int k = 0; k < C::HV; ++k) {
            const float t = __shfl_sync(0xffffffffu, mx[k], src);
            if (k == kk) rm = t;
          }
          mnew[g] = fmaxf(m_run[g], rm);
          alpha[g] = exp2_approx(m_run[g] - mnew[g]);
          m_run[g] = mnew[g];
        }
        // ---- probabilities to shared memory
        const bool owner = (C::V >= C::TG) || ((li & ((1 << (C::LT - C::LV)) - 1)) == 0);
#pragma unroll
        for (int k = 0; k < C::HV; ++k) {
          const int i = held_index<C>(li, k);
          const int g = i % G;
          float mg = mnew[0];
#pragma unroll
          for (int gg = 1; gg < G; ++gg)
            if (gg == g) mg = mnew[gg];
          const float p = exp2_approx(sc[k] - mg);
          if (owner) my_p[((i / G) * C::NG + grp) * G + g] = p;
        }
        __syncwarp();
        // ---- rescale and P.V
#pragma unroll
        for (int g = 0; g < G; ++g) {
          l_run[g] *= alpha[g];
          const float2 a2 = make_float2(alpha[g], alpha[g]);
#pragma unroll
          for (int j = 0; j < C::VEC / 2; ++j) o2[g][j] = __fmul2_rn(o2[g][j], a2);
        }
#pragma unroll
        for (int st = 0; st < C::S; ++st) {
          const int rr = st * C::NG + grp;
          const int row = rbase + rr;
          if (row < nvalid) {
            const uint4 w = *reinterpret_cast<const uint4*>(vs + (row * D + li * C::VEC) * ESIZE);
            float2 vf[C::VEC / 2];
            cvt16(w, vf);
            float p[G];
#pragma unroll
            for (int g = 0; g < G; ++g) p[g] = my_p[rr * G + g];
#pragma unroll
            for (int g = 0; g < G; ++g) {
              l_run[g] += p[g];
              const float2 p2 = make_float2(p[g], p[g]);
#pragma unroll
              for (int j = 0; j < C::VEC / 2; ++j) o2[g][j] = __ffma2_rn(p2, vf[j], o2[g][j]);
            }
          }
        }
        __syncwarp();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++stage;
    }

    // ---- combine the 4 warps' states for this piece
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int b = C::LT; b < 5; ++b) {
        l_run[g] += __shfl_xor_sync(0xffffffffu, l_run[g], 1 << b);
#pragma unroll
        for (int j = 0; j < C::VEC / 2; ++j) {
          o2[g][j].x += __shfl_xor_sync(0xffffffffu, o2[g][j].x, 1 << b);
          o2[g][j].y += __shfl_xor_sync(0xffffffffu, o2[g][j].y, 1 << b);
        }
      }
    }
    if (grp == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float* dst = cmb_o + (warp * G + g) * D + li * C::VEC;
#pragma unroll
        for (int j = 0; j < C::VEC / 2; ++j) {
          dst[2 * j] = o2[g][j].x;
          dst[2 * j + 1] = o2[g][j].y;
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        cmb_ml[(warp * G + g) * 2] = m_run[g];
        cmb_ml[(warp * G + g) * 2 + 1] = l_run[g];
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);
    const long long slot_id = (long long)blockIdx.x + (long long)pw.seq * a.n_kv_heads + pw.head;
    for (int idx = ctid; idx < G * D; idx += kConsumerWarps * 32) {
      const int g = idx / D, d = idx - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cmb_ml[(w * G + g) * 2]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = cmb_ml[(w * G + g) * 2];
        const float f = mw == -INFINITY ? 0.f : exp2_approx(mw - M);
        L += f * cmb_ml[(w * G + g) * 2 + 1];
        O += f * cmb_o[(w * G + g) * D + d];
      }
      a.ws_o[(slot_id * G + g) * D + d] = O;
      if (d == 0) {
        a.ws_ml[(slot_id * G + g) * 2] = M;
        a.ws_ml[(slot_id * G + g) * 2 + 1] = L;
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);
  }
}

}  // namespace pkv
