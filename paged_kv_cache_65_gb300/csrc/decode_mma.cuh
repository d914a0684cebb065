// Split-K paged decode attention, partial pass, bfloat16 K/V on tensor cores.
//
// Same contract, work split and workspace as decode.cuh (see there): per
// (sequence, K/V head, block range) it emits the base-2 online-softmax
// statistics m, l and the unnormalised O for the G query heads of the group.
//
// The two products of a 16-token tile are small MMAs over the query group
// (m16n8k16, bf16 in, f32 accumulate):
//     S^T [16 tokens x 8 heads] = K [16 x D] . Q^T [D x 8]       (D/16 MMAs)
//     O^T [D x 8 heads]        += V^T [D x 16] . P^T [16 x 8]     (2 x D/16)
// K and V^T come straight from shared memory with ldmatrix (V transposed on
// load), Q^T lives in registers for the whole piece, and P^T is the S^T
// accumulator turned into bf16 and transposed inside the warp with movmatrix.
// P is split into a bf16 high part and a bf16 remainder (two MMAs) so that
// the weights keep ~16 mantissa bits.  Query heads beyond G are zero padding.
//
// Shared memory: each stage holds TS token rows of K and of V for one K/V
// head (64 tokens at D = 128), written by TMA with the 128-byte swizzle (rows
// of 64 elements, the 16-byte chunk c of row r stored at chunk c ^ (r mod 8)),
// so the 8 rows an ldmatrix phase reads fall in 8 different bank groups.  All
// four consumer warps consume every stage, warp w taking its 16-token tile(s)
// with its own running softmax state; the four states are merged through
// shared memory at the end of each piece.
#pragma once

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

// Tokens per stage of the tensor-core pass: one 16-token tile per consumer
// warp (16 KiB of K and 16 KiB of V at D = 128).
constexpr int mma_stage_tokens(int D) { return 16 * 4 * (D == 64 ? 2 : 1); }

template <int D, int G>
struct MmaCfg {
  static constexpr int TS = mma_stage_tokens(D);  // tokens per stage
  static constexpr int TPW = TS / 16 / kConsumerWarps;  // tiles per warp per stage
  static constexpr int KS = D / 16;               // k-steps of Q.K and m-tiles of O^T
  static constexpr int HALVES = D / 64;           // 64-element swizzled row halves
  static constexpr int HALF_BYTES = TS * 128;     // one half of a K (or V) stage
  static constexpr int STAGE_BYTES = TS * D * 2;  // K (or V) per stage
  static constexpr int NST = 3;                   // stages in the ring
  static constexpr int GC = G < 4 ? G : 4;        // heads per combine pass
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(G >= 1 && G <= 8, "group size");
  static_assert(TS % (16 * kConsumerWarps) == 0, "whole tiles per warp");
};

template <int D, int G>
constexpr int decode_mma_smem_bytes() {
  using C = MmaCfg<D, G>;
  return 2 * C::NST * C::STAGE_BYTES        // K and V stages
         + kConsumerWarps * C::GC * D * 4   // combine: O per warp, GC heads at a time
         + kConsumerWarps * G * 2 * 4       // combine: m, l per warp
         + 2 * C::NST * 8                   // mbarriers
         + kTableCache * 4                  // producer table cache
         + 64 + 1024;                       // walk state + 1 KiB alignment
}

// swizzled shared address of (row r, 8-element chunk c) inside a half
__device__ __forceinline__ uint32_t swz(uint32_t half_base, int r, int c) {
  return half_base + r * 128 + ((c ^ (r & 7)) << 4);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
  using C = MmaCfg<D, G>;
  constexpr int NST = C::NST;
  // the declared alignment stays at 16 so that the explicit round-up to the
  // 1 KiB the 128-byte swizzle needs is never folded away
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* k_st = smem;
  unsigned char* v_st = k_st + NST * C::STAGE_BYTES;
  float* cmb_o = reinterpret_cast<float*>(v_st + NST * C::STAGE_BYTES);
  float* cmb_ml = cmb_o + kConsumerWarps * C::GC * D;
  uint64_t* full = reinterpret_cast<uint64_t*>(cmb_ml + kConsumerWarps * G * 2);
  uint64_t* empty = full + NST;
  long long* walk = reinterpret_cast<long long*>(empty + NST);
  int32_t* tcache = reinterpret_cast<int32_t*>(walk + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int UR = B < C::TS ? B : C::TS;      // rows per TMA box (a multiple of 8)
  const int SB = B < C::TS ? C::TS / B : 1;  // boxes per stage
  const int STG = SB * UR;                   // tokens per stage
  const uint32_t unit_bytes = (uint32_t)UR * D * 2;  // K (or V) bytes of one box row set

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
    fence_barrier_init();
  }
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
        const int slot = stage % NST;
        if (stage >= NST && alive) {
          if (!mbar_wait_bounded(&empty[slot], ((stage / NST) & 1) ^ 1, kWaitLimitNs)) {
            alive = false;
            if (lane == 0) record_status(a.status, 8);
          }
        }
        const int nvalid = tok_end - tok0 < STG ? tok_end - tok0 : STG;
        const int nunits = (nvalid + UR - 1) / UR;
        tc.ensure(a.table, a.max_blocks, pw.seq, tok0 / B, (tok0 + (nunits - 1) * UR) / B, lane);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2u * nunits * unit_bytes);
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
          const int y = (a.layer * a.n_blocks + pid) * B + row;
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h) {
            const int x = pw.head * D + h * 64;
            const int off = slot * C::STAGE_BYTES + h * C::HALF_BYTES + u * UR * 128;
            tma_load_2d(k_st + off, &tmap_k, x, y, &full[slot]);
            tma_load_2d(v_st + off, &tmap_v, x, y, &full[slot]);
          }
        }
        ++stage;
      }
    }
    const int first = stage > NST ? stage - NST : 0;
    for (int k = first; k < stage; ++k)
      mbar_wait_bounded(&full[k % NST], (k / NST) & 1, kWaitLimitNs);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;  // groupID: row of A / C, column of B
  const int t = lane & 3;   // thread in group
  const uint32_t k_base = smem_u32(k_st);
  const uint32_t v_base = smem_u32(v_st);
  bool alive = true;
  int stage = 0;

  while (pw.next()) {
    // Q^T fragments: head g of the group, dims ks*16 + 2t (+1) and + 8
    uint32_t qf[C::KS][2];
    {
      const uint32_t* qw = reinterpret_cast<const uint32_t*>(
          reinterpret_cast<const unsigned char*>(a.q) +
          ((long long)pw.seq * a.n_q_heads + (long long)pw.head * G + (g < G ? g : 0)) * D * 2);
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        qf[ks][0] = g < G ? qw[(ks * 16 + 2 * t) / 2] : 0u;
        qf[ks][1] = g < G ? qw[(ks * 16 + 2 * t + 8) / 2] : 0u;
      }
    }
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[C::KS][4];
#pragma unroll
    for (int mt = 0; mt < C::KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    const int tok_end = pw.b1 * B < pw.ctx_len ? pw.b1 * B : pw.ctx_len;
    for (int tok0 = pw.b0 * B; tok0 < tok_end; tok0 += STG, ++stage) {
      // every consumer warp waits on every stage and takes its own tiles of it
      const int slot = stage % NST;
      if (alive && !mbar_wait_bounded(&full[slot], (stage / NST) & 1, kWaitLimitNs)) {
        alive = false;
        if (lane == 0) record_status(a.status, 8);
      }
      alive = __all_sync(0xffffffffu, alive);  // reconverge before ldmatrix / mma.sync
      const int nvalid = tok_end - tok0 < STG ? tok_end - tok0 : STG;
      const uint32_t kb = k_base + slot * C::STAGE_BYTES;
      const uint32_t vb = v_base + slot * C::STAGE_BYTES;
#pragma unroll 1
      for (int tw = 0; tw < C::TPW; ++tw) {
        const int tt = tw * kConsumerWarps + warp;
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
#pragma unroll
          for (int i = 0; i < 4; ++i) s[i] += s2[i];
        }
        // ---- scale, mask, tile max per head (heads 2t, 2t+1; tokens g, g+8)
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
        // ---- P^T fragments: bf16 high part and remainder, transposed
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
        const int nv = nvalid - tt * 16;
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (nv < 16) {
          mlo = (2 * t < nv ? 0x0000ffffu : 0u) | (2 * t + 1 < nv ? 0xffff0000u : 0u);
          mhi = (2 * t + 8 < nv ? 0x0000ffffu : 0u) | (2 * t + 9 < nv ? 0xffff0000u : 0u);
        }
        {
          const int r = tt * 16 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
          for (int mt = 0; mt < C::KS; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
            const int d0 = mt * 16 + ((lane >> 3) & 1) * 8;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(swz(vb + (d0 >> 6) * C::HALF_BYTES, r, (d0 & 63) >> 3), a0, a1, a2, a3);
            a0 &= mlo;
            a1 &= mlo;
            a2 &= mhi;
            a3 &= mhi;
            mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
            mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ---- combine the 4 warps' states for this piece
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
      l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
    }
    if (g == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int h = 2 * t + k;
        if (h < G) {
          cmb_ml[(warp * G + h) * 2] = m_run[k];
          cmb_ml[(warp * G + h) * 2 + 1] = l_run[k];
        }
      }
    }
    const long long slot_id = (long long)blockIdx.x + (long long)pw.seq * a.n_kv_heads + pw.head;
#pragma unroll
    for (int h0 = 0; h0 < G; h0 += C::GC) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int h = 2 * t + k;
        if (h >= h0 && h < h0 + C::GC) {
#pragma unroll
          for (int mt = 0; mt < C::KS; ++mt) {
            cmb_o[(warp * C::GC + h - h0) * D + mt * 16 + g] = o[mt][k];
            cmb_o[(warp * C::GC + h - h0) * D + mt * 16 + g + 8] = o[mt][2 + k];
          }
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
      for (int idx = threadIdx.x; idx < C::GC * D; idx += kConsumerWarps * 32) {
        const int hh = idx / D, d = idx - hh * D;
        const int h = h0 + hh;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cmb_ml[(w * G + h) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float mw = cmb_ml[(w * G + h) * 2];
          const float f = mw == -INFINITY ? 0.f : exp2_approx(mw - M);
          L += f * cmb_ml[(w * G + h) * 2 + 1];
          O += f * cmb_o[(w * C::GC + hh) * D + d];
        }
        a.ws_o[(slot_id * G + h) * D + d] = O;
        if (d == 0) {
          a.ws_ml[(slot_id * G + h) * 2] = M;
          a.ws_ml[(slot_id * G + h) * 2 + 1] = L;
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
    }
  }
}

}  // namespace pkv
