// Decode plan: the work list of a sharing-aware decode pass, built on the
// host from the block manager's tables and uploaded to the device as-is.
//
// A segment is a block range of one sequence's table and one K/V head, read
// once, whose query columns belong to one or more member sequences (G query
// heads of the K/V head per member).  Sequences whose tables share leading
// full blocks get one segment per head for that shared prefix (all members'
// columns) and one private segment per head for the rest; the merge entries
// list, per (sequence, K/V head), the segments and column offsets whose
// partials make up that sequence's softmax.
//
// Work units: block j of a segment occupies units [wpre + j*w, wpre + (j+1)*w);
// the split pass gives CTA c the units [c*chunk, (c+1)*chunk) and with them
// the blocks whose first unit falls in that range (possibly none: the CTA then
// writes an empty partial, m = -inf, l = 0).  The CTAs holding pieces of a
// segment are wpre / chunk .. (wpre + len*w - 1) / chunk.
#pragma once

#include <cstdint>

struct PlanHeader {
  int64_t W;          // total work units over all segments
  int32_t n_segs;
  int32_t n_members;
  int32_t n_entries;
  int32_t c_max;      // largest column count of a segment (a multiple of G, <= 32)
  int32_t n_seq;      // listed sequences (rows of the block table)
  int32_t n_kv_heads;
  int32_t group;      // G = H_q / H_kv
  int32_t block_size;
  int32_t seg_off;    // byte offsets from the start of the plan
  int32_t mem_off;
  int32_t eoff_off;
  int32_t ent_off;
  int32_t n_shared_segs;
  int32_t kernel;     // split-pass kernel the work units are weighted for (kPlanKernel*)
  int32_t start_off;  // byte offset of the CTA start records (0: none)
  int32_t start_grid; // CTA count the start records were built for (0: none)
  int32_t pad[2];
};
static_assert(sizeof(PlanHeader) == 80, "plan header layout");

struct PlanSeg {
  int64_t wpre;     // work units of all segments before this one
  int32_t rep;      // table row (listed sequence index) the blocks come from
  int32_t b0, b1;   // blocks [b0, b1) of that row
  int32_t tok_end;  // tokens at or past this position are not read
  int32_t head;     // K/V head
  int32_t ncols;    // query columns: members * G
  int32_t mem;      // index of the first member in the member list
  int32_t w;        // work units per block (cost weight of the segment's width)
};
static_assert(sizeof(PlanSeg) == 40, "plan segment layout");

// Start record of CTA c of a split pass launched with start_grid CTAs: the
// first piece PlanWalker::next yields from the CTA's first work unit, the
// walk position after it, and the physical ids of the piece's first blocks
// (the table entries of row `rep` from b0 on), so that the CTA's first copies
// need neither a search of the segments nor a block-table read.
constexpr int kPlanStartPids = 16;
struct PlanStart {
  int32_t seg;      // segment of the first piece; -1: the CTA has no work unit
  int32_t rep, head, b0, b1, tok_end, ncols, mem;
  int64_t r_after;  // work unit after the first piece
  int32_t n_pid;    // valid entries of pid (blocks b0 .. b0 + n_pid - 1)
  int32_t last;     // 1: the piece holds the segment's last block
  int32_t pid[kPlanStartPids];
  int32_t pad1[4];
};
static_assert(sizeof(PlanStart) == 128, "plan start record layout");

struct PlanEntry {
  int32_t seg;       // segment holding partials of this (sequence, head)
  int32_t col_base;  // the sequence's first column in that segment
};

// Most query columns one segment carries (four 8-column MMA n-tiles).
constexpr int kPlanMaxCols = 32;

// Most shared runs one sequence is read through (nested forks beyond this
// depth are read privately).
constexpr int kPlanMaxLevels = 3;

// Most segments a plan of n_seq sequences can hold.
constexpr int plan_max_segs(int n_seq, int n_kv_heads) {
  return (n_seq + (kPlanMaxLevels * n_seq + 1) / 2) * n_kv_heads;
}

// Split-pass kernels a plan can be built for (the values of the pool's
// decode-path option).
constexpr int kPlanKernelMma = 2;  // warp-level MMA (mma.sync)
constexpr int kPlanKernelTc = 3;   // tcgen05, TMEM accumulators

// Work units per block.  The split pass balances units.  On the warp-level
// MMA kernel a block costs more the more 8-column n-tiles it carries (1, 2,
// 3-4 tiles: 3, 4, 5 parts), so blocks of wide shared segments are spread
// over more CTAs; on the tcgen05 kernel the tensor work is small against the
// block's bytes, and only the 32-column softmax adds to a block's time
// (4, 4, 5 parts).  A part is 8 units.
constexpr int kPlanUnitsPerPart = 8;
constexpr int plan_block_weight(int ncols, int kernel) {
  return kPlanUnitsPerPart * (kernel == kPlanKernelTc ? (ncols <= 16 ? 4 : 5)
                                                      : (ncols <= 8 ? 3 : (ncols <= 16 ? 4 : 5)));
}
// Fixed cost of a piece (its start and its partials), in units: about one
// pipeline stage of narrow blocks on the warp-level pass (64 tokens), four
// on tcgen05 (4 x 128 tokens: a piece there also waits for its Q tile and
// for the previous piece's O^T readout; found by timing 1, 2 and 4).  Each segment carries it spread over
// its blocks, so a CTA whose range holds many short segments (the one-block
// private tails of forked branches) is given fewer blocks.
constexpr int plan_piece_units(int kernel) {
  return kernel == kPlanKernelTc ? 32 * plan_block_weight(8, kernel)
                                 : 4 * plan_block_weight(8, kernel);
}
// Units per block of a segment of n_blocks blocks.
constexpr int plan_seg_weight(int ncols, int kernel, int n_blocks) {
  return plan_block_weight(ncols, kernel) +
         (n_blocks > 0 ? (plan_piece_units(kernel) + n_blocks - 1) / n_blocks : 0);
}
