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
#pragma once

#include <cstdint>

struct PlanHeader {
  int64_t W;          // total blocks over all segments
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
  int32_t pad[5];
};
static_assert(sizeof(PlanHeader) == 80, "plan header layout");

struct PlanSeg {
  int64_t wpre;     // blocks of all segments before this one
  int32_t rep;      // table row (listed sequence index) the blocks come from
  int32_t b0, b1;   // blocks [b0, b1) of that row
  int32_t tok_end;  // tokens at or past this position are not read
  int32_t head;     // K/V head
  int32_t ncols;    // query columns: members * G
  int32_t mem;      // index of the first member in the member list
  int32_t pad;
};
static_assert(sizeof(PlanSeg) == 40, "plan segment layout");

struct PlanEntry {
  int32_t seg;       // segment holding partials of this (sequence, head)
  int32_t col_base;  // the sequence's first column in that segment
};

// Most query columns one segment carries (four 8-column MMA n-tiles).
constexpr int kPlanMaxCols = 32;
