// Host builder of the sharing-aware decode plan (see plan.h).
//
// Prefix sharing comes from fork (one table copied into another, "KV 缓存管理",
// zero-copy branching section) and from shared prompts ("第 8 章 推理优化"
// §8.3.2): the blocks stay shared until a write into a partly filled tail
// copies it.  Decode attention only reads, so every block that several
// listed sequences' tables name at the same logical position, within all of
// their contexts, can be read once for all of them.
//
// Grouping: listed sequences are grouped by the physical id of their first
// block; a group's shared prefix is the longest run of leading blocks common
// to all members, cut to whole blocks inside every member's context.  Groups
// wider than kPlanMaxCols / G members are cut into sub-groups (each reads the
// prefix once).  Prefixes shorter than `min_shared_tokens` are not shared.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "plan.h"
#include "pool.h"

namespace {

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Length of the common prefix of a[0, n) and b[0, n): 64 entries at a time
// with memcmp, then entry by entry.
int common_prefix(const int32_t* a, const int32_t* b, int n) {
  constexpr int kRun = 64;
  int j = 0;
  while (j + kRun <= n && std::memcmp(a + j, b + j, kRun * sizeof(int32_t)) == 0) j += kRun;
  while (j < n && a[j] == b[j]) ++j;
  return j;
}

struct Layout {
  size_t seg, mem, eoff, ent, start, total;
};

Layout plan_layout(int n_seq, int H, int n_segs, int n_members, int n_entries, int n_start) {
  Layout l;
  size_t off = align16(sizeof(PlanHeader));
  l.seg = off;
  off += align16(sizeof(PlanSeg) * static_cast<size_t>(n_segs));
  l.mem = off;
  off += align16(sizeof(int32_t) * static_cast<size_t>(n_members));
  l.eoff = off;
  off += align16(sizeof(int32_t) * (static_cast<size_t>(n_seq) * H + 1));
  l.ent = off;
  off += align16(sizeof(PlanEntry) * static_cast<size_t>(n_entries));
  l.start = off;
  off += sizeof(PlanStart) * static_cast<size_t>(n_start);
  l.total = off;
  return l;
}

// CTA count of the split pass for the plan's kernel: the count the launcher
// has settled on for this pool, else the kernel's design occupancy (two CTAs
// per SM for the warp-level MMA pass, one for the tcgen05 pass) once the
// device is known, else 0 (no start records).  A record set built for another
// count than the launch's is ignored by the kernels.
int plan_grid(const kvPool* p, int kernel, int G) {
  if (p->plan_grid > 0) return p->plan_grid < kMaxDecodeCtas ? p->plan_grid : kMaxDecodeCtas;
  int g = 0;
  if (kernel == kPlanKernelTc) {
    g = p->grid_tc > 0 ? p->grid_tc : pool_sm_count(p);
  } else {
    const int lg = G <= 1 ? 0 : (G == 2 ? 1 : (G == 4 ? 2 : 3));
    g = p->grid_by_g[lg] > 0 ? p->grid_by_g[lg] : 2 * pool_sm_count(p);
  }
  return g < kMaxDecodeCtas ? g : kMaxDecodeCtas;
}

// Start records for `grid` CTAs, following the device's split exactly: CTA c
// takes the work units [c * chunk, min((c + 1) * chunk, W)), chunk =
// ceil(W / grid) (at least 1); its walk starts at the last segment whose
// first unit is at or before c * chunk and yields the pieces PlanWalker::next
// does.
void plan_starts(const std::vector<PlanSeg>& segs, int64_t W, int grid, int B,
                 const std::vector<const kvSeq*>& seqs, PlanStart* out) {
  int64_t chunk = (W + grid - 1) / grid;
  if (chunk == 0) chunk = 1;
  const int n = static_cast<int>(segs.size());
  int lo = 0;  // last segment with wpre <= r0; r0 grows with c, so lo only moves on
  for (int c = 0; c < grid; ++c) {
    PlanStart& R = out[c];
    std::memset(&R, 0, sizeof(R));
    R.seg = -1;
    const int64_t r0 = static_cast<int64_t>(c) * chunk;
    if (r0 >= W) continue;
    const int64_t r1 = std::min(r0 + chunk, W);
    while (lo + 1 < n && segs[lo + 1].wpre <= r0) ++lo;
    for (int s = lo; s < n; ++s) {
      const PlanSeg& sg = segs[s];
      const int64_t len = sg.b1 - sg.b0;
      const int64_t w = sg.w > 0 ? sg.w : 1;
      if (len <= 0 || r0 >= sg.wpre + len * w) continue;
      const int64_t end = std::min(r1, sg.wpre + len * w);
      const int64_t jb = (r0 - sg.wpre + w - 1) / w, je = (end - sg.wpre + w - 1) / w;
      R.seg = s;
      R.rep = sg.rep;
      R.head = sg.head;
      R.b0 = sg.b0 + static_cast<int32_t>(jb);
      R.b1 = sg.b0 + static_cast<int32_t>(je);
      R.tok_end = static_cast<int32_t>(std::min<int64_t>(static_cast<int64_t>(R.b1) * B, sg.tok_end));
      R.ncols = sg.ncols;
      R.mem = sg.mem;
      R.last = R.b1 == sg.b1 ? 1 : 0;
      R.r_after = end;
      const std::vector<int32_t>& t = seqs[sg.rep]->table;
      int k = 0;
      for (; k < kPlanStartPids && R.b0 + k < R.b1 && R.b0 + k < static_cast<int>(t.size()); ++k)
        R.pid[k] = t[R.b0 + k];
      R.n_pid = k;
      break;
    }
  }
}

// Working arrays of the plan builder, kept per thread so that a step's plan
// reuses the previous one's allocations.
struct PlanScratch {
  std::vector<const kvSeq*> seqs;
  std::vector<int32_t> sorted;
  std::vector<int> n_levels, priv_from, priv_mem, node_mem0, ungrouped, order;
  std::vector<char> grouped;
  std::vector<PlanSeg> segs;
  std::vector<int32_t> members;
  std::vector<PlanEntry> entk;
  std::vector<uint8_t> n_ent;
};
thread_local PlanScratch t_scratch;

}  // namespace

size_t plan_workspace_bytes(int n_segs, int c_max, int D) {
  const size_t n_slots = static_cast<size_t>(kMaxDecodeCtas) + static_cast<size_t>(n_segs);
  const size_t ml = (n_slots * c_max * 2 * sizeof(float) + 255) & ~size_t(255);
  return ml + n_slots * c_max * D * sizeof(float);
}

extern "C" {

size_t paged_decode_plan_bytes(const kvPool* p, int n_seq, int n_q_heads) {
  if (!p || n_seq < 0 || n_q_heads <= 0 || n_q_heads % p->H != 0) return 0;
  // per (sequence, head) at most kPlanMaxLevels shared runs and one private
  // rest (a shared run has two or more members, so there are at most
  // kPlanMaxLevels * n_seq / 2 of them per head), member slots and entries
  // to match; start records for the larger of the two kernels' CTA counts
  const int G = n_q_heads / p->H;
  const int n_start = std::max(plan_grid(p, kPlanKernelMma, G), plan_grid(p, kPlanKernelTc, G));
  const int segs_max = plan_max_segs(n_seq, p->H);
  const int mem_max = (kPlanMaxLevels + 1) * n_seq;
  return plan_layout(n_seq, p->H, segs_max, mem_max, (kPlanMaxLevels + 1) * n_seq * p->H,
                     n_start).total;
}

kvStatus paged_decode_plan(const kvPool* p, const int32_t* seq_ids, int n_seq, int n_q_heads,
                           int max_blocks, int min_shared_tokens, void* h_plan, size_t plan_bytes,
                           size_t* out_workspace_bytes) {
  return plan_build(p, seq_ids, n_seq, n_q_heads, max_blocks, min_shared_tokens, h_plan,
                    plan_bytes, out_workspace_bytes, true);
}

}  // extern "C"

kvStatus plan_build(const kvPool* p, const int32_t* seq_ids, int n_seq, int n_q_heads,
                    int max_blocks, int min_shared_tokens, void* h_plan, size_t plan_bytes,
                    size_t* out_workspace_bytes, bool start_records) {
  if (!p || n_seq < 0 || (n_seq > 0 && !seq_ids) || !h_plan || max_blocks <= 0)
    return KV_ERR_INVALID_ARG;
  if (n_q_heads <= 0 || n_q_heads % p->H != 0) return KV_ERR_INVALID_ARG;
  const int H = p->H, B = p->B, G = n_q_heads / H;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KV_ERR_UNSUPPORTED;
  if (plan_bytes < paged_decode_plan_bytes(p, n_seq, n_q_heads)) return KV_ERR_INVALID_ARG;
  if (min_shared_tokens <= 0) min_shared_tokens = 128;
  PlanScratch& sc = t_scratch;
  std::vector<const kvSeq*>& seqs = sc.seqs;
  seqs.assign(n_seq, nullptr);
  {
    std::vector<int32_t>& sorted = sc.sorted;
    sorted.assign(seq_ids, seq_ids + n_seq);
    std::sort(sorted.begin(), sorted.end());
    if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return KV_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_seq; ++i) {
    auto it = p->seqs.find(seq_ids[i]);
    if (it == p->seqs.end()) return KV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(it->second.table.size()) > max_blocks) return KV_ERR_INVALID_ARG;
    if (it->second.len > static_cast<int64_t>(max_blocks) * B) return KV_ERR_INVALID_ARG;
    seqs[i] = &it->second;
  }
  const int max_members = kPlanMaxCols / G;
  // whole blocks of a sequence inside its context (a shared run never
  // reaches into a partly filled block)
  auto full_blocks = [&](int i) {
    return static_cast<int>(std::min<int64_t>(static_cast<int64_t>(seqs[i]->table.size()),
                                              seqs[i]->len / B));
  };

  // ---- shared runs, found like a radix walk over the listed tables: the
  // sequences with the same first physical block form a group; a group's
  // common run from its start s0 is read once for all of its members when it
  // is at least min_shared_tokens long (members cut into sub-groups of at
  // most max_members, equal in size); after the run, the members are split
  // by their next physical block and each part with two or more members goes
  // on from there (a branch that forked deeper in a shared prompt shares
  // that deeper run with its siblings).  A run too short to share is read
  // privately, and the parts continue from the same start.  A sequence joins
  // at most kPlanMaxLevels shared runs.
  struct Node {
    std::vector<int> mem;  // members, ascending
    int b0, b1;            // the run of blocks [b0, b1)
  };
  std::vector<Node> nodes;
  std::vector<int>& n_levels = sc.n_levels;    // shared runs each sequence has joined
  std::vector<int>& priv_from = sc.priv_from;  // first block read privately
  n_levels.assign(n_seq, 0);
  priv_from.assign(n_seq, 0);
  std::vector<int> roots;  // first node of each root group
  auto run_group = [&](auto&& self, std::vector<int> mem, int s0) -> void {
    // common run from s0 among the members
    int P = full_blocks(mem[0]);
    const std::vector<int32_t>& t0 = seqs[mem[0]]->table;
    for (size_t k = 1; k < mem.size() && P > s0; ++k) {
      const std::vector<int32_t>& t = seqs[mem[k]]->table;
      P = std::min(P, full_blocks(mem[k]));
      if (P > s0) P = s0 + common_prefix(t0.data() + s0, t.data() + s0, P - s0);
    }
    if (P < s0) P = s0;
    int next_s0 = s0;
    bool room = true;
    for (int m : mem) room = room && n_levels[m] < kPlanMaxLevels;
    if (room && static_cast<int64_t>(P - s0) * B >= min_shared_tokens) {
      const int n_sub = static_cast<int>((mem.size() + max_members - 1) / max_members);
      size_t c0 = 0;
      for (int c = 0; c < n_sub; ++c) {
        const size_t c1 = c0 + (mem.size() - c0) / static_cast<size_t>(n_sub - c);
        Node nd;
        nd.mem.assign(mem.begin() + static_cast<long>(c0), mem.begin() + static_cast<long>(c1));
        nd.b0 = s0;
        nd.b1 = P;
        for (int m : nd.mem) {
          n_levels[m] += 1;
          priv_from[m] = P;
        }
        nodes.push_back(std::move(nd));
        c0 = c1;
      }
      next_s0 = P;
    }
    // the members that go on past P, split by their block there
    std::vector<int> more;
    for (int m : mem)
      if (full_blocks(m) > P) more.push_back(m);
    std::stable_sort(more.begin(), more.end(), [&](int x, int y) {
      return seqs[x]->table[P] < seqs[y]->table[P];
    });
    for (size_t a0 = 0; a0 < more.size();) {
      size_t b0 = a0 + 1;
      while (b0 < more.size() && seqs[more[b0]]->table[P] == seqs[more[a0]]->table[P]) ++b0;
      if (b0 - a0 >= 2) {
        std::vector<int> part(more.begin() + static_cast<long>(a0),
                              more.begin() + static_cast<long>(b0));
        std::sort(part.begin(), part.end());
        self(self, std::move(part), next_s0);
      }
      a0 = b0;
    }
  };
  {
    std::vector<int>& order = sc.order;
    order.clear();
    for (int i = 0; i < n_seq; ++i)
      if (full_blocks(i) > 0) order.push_back(i);
    // by first block, listing order among equals (a stable sort without its
    // temporary buffer)
    std::sort(order.begin(), order.end(), [&](int x, int y) {
      const int32_t bx = seqs[x]->table[0], by = seqs[y]->table[0];
      return bx < by || (bx == by && x < y);
    });
    for (size_t a0 = 0; a0 < order.size();) {
      size_t b0 = a0 + 1;
      while (b0 < order.size() && seqs[order[b0]]->table[0] == seqs[order[a0]]->table[0]) ++b0;
      if (b0 - a0 >= 2) {
        std::vector<int> grp(order.begin() + static_cast<long>(a0),
                             order.begin() + static_cast<long>(b0));
        std::sort(grp.begin(), grp.end());
        const size_t before = nodes.size();
        run_group(run_group, std::move(grp), 0);
        if (nodes.size() > before) roots.push_back(static_cast<int>(before));
      }
      a0 = b0;
    }
  }
  // nodes of root group r: [roots[r], roots[r + 1])
  roots.push_back(static_cast<int>(nodes.size()));

  // ---- segments, members, entries.  Order: per root group and K/V head,
  // its shared runs (in the order found) followed by the members' private
  // rests of that head; these (group, head) items are spread evenly among
  // the sequences outside every group (item i before ungrouped sequence
  // ceil(i * n_ungrouped / n_items)).  Tiny private rests are thus spread over
  // the work list instead of piling up at its end, and the wide shared
  // segments, whose blocks cost more, fall to different CTAs (the split
  // balances work units).
  std::vector<PlanSeg>& segs = sc.segs;
  std::vector<int32_t>& members = sc.members;
  segs.clear();
  members.clear();
  segs.reserve(static_cast<size_t>(nodes.size() + n_seq) * H);
  members.reserve(static_cast<size_t>(n_seq) * (kPlanMaxLevels + 1));
  // merge entries per (sequence, head): its shared runs and its private rest
  constexpr int kEnt = kPlanMaxLevels + 1;
  std::vector<PlanEntry>& entk = sc.entk;  // entries of (sequence, head) sh: kEnt * sh ..
  std::vector<uint8_t>& n_ent = sc.n_ent;   // .. + n_ent[sh] - 1
  if (entk.size() < static_cast<size_t>(kEnt) * n_seq * H)
    entk.resize(static_cast<size_t>(kEnt) * n_seq * H);
  n_ent.assign(static_cast<size_t>(n_seq) * H, 0);
  auto add_entry = [&](size_t sh, PlanEntry e) { entk[kEnt * sh + n_ent[sh]++] = e; };
  int c_max = G;
  std::vector<int>& priv_mem = sc.priv_mem;  // member-list slot of a sequence's private rest
  priv_mem.assign(n_seq, -1);
  auto private_member = [&](int i) {
    if (priv_mem[i] < 0) {
      priv_mem[i] = static_cast<int>(members.size());
      members.push_back(i);
    }
    return priv_mem[i];
  };
  auto push_private = [&](int i, int h) {
    const int nb = static_cast<int>((seqs[i]->len + B - 1) / B);
    if (nb <= priv_from[i]) return;
    PlanSeg s{};
    s.rep = i;
    s.b0 = priv_from[i];
    s.b1 = nb;
    s.tok_end = static_cast<int32_t>(seqs[i]->len);
    s.head = h;
    s.ncols = G;
    s.mem = private_member(i);
    const int si = static_cast<int>(segs.size());
    segs.push_back(s);
    add_entry(static_cast<size_t>(i) * H + h, {si, 0});
  };
  std::vector<int>& node_mem0 = sc.node_mem0;  // member-list slot of each node
  node_mem0.assign(nodes.size(), -1);
  auto push_group_head = [&](size_t r, int h) {
    std::vector<int> grp_members;
    for (int ni = roots[r]; ni < roots[r + 1]; ++ni) {
      const Node& nd = nodes[ni];
      if (node_mem0[ni] < 0) {
        node_mem0[ni] = static_cast<int>(members.size());
        for (int m : nd.mem) members.push_back(m);
      }
      const int ncols = static_cast<int>(nd.mem.size()) * G;
      c_max = std::max(c_max, ncols);
      PlanSeg s{};
      s.rep = nd.mem[0];
      s.b0 = nd.b0;
      s.b1 = nd.b1;
      s.tok_end = nd.b1 * B;
      s.head = h;
      s.ncols = ncols;
      s.mem = node_mem0[ni];
      const int si = static_cast<int>(segs.size());
      segs.push_back(s);
      for (size_t k = 0; k < nd.mem.size(); ++k)
        add_entry(static_cast<size_t>(nd.mem[k]) * H + h, {si, static_cast<int>(k) * G});
      grp_members.insert(grp_members.end(), nd.mem.begin(), nd.mem.end());
    }
    std::sort(grp_members.begin(), grp_members.end());
    grp_members.erase(std::unique(grp_members.begin(), grp_members.end()), grp_members.end());
    for (int m : grp_members) push_private(m, h);
  };
  std::vector<char>& grouped = sc.grouped;
  grouped.assign(n_seq, 0);
  for (const Node& nd : nodes)
    for (int m : nd.mem) grouped[m] = 1;
  std::vector<int>& ungrouped = sc.ungrouped;
  ungrouped.clear();
  for (int i = 0; i < n_seq; ++i)
    if (!grouped[i]) ungrouped.push_back(i);
  const size_t n_roots = roots.size() - 1;
  const size_t n_i = n_roots * H, n_u = ungrouped.size();
  size_t it = 0;
  auto push_item = [&](size_t i) { push_group_head(i % n_roots, static_cast<int>(i / n_roots)); };
  for (size_t k = 0; k < n_u; ++k) {
    while (it < n_i && it * n_u <= k * n_i) push_item(it++);
    for (int h = 0; h < H; ++h) push_private(ungrouped[k], h);
  }
  while (it < n_i) push_item(it++);

  // ---- the kernel the work units are weighted for: the pool's decode path;
  // automatic: tcgen05 when segments of more than 16 columns hold at least
  // half of the blocks read (many sharers of long prefixes: its S and P.V
  // cost little per byte at any width), else the warp-level MMA pass (which
  // streams narrow segments faster)
  int kernel = kPlanKernelMma;
  if (pool_tc_decode_shape(p)) {
    if (p->decode_path == 3) {
      kernel = kPlanKernelTc;
    } else if (p->decode_path == 0) {
      int64_t wide = 0, all = 0;
      for (const PlanSeg& s : segs) {
        all += s.b1 - s.b0;
        if (s.ncols > 16) wide += s.b1 - s.b0;
      }
      if (all > 0 && 2 * wide >= all) kernel = kPlanKernelTc;
    }
  }
  int64_t W = 0;
  for (PlanSeg& s : segs) {
    s.w = plan_seg_weight(s.ncols, kernel, s.b1 - s.b0);
    s.wpre = W;
    W += static_cast<int64_t>(s.b1 - s.b0) * s.w;
  }
  int n_entries = 0;
  for (uint8_t c : n_ent) n_entries += c;

  // ---- serialise (start records only where the buffer has room for them:
  // a buffer sized before the device was known holds none)
  int grid = start_records ? plan_grid(p, kernel, G) : 0;
  Layout l = plan_layout(n_seq, H, static_cast<int>(segs.size()),
                         static_cast<int>(members.size()), n_entries, grid);
  if (l.total > plan_bytes || W == 0) {
    grid = 0;
    l = plan_layout(n_seq, H, static_cast<int>(segs.size()), static_cast<int>(members.size()),
                    n_entries, 0);
  }
  if (l.total > plan_bytes) return KV_ERR_INVALID_ARG;
  unsigned char* out = static_cast<unsigned char*>(h_plan);
  std::memset(out, 0, l.start);  // the start records are written whole below
  PlanHeader hd{};
  hd.W = W;
  hd.n_segs = static_cast<int32_t>(segs.size());
  hd.n_members = static_cast<int32_t>(members.size());
  hd.n_entries = n_entries;
  hd.c_max = c_max;
  hd.n_seq = n_seq;
  hd.n_kv_heads = H;
  hd.group = G;
  hd.block_size = B;
  hd.seg_off = static_cast<int32_t>(l.seg);
  hd.mem_off = static_cast<int32_t>(l.mem);
  hd.eoff_off = static_cast<int32_t>(l.eoff);
  hd.ent_off = static_cast<int32_t>(l.ent);
  hd.n_shared_segs = static_cast<int32_t>(nodes.size()) * H;
  hd.kernel = kernel;
  hd.start_off = grid > 0 ? static_cast<int32_t>(l.start) : 0;
  hd.start_grid = grid;
  std::memcpy(out, &hd, sizeof(hd));
  if (grid > 0)
    plan_starts(segs, W, grid, B, seqs, reinterpret_cast<PlanStart*>(out + l.start));
  if (!segs.empty()) std::memcpy(out + l.seg, segs.data(), sizeof(PlanSeg) * segs.size());
  if (!members.empty()) std::memcpy(out + l.mem, members.data(), sizeof(int32_t) * members.size());
  int32_t* eoff = reinterpret_cast<int32_t*>(out + l.eoff);
  PlanEntry* ent = reinterpret_cast<PlanEntry*>(out + l.ent);
  int k = 0;
  for (size_t i = 0; i < n_ent.size(); ++i) {
    eoff[i] = k;
    for (int j = 0; j < n_ent[i]; ++j) ent[k++] = entk[kEnt * i + j];
  }
  eoff[n_ent.size()] = k;
  if (out_workspace_bytes) *out_workspace_bytes = plan_workspace_bytes(hd.n_segs, c_max, p->D);
  return KV_OK;
}

extern "C" {


// Heaviest-first order of the chunked-prefill work items.  An item is one
// tile of 128 / G query tokens of one sequence's chunk (all query heads of a
// K/V head: 128 tile rows); its work is the number of 128-key blocks its
// queries read, ceil((h + min(c, (t + 1) T)) / 128) for history h, chunk c
// and tile t.  One CTA runs an item per K/V head and the hardware hands
// CTAs to free SMs in launch order, so launching the longest items first is
// list scheduling in decreasing-time order: the last CTAs to start are short
// and the SMs run out together, where the natural grid (sequences in
// caller order, tiles in token order) starts the longest histories last.
size_t paged_prefill_schedule_bytes(const kvPool* p, int n_seq, int n_q_heads, int max_chunk) {
  if (!p || n_seq < 0 || max_chunk < 0 || n_q_heads <= 0 || n_q_heads % p->H != 0) return 0;
  const int G = n_q_heads / p->H;
  if (G != 1 && G != 2 && G != 4 && G != 8) return 0;
  const long long T = 128 / G;
  return static_cast<size_t>(n_seq) * static_cast<size_t>((max_chunk + T - 1) / T) * 16;
}

kvStatus paged_prefill_schedule(const kvPool* p, const int32_t* h_chunk_start,
                                const int32_t* h_context_lens, int n_seq, int n_q_heads,
                                void* h_sched, size_t sched_bytes, int* out_n_items) {
  if (!p || n_seq < 0 || !out_n_items || n_q_heads <= 0 || n_q_heads % p->H != 0)
    return KV_ERR_INVALID_ARG;
  if (n_seq > 0 && (!h_chunk_start || !h_context_lens || !h_sched)) return KV_ERR_INVALID_ARG;
  const int G = n_q_heads / p->H;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KV_ERR_UNSUPPORTED;
  const int T = 128 / G;
  struct Item {
    int32_t s, t, c, nkb;
  };
  std::vector<Item> items;
  for (int s = 0; s < n_seq; ++s) {
    const long long c = static_cast<long long>(h_chunk_start[s + 1]) - h_chunk_start[s];
    const int32_t ctx = h_context_lens[s];
    if (c < 0 || ctx < c || h_chunk_start[s] < 0) return KV_ERR_INVALID_ARG;
    const long long h = ctx - c;
    for (long long t = 0; t * T < c; ++t) {
      const long long last = std::min(c, (t + 1) * T);  // tokens up to the tile's last
      items.push_back({s, static_cast<int32_t>(t), static_cast<int32_t>(c),
                       static_cast<int32_t>((h + last + 127) / 128)});
    }
  }
  if (items.size() * 16 > sched_bytes ||
      items.size() * static_cast<size_t>(p->H) > static_cast<size_t>(INT32_MAX))
    return KV_ERR_INVALID_ARG;
  // decreasing work; equal work in (sequence, tile) order, so the order is
  // a function of the chunk geometry alone
  std::stable_sort(items.begin(), items.end(),
                   [](const Item& x, const Item& y) { return x.nkb > y.nkb; });
  std::memcpy(h_sched, items.data(), items.size() * sizeof(Item));
  *out_n_items = static_cast<int>(items.size());
  return KV_OK;
}

}  // extern "C"
