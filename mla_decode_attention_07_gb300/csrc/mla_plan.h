// Split-KV tile metadata shared by the planner, the decode kernel and the
// combine kernel.  Everything here is integer arithmetic and compiles for
// both host and device so the host planner and the device planner give
// bit-identical plans.
//
// Work model.  Query rows of one batch entry (s_q * h_q of them) are cut into
// T tiles of 128 rows.  The grid's clusters are split into T equal groups;
// group t handles tile t of every batch entry, and every group uses the same
// partition of pages, so the clusters working on the two tiles of one page
// range run at the same time and share its reads through L2.
//
// Within a group, batch entry b with P_b = ceil(L_b / 64) > 0 pages occupies
// an interval of P_b + kSplitOverhead "virtual units" on a line (the extra
// units stand for the fixed cost of a split: loading Q and writing the
// result).  Cluster c of G_used takes the units [c*V/G_used, (c+1)*V/G_used)
// and processes the pages whose units fall inside.  Every cluster gets at
// least one unit, so the clusters touching entry b are consecutive and each
// holds at least one of its pages: entry b has c_last - c_first + 1 splits and
// cluster c's part of it has split index c - c_first.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define MLA_HD __host__ __device__ __forceinline__
#else
#define MLA_HD inline
#endif

namespace mla {

constexpr int kPageTokens = 64;
constexpr int kTileRows = 128;
constexpr int kSplitOverhead = 6;   // virtual units charged per batch entry (best of 2/4/6/8 measured)
constexpr int kMinUnitsPerCluster = 4;
constexpr int kPlanMagic = 0x4D4C4131;  // "MLA1"

// header words
enum PlanHeader {
  H_MAGIC = 0, H_BATCH, H_SQ, H_HQ, H_TILES, H_GT, H_GUSED, H_STOTAL, H_OVH, H_NCLUSTERS,
  H_WORDS = 16
};
constexpr int kClusterWords = 8;  // b0, p0, b1, p1, split0, 0, 0, 0
constexpr int kItemWords = 4;     // pages, num_splits, split_base, c_first

MLA_HD int plan_tiles(int s_q, int h_q) { return (s_q * h_q + kTileRows - 1) / kTileRows; }
MLA_HD int plan_group_clusters(int num_clusters, int tiles) { return num_clusters / tiles; }

// Byte offsets of the sections of a plan.
MLA_HD int64_t plan_off_clusters() { return 4 * (int64_t)H_WORDS; }
MLA_HD int64_t plan_off_items(int gt) { return plan_off_clusters() + 4 * (int64_t)kClusterWords * gt; }
MLA_HD int64_t plan_off_starts(int batch, int gt) {
  int64_t o = plan_off_items(gt) + 4 * (int64_t)kItemWords * batch;
  return (o + 7) & ~(int64_t)7;
}
MLA_HD int64_t plan_bytes(int batch, int gt) {
  return plan_off_starts(batch, gt) + 8 * (int64_t)(batch + 1);
}

MLA_HD int pages_of(int seqlen) { return seqlen > 0 ? (seqlen + kPageTokens - 1) / kPageTokens : 0; }
MLA_HD int64_t units_of(int pages) { return pages > 0 ? (int64_t)pages + kSplitOverhead : 0; }

// Clusters that receive work for V units and gt clusters in the group.
MLA_HD int plan_used_clusters(int64_t V, int gt) {
  if (V <= 0 || gt <= 0) return 0;
  int64_t g = V / kMinUnitsPerCluster;
  if (g < 1) g = 1;
  if (g > gt) g = gt;
  return (int)g;
}

// First unit of cluster c.
MLA_HD int64_t cluster_begin(int c, int64_t V, int g) { return (int64_t)c * V / g; }

// Cluster whose unit range contains unit x (0 <= x < V).
MLA_HD int cluster_of(int64_t x, int64_t V, int g) { return (int)(((x + 1) * g + V - 1) / V - 1); }

// Largest b with starts[b] <= x (starts non-decreasing, starts[0] = 0,
// starts[batch] = V); returns batch when x >= V.
MLA_HD int item_of(const int64_t* starts, int batch, int64_t x) {
  if (x >= starts[batch]) return batch;
  int lo = 0, hi = batch;  // invariant: starts[lo] <= x < starts[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (starts[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Cursor (item, page) of the first page whose unit is >= x, normalised so
// that it never points past the end of an item (it moves to page 0 of the
// next item with pages, or to (batch, 0)).
MLA_HD void cursor_of(const int64_t* starts, int batch, int64_t x, int* b_out, int* p_out) {
  int b = item_of(starts, batch, x);
  int p = 0;
  if (b < batch) {
    int64_t len = starts[b + 1] - starts[b];
    int pages = len > 0 ? (int)(len - kSplitOverhead) : 0;
    int64_t rel = x - starts[b] - kSplitOverhead;
    p = rel < 0 ? 0 : (rel > pages ? pages : (int)rel);
    if (p >= pages) {
      // past the last page: next item that has pages
      b += 1;
      while (b < batch && starts[b + 1] == starts[b]) ++b;
      p = 0;
    }
  }
  *b_out = b;
  *p_out = p;
}

// Segments of the cluster's page range: item b, pages [pb, pe).
struct SegIter {
  int b, p, b1, p1;
  const int32_t* items;
  MLA_HD bool next(int& sb, int& spb, int& spe) {
    while (b < b1 || (b == b1 && p < p1)) {
      const int P = items[b * kItemWords + 0];
      const int pe = (b == b1) ? p1 : P;
      const int cb = b, cp = p;
      b += 1;
      p = 0;
      if (cp < pe) {
        sb = cb;
        spb = cp;
        spe = pe;
        return true;
      }
    }
    return false;
  }
};

}  // namespace mla
