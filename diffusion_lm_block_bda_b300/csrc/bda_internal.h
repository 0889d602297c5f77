// bda_internal.h -- shared between the host planner and the CUDA kernels:
// the work-item layout written into the workspace and the mask in interval
// form.  (The CPU oracle has its own, independent mask code.)
//
// Mask (ORL announcement thread, 24vids.com mirror: highlight 3 for
// block-causal, Insight 3 for staircase; ORL paper card, thelatestinai.com,
// Figure 3 caption).  Block-causal is the staircase with prefix P = Lk (no
// copies), so one form serves both.  For a query at key position p:
//   p <  P : keys [0, min(P, (p/B + 1) * B))                 (block-causal)
//   p >= P : keys [0, V) and its own copy [P + cB, P + cB + B), c = (p-P)/B
// where V = P for the staircase; and, transposed, key j is seen by query
// positions
//   j <  P : [ (j/B) * B, P ) and the copy rows whose V exceeds j
//   j >= P : [ P + cB, P + cB + B ),  c = (j-P)/B
// Multi-block staircase (several active blocks per trajectory, the
// "irregular trajectories" of the announcement thread, Insight 3): the copy
// rows [P, Lk) are cut into groups, one per active block, and the copies of
// group g see V = visible_g clean keys.  Groups come in block order, so
// visible_g does not decrease along the sequence and the copy rows that see
// a clean key j form one suffix [start of the first group with V > j, Lk).
// The plan carries the non-empty groups of each sequence as a table of
// (start position, V) pairs.
#pragma once
#include <cstdint>
#include <vector_types.h>  // int2

#if defined(__CUDACC__)
#define BDA_HD __host__ __device__ __forceinline__
#else
#define BDA_HD inline
#endif

namespace bda {

constexpr int kTileM = 128;  // query-tile rows (tokens x heads of one KV group)
constexpr int kTileN = 128;  // keys per key tile
constexpr uint32_t kPlanMagic = 0x42444131u;  // "BDA1"
constexpr int kHeaderBytes = 256;

// One forward work unit: a query tile (tok tokens of one sequence x hg query
// heads); its key tiles are [0, r1_end) then [r2_begin, r2_end); tiles below
// n_full need no mask.
struct FwdItem {
  int32_t q_row;     // global row of the tile's first query token
  int32_t q_len;     // valid query tokens in the tile (1..tok)
  int32_t pos0;      // key position of the tile's first query token
  int32_t k_row;     // global row of the sequence's first key
  int32_t lk;        // keys in the sequence
  int32_t prefix;    // staircase prefix length; lk for block-causal
  int32_t n_full;    // key tiles [0, n_full) are FULL
  int32_t r1_end;    // key tiles [n_full, r1_end) are PARTIAL
  int32_t r2_begin;  // key tiles [r2_begin, r2_end) are PARTIAL
  int32_t r2_end;
  int32_t work;      // number of key tiles
  int32_t seq;
  int32_t grp_off;   // the sequence's copy groups in the plan's table ...
  int32_t n_grp;     // ... (0: every copy sees the whole prefix)
  int32_t n_split;   // split forward: key-tile chunks of this tile (1: none) ...
  int32_t part0;     // ... and the first partial-result slot of its chunks
};
static_assert(sizeof(FwdItem) == 64, "FwdItem layout");

// One unit of the split (decode) forward: key tiles [kt_lo, kt_hi) of the
// tile list of forward item `item`; `part` is its partial-result slot, or -1
// when the item is not split (the unit then writes O and LSE itself).
struct DecItem {
  int32_t item;
  int32_t kt_lo;
  int32_t kt_hi;
  int32_t part;
};
static_assert(sizeof(DecItem) == 16, "DecItem layout");

// One backward work unit: a 128-key tile of one sequence (all KV heads run it
// in parallel); query tokens [q_begin, q_end) are the ones that see it.
struct BwdItem {
  int32_t k_row;     // global row of the tile's first key
  int32_t k_len;     // valid keys in the tile (1..128)
  int32_t kpos0;     // position of the tile's first key in its sequence
  int32_t q_row;     // global row of the sequence's first query token
  int32_t lq;
  int32_t lk;
  int32_t prefix;    // staircase prefix length; lk for block-causal
  int32_t q_begin;   // local query tokens [q_begin, q_end) and [q2_begin, q2_end)
  int32_t q_end;     // hold every query that sees some key of the tile; the
  int32_t q2_begin;  // second range is empty unless copy groups that do not
  int32_t q2_end;    // see the tile's clean keys sit between the two
  int32_t n_tiles1;  // query-token tiles of the first range
  int32_t work;      // query tiles to visit per KV head
  int32_t seq;
  int32_t grp_off;   // as in FwdItem
  int32_t n_grp;
};
static_assert(sizeof(BwdItem) == 64, "BwdItem layout");

struct PlanHeader {
  uint32_t status;   // device-written error bits (BDA_ERR_DEVICE_TIMEOUT ...)
  uint32_t magic;
  int32_t n_fwd;
  int32_t n_bwd;
  int32_t hg;
  int32_t tok;
  int32_t total_q;
  int32_t total_k;
  int32_t n_cgroups;  // entries of the copy-group table (after the items)
  int32_t n_dec;      // split-forward units (after the copy-group table)
  int32_t n_parts;    // partial-result slots of split forward items
  int32_t split_c;    // key tiles per split-forward unit (0: no item is split)
};

// Keys visible to the query at position p: [0, a) U [b, e).
struct RowKeys {
  int a, b, e;
};
BDA_HD RowKeys row_keys(int p, int P, int B, int Lk) {
  RowKeys r;
  if (p < P) {
    const int lim = (p / B + 1) * B;
    r.a = lim < P ? lim : P;
    r.b = 0;
    r.e = 0;
  } else {
    r.a = P;
    r.b = P + ((p - P) / B) * B;
    const int e = r.b + B;
    r.e = e < Lk ? e : Lk;
  }
  if (r.a > Lk) r.a = Lk;
  return r;
}

// Copy groups of a multi-block staircase sequence: grp[0..n) = (start, V),
// starts increasing, V non-decreasing.
// V of the copy row at position p >= grp[0].x: the last group starting at or
// before p.
BDA_HD int group_visible(int p, const int2* grp, int n) {
  int lo = 0, hi = n - 1;  // invariant: grp[lo].x <= p
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (grp[mid].x <= p) lo = mid; else hi = mid - 1;
  }
  return grp[lo].y;
}
// First copy row that sees clean key j: the start of the first group with
// V > j, or Lk if none.
BDA_HD int group_rows_from(int j, const int2* grp, int n, int Lk) {
  int lo = 0, hi = n;  // first index with V > j
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (grp[mid].y > j) hi = mid; else lo = mid + 1;
  }
  return lo < n ? grp[lo].x : Lk;
}

// Keys visible to the query at position p when copies see V = grp-table
// values (n > 0) instead of the whole prefix.
BDA_HD RowKeys row_keys_g(int p, int P, int B, int Lk, const int2* grp, int n) {
  RowKeys r = row_keys(p, P, B, Lk);
  if (n > 0 && p >= P) r.a = group_visible(p, grp, n);
  return r;
}

// Query positions that see key j: [lo, hi) and [lo2, hi2) (the second
// interval is empty unless copy groups that do not see j separate the two).
struct KeyRows {
  int lo, hi, lo2, hi2;
};
BDA_HD KeyRows key_rows(int j, int P, int B, int Lk, const int2* grp = nullptr, int n = 0) {
  KeyRows r;
  r.lo2 = r.hi2 = 0;
  if (j < P) {
    r.lo = (j / B) * B;
    r.hi = Lk;
    if (n > 0) {
      const int from = group_rows_from(j, grp, n, Lk);
      if (from > P) {  // prefix rows, then the copies of the groups that see j
        r.hi = P;
        r.lo2 = from;
        r.hi2 = Lk;
      }
    }
  } else {
    r.lo = P + ((j - P) / B) * B;
    const int hi = r.lo + B;
    r.hi = hi < Lk ? hi : Lk;
  }
  return r;
}

}  // namespace bda
