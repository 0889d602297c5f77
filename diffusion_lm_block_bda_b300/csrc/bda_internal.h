// bda_internal.h -- shared between the host planner and the CUDA kernels:
// the work-item layout written into the workspace and the mask in interval
// form.  (The CPU oracle has its own, independent mask code.)
//
// Mask (ORL announcement thread, 24vids.com mirror: highlight 3 for
// block-causal, Insight 3 for staircase; ORL paper card, thelatestinai.com,
// Figure 3 caption).  Block-causal is the staircase with prefix P = Lk (no
// copies), so one form serves both.  For a query at key position p:
//   p <  P : keys [0, min(P, (p/B + 1) * B))                 (block-causal)
//   p >= P : keys [0, P) and its own copy [P + cB, P + cB + B), c = (p-P)/B
// and, transposed, key j is seen by query positions
//   j <  P : [ (j/B) * B, Lk )
//   j >= P : [ P + cB, P + cB + B ),  c = (j-P)/B
#pragma once
#include <cstdint>

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
  int32_t pad[4];
};
static_assert(sizeof(FwdItem) == 64, "FwdItem layout");

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
  int32_t q_begin;   // local query tokens [q_begin, q_end) see some key of the tile
  int32_t q_end;
  int32_t work;      // query tiles to visit per KV head
  int32_t seq;
  int32_t pad[5];
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

// Query positions that see key j: [lo, hi).
struct KeyRows {
  int lo, hi;
};
BDA_HD KeyRows key_rows(int j, int P, int B, int Lk) {
  KeyRows r;
  if (j < P) {
    r.lo = (j / B) * B;
    r.hi = Lk;
  } else {
    r.lo = P + ((j - P) / B) * B;
    const int hi = r.lo + B;
    r.hi = hi < Lk ? hi : Lk;
  }
  return r;
}

}  // namespace bda
