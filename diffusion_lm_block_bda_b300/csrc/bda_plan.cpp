// bda_plan.cpp -- argument validation and the varlen tile planner (host).
//
// "Packed compute-balanced training" (ORL announcement thread, Insight 3) and
// "packed and load-balanced" states (ORL paper card, Figure 3 caption): the
// packed sequences have unequal lengths and, under a block-causal mask, query
// tiles late in a sequence see many more keys than early ones.  The planner
// lists every non-empty query tile (forward) and key tile (backward) with the
// exact range of tiles it must visit, then orders the units longest-first
// (LPT).  CTAs are dispatched in that order, so each SM greedily takes the
// longest remaining unit -- list scheduling, whose makespan is within one unit
// of the lower bound max(total / SMs, longest unit).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>

#include "bda_host.h"
#include "bda_internal.h"

namespace bda {

namespace {

int largest_pow2_divisor(int g, int cap) {
  int h = 1;
  while (h * 2 <= cap && g % (h * 2) == 0) h *= 2;
  return h;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

int seq_prefix(const bda_mask_desc* m, int s, int lk) {
  return m->kind != BDA_MASK_BLOCK_CAUSAL ? m->prefix_len_host[s] : lk;
}

// The forward item of the query tile starting at local token t0 of sequence
// sq: its key tiles [0, r1_end) and [r2_begin, r2_end), the first n_full of
// them FULL.
FwdItem make_fwd_item(const Shape& s, int sq, int q0, int lq, int k0, int lk, int P, int t0,
                      int grp_off, int n_grp, const int2* grp) {
  const int B = s.B;
  FwdItem it{};
  it.q_row = q0 + t0;
  it.q_len = std::min(s.tok, lq - t0);
  it.pos0 = t0 + (lk - lq);
  it.k_row = k0;
  it.lk = lk;
  it.prefix = P;
  it.seq = sq;
  it.grp_off = grp_off;
  it.n_grp = n_grp;
  it.n_split = 1;
  it.part0 = -1;
  const int p_lo = it.pos0, p_hi = it.pos0 + it.q_len - 1;
  // Rows see [0, a(p)) and their own copy.  Without copy groups a(p) grows
  // with p; with them, take the extremes over the tile's rows.
  int a_min, a_max;
  if (n_grp == 0) {
    a_min = row_keys(p_lo, P, B, lk).a;
    a_max = row_keys(p_hi, P, B, lk).a;
  } else {
    a_min = lk;
    a_max = 0;
    for (int q = p_lo; q <= p_hi; ++q) {
      const int a = row_keys_g(q, P, B, lk, grp, n_grp).a;
      a_min = std::min(a_min, a);
      a_max = std::max(a_max, a);
    }
  }
  // Key tiles inside [0, a_min) are FULL for every row.
  it.n_full = a_min / kTileN;
  it.r1_end = ceil_div(a_max, kTileN);
  it.r2_begin = it.r2_end = 0;
  if (p_hi >= P) {  // copy rows: their own copies span [b(first copy row), e(p_hi))
    const RowKeys c = row_keys(std::max(p_lo, P), P, B, lk);
    const RowKeys hi = row_keys(p_hi, P, B, lk);
    int b0 = c.b / kTileN, b1 = ceil_div(hi.e, kTileN);
    if (b0 <= it.r1_end) {
      it.r1_end = std::max(it.r1_end, b1);
    } else {
      it.r2_begin = b0;
      it.r2_end = b1;
    }
  }
  it.work = it.r1_end + (it.r2_end - it.r2_begin);
  return it;
}

// Copy groups of sequence sq (non-empty only), as (first position, visible).
int seq_groups(const bda_mask_desc* m, int sq, int P, int B, int2* out) {
  int n = 0, start = P;
  for (int g = m->group_offsets_host[sq]; g < m->group_offsets_host[sq + 1]; ++g) {
    const int c = m->group_copies_host[g];
    if (c == 0) continue;
    out[n++] = int2{start, m->group_visible_host[g]};
    start += c * B;
  }
  return n;
}

// Split chunk for a problem with few forward units: key tiles per unit so
// that the units number about kSplitTargetUnits (0: no split).  Sums the
// items' key-tile counts, so it builds them (only when few).
int split_chunk(const bda_problem* p, const bda_mask_desc* m, const Shape& s) {
  const int n_groups = s.hq / s.hg;
  if (int64_t(s.n_fwd) * n_groups >= kSplitMaxUnits || s.n_fwd == 0) return 0;
  std::vector<int2> grp(size_t(s.n_cgroups) + 1);
  int64_t tiles = 0;
  int max_work = 0;
  for (int sq = 0; sq < s.nseq; ++sq) {
    const int q0 = p->cu_seqlens_q_host[sq], lq = p->cu_seqlens_q_host[sq + 1] - q0;
    const int k0 = p->cu_seqlens_k_host[sq], lk = p->cu_seqlens_k_host[sq + 1] - k0;
    const int P = seq_prefix(m, sq, lk);
    const int n_grp = s.kind == BDA_MASK_STAIRCASE_MULTI ? seq_groups(m, sq, P, s.B, grp.data()) : 0;
    for (int t0 = 0; t0 < lq; t0 += s.tok) {
      const FwdItem it = make_fwd_item(s, sq, q0, lq, k0, lk, P, t0, 0, n_grp, grp.data());
      tiles += it.work;
      max_work = std::max(max_work, it.work);
    }
  }
  const int64_t units = tiles * n_groups;
  const int c = int(std::max<int64_t>(1, (units + kSplitTargetUnits - 1) / kSplitTargetUnits));
  return c < max_work ? c : 0;  // 0 when no item would be cut
}

}  // namespace

bda_status validate(const bda_problem* p, const bda_mask_desc* m, Shape* s, bool count_only) {
  if (!p || !m || !s) return BDA_ERR_INVALID_ARG;
  if (p->nseq < 0 || p->hq <= 0 || p->hkv <= 0 || p->head_dim <= 0) return BDA_ERR_INVALID_ARG;
  if (p->hq % p->hkv != 0) return BDA_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return BDA_ERR_UNSUPPORTED;
  const bool multi = m->kind == BDA_MASK_STAIRCASE_MULTI;
  if (m->kind != BDA_MASK_BLOCK_CAUSAL && m->kind != BDA_MASK_STAIRCASE && !multi)
    return BDA_ERR_INVALID_ARG;
  if (m->block_size < 1) return BDA_ERR_INVALID_ARG;
  if (!(p->softmax_scale == p->softmax_scale) || std::isinf(p->softmax_scale))
    return BDA_ERR_INVALID_ARG;
  if (p->nseq > 0 && (!p->cu_seqlens_q_host || !p->cu_seqlens_k_host)) return BDA_ERR_INVALID_ARG;
  if (p->nseq > 0 && m->kind != BDA_MASK_BLOCK_CAUSAL && !m->prefix_len_host)
    return BDA_ERR_INVALID_ARG;
  if (p->nseq > 0 && multi &&
      (!m->group_offsets_host || !m->group_copies_host || !m->group_visible_host ||
       m->group_offsets_host[0] != 0))
    return BDA_ERR_INVALID_ARG;
  Shape r;
  r.nseq = p->nseq;
  r.hq = p->hq;
  r.hkv = p->hkv;
  r.d = p->head_dim;
  r.G = p->hq / p->hkv;
  r.hg = largest_pow2_divisor(r.G, 16);
  r.lg_hg = 0;
  while ((1 << r.lg_hg) < r.hg) ++r.lg_hg;
  r.tok = kTileM / r.hg;
  r.kind = m->kind;
  r.B = m->block_size;
  r.scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt(float(p->head_dim));
  if (p->nseq > 0) {
    const int32_t* cq = p->cu_seqlens_q_host;
    const int32_t* ck = p->cu_seqlens_k_host;
    if (cq[0] != 0 || ck[0] != 0) return BDA_ERR_INVALID_ARG;
    int64_t nf = 0, nb = 0, ng = 0;
    bool block_order = true;
    for (int i = 0; i < p->nseq; ++i) {
      const int64_t lq = int64_t(cq[i + 1]) - cq[i];
      const int64_t lk = int64_t(ck[i + 1]) - ck[i];
      if (lq < 0 || lk < 0) return BDA_ERR_INVALID_ARG;
      if (lq > 0 && lk == 0) return BDA_ERR_INVALID_ARG;  // queries with nothing to see
      if (m->kind == BDA_MASK_BLOCK_CAUSAL) {
        if (lq > lk) return BDA_ERR_INVALID_ARG;  // early queries would see no key
      } else if (!multi) {
        const int64_t P = m->prefix_len_host[i];
        if (lq != lk || P < 0 || P > lk || (lk - P) % m->block_size != 0)
          return BDA_ERR_INVALID_ARG;
      } else {
        // groups of copies tile [P, L) and see at most the prefix
        const int64_t P = m->prefix_len_host[i];
        const int32_t g0 = m->group_offsets_host[i], g1 = m->group_offsets_host[i + 1];
        if (lq != lk || P < 0 || P > lk || g1 < g0) return BDA_ERR_INVALID_ARG;
        int64_t tokens = 0, last_v = -1;
        for (int32_t g = g0; g < g1; ++g) {
          const int64_t c = m->group_copies_host[g], v = m->group_visible_host[g];
          if (c < 0 || v < 0 || v > P) return BDA_ERR_INVALID_ARG;
          tokens += c * m->block_size;
          if (c > 0) {
            if (v < last_v) block_order = false;
            last_v = v;
            ++ng;
          }
        }
        if (tokens != lk - P) return BDA_ERR_INVALID_ARG;
      }
      nf += (lq + r.tok - 1) / r.tok;
      nb += (lk + kTileN - 1) / kTileN;
    }
    r.total_q = cq[p->nseq];
    r.total_k = ck[p->nseq];
    // Row indices and element offsets stay in 32-bit / 64-bit ranges.
    if (r.total_q >= (int64_t(1) << 31) || r.total_k >= (int64_t(1) << 31))
      return BDA_ERR_INVALID_ARG;
    if (nf >= (int64_t(1) << 30) / r.hq || nb >= (int64_t(1) << 30)) return BDA_ERR_INVALID_ARG;
    if (ng >= (int64_t(1) << 30)) return BDA_ERR_INVALID_ARG;
    r.n_fwd = int(nf);
    r.n_bwd = int(nb);
    r.n_cgroups = int(ng);
    // Split forward: units and partial slots follow from the chunk size.
    r.split_c = split_chunk(p, m, r);
    r.n_dec = r.n_fwd;
    r.n_parts = 0;
    if (r.split_c > 0) {
      std::vector<FwdItem> fw;
      std::vector<int2> grp(size_t(r.n_cgroups) + 1);
      r.n_dec = 0;
      for (int i = 0; i < p->nseq; ++i) {
        const int q0 = cq[i], lq = cq[i + 1] - q0, k0 = ck[i], lk = ck[i + 1] - k0;
        const int P = seq_prefix(m, i, lk);
        const int n_grp = multi ? seq_groups(m, i, P, r.B, grp.data()) : 0;
        for (int t0 = 0; t0 < lq; t0 += r.tok) {
          const int w = make_fwd_item(r, i, q0, lq, k0, lk, P, t0, 0, n_grp, grp.data()).work;
          const int n_split = std::max(1, (w + r.split_c - 1) / r.split_c);
          r.n_dec += n_split;
          if (n_split > 1) r.n_parts += n_split;
        }
      }
    }
    *s = r;
    // Groups out of block order are counted but not computed.
    return block_order || count_only ? BDA_OK : BDA_ERR_UNSUPPORTED;
  }
  *s = r;
  return BDA_OK;
}

size_t plan_group_offset(const Shape& s, bool with_bwd) {
  return kHeaderBytes + sizeof(FwdItem) * size_t(s.n_fwd) +
         (with_bwd ? sizeof(BwdItem) * size_t(s.n_bwd) : 0);
}

size_t plan_dec_offset(const Shape& s, bool with_bwd) {
  return plan_group_offset(s, with_bwd) + ((sizeof(int2) * size_t(s.n_cgroups) + 15) & ~size_t(15));
}

size_t plan_bytes(const Shape& s, bool with_bwd) {
  return plan_dec_offset(s, with_bwd) + sizeof(DecItem) * size_t(s.n_dec);
}

size_t ws_offset_parts(const Shape& s) { return align256(plan_bytes(s)); }

size_t ws_offset_part_lse(const Shape& s) {
  const size_t slots = size_t(s.n_parts) * size_t(s.hq / s.hg);
  return ws_offset_parts(s) + align256(sizeof(float) * slots * size_t(s.d) * kTileM);
}

size_t ws_offset_D(const Shape& s) {
  const size_t slots = size_t(s.n_parts) * size_t(s.hq / s.hg);
  return ws_offset_part_lse(s) + align256(sizeof(float) * slots * kTileM);
}

size_t ws_offset_dqacc(const Shape& s) {
  return ws_offset_D(s) + align256(sizeof(float) * size_t(s.hq) * size_t(s.total_q));
}

size_t workspace_bytes(const Shape& s, bool with_bwd) {
  if (!with_bwd) return ws_offset_D(s);
  return ws_offset_dqacc(s) +
         align256(sizeof(float) * size_t(s.total_q) * size_t(s.hq) * size_t(s.d));
}

void build_plan(const bda_problem* p, const bda_mask_desc* m, const Shape& s, uint8_t* out,
                bool with_bwd) {
  std::memset(out, 0, plan_bytes(s, with_bwd));
  PlanHeader* h = reinterpret_cast<PlanHeader*>(out);
  h->status = 0;
  h->magic = kPlanMagic;
  h->n_fwd = s.n_fwd;
  h->n_bwd = with_bwd ? s.n_bwd : 0;
  h->hg = s.hg;
  h->tok = s.tok;
  h->total_q = int32_t(s.total_q);
  h->total_k = int32_t(s.total_k);
  h->n_cgroups = s.n_cgroups;
  h->n_dec = s.n_dec;
  h->n_parts = s.n_parts;
  h->split_c = s.split_c;
  std::vector<FwdItem> fw;
  std::vector<BwdItem> bw;
  fw.reserve(s.n_fwd);
  if (with_bwd) bw.reserve(s.n_bwd);
  // Copy-group table of the multi-block staircase: the non-empty groups of
  // every sequence, each as (first position, clean keys its copies see).
  int2* table = reinterpret_cast<int2*>(out + plan_group_offset(s, with_bwd));
  int n_table = 0;
  const bool multi = s.kind == BDA_MASK_STAIRCASE_MULTI;
  const int B = s.B;
  for (int sq = 0; sq < s.nseq; ++sq) {
    const int q0 = p->cu_seqlens_q_host[sq], lq = p->cu_seqlens_q_host[sq + 1] - q0;
    const int k0 = p->cu_seqlens_k_host[sq], lk = p->cu_seqlens_k_host[sq + 1] - k0;
    const int P = seq_prefix(m, sq, lk);
    const int delta = lk - lq;
    const int grp_off = n_table;
    if (multi) n_table += seq_groups(m, sq, P, B, table + n_table);
    const int n_grp = n_table - grp_off;
    const int2* grp = table + grp_off;
    // forward: query tiles of tok tokens
    for (int t0 = 0; t0 < lq; t0 += s.tok)
      fw.push_back(make_fwd_item(s, sq, q0, lq, k0, lk, P, t0, grp_off, n_grp, grp));
    // backward: key tiles of 128 keys
    for (int kp = 0; with_bwd && kp < lk; kp += kTileN) {
      BwdItem it{};
      it.k_row = k0 + kp;
      it.k_len = std::min(kTileN, lk - kp);
      it.kpos0 = kp;
      it.q_row = q0;
      it.lq = lq;
      it.lk = lk;
      it.prefix = P;
      it.seq = sq;
      it.grp_off = grp_off;
      it.n_grp = n_grp;
      // Query positions that see some key of the tile.  Its first key sees
      // the most rows of the prefix and of the copy groups; its copy keys
      // (if any) are seen by their own copies, which follow the prefix.
      const int kl = kp + it.k_len - 1;
      const KeyRows first = key_rows(kp, P, B, lk, grp, n_grp);
      const KeyRows last = key_rows(kl, P, B, lk, grp, n_grp);
      int lo1 = first.lo, hi1 = std::max(first.hi, kl >= P ? last.hi : 0);
      int lo2 = first.lo2, hi2 = first.hi2;
      bool two = hi2 > lo2;
      if (two && lo2 <= hi1) {  // the ranges touch: one range
        hi1 = std::max(hi1, hi2);
        two = false;
      }
      if (!two) lo2 = hi2 = 0;
      auto clip = [&](int x) { return std::min(lq, std::max(0, x - delta)); };
      it.q_begin = clip(lo1);
      it.q_end = std::max(it.q_begin, clip(hi1));
      it.q2_begin = clip(lo2);
      it.q2_end = std::max(it.q2_begin, clip(hi2));
      it.n_tiles1 = ceil_div(it.q_end - it.q_begin, s.tok);
      // The first range's last tile must not reach into the second range
      // (a query row visited twice would be counted twice): merge them.
      if (it.q2_end > it.q2_begin && it.q2_begin < it.q_begin + it.n_tiles1 * s.tok) {
        it.q_end = it.q2_end;
        it.q2_begin = it.q2_end = 0;
        it.n_tiles1 = ceil_div(it.q_end - it.q_begin, s.tok);
      }
      const int n_tiles2 = ceil_div(it.q2_end - it.q2_begin, s.tok);
      it.work = (it.n_tiles1 + n_tiles2) * (s.G / s.hg);
      bw.push_back(it);
    }
  }
  // Forward: longest-first; ties keep packing order.
  std::stable_sort(fw.begin(), fw.end(),
                   [](const FwdItem& a, const FwdItem& b) { return a.work > b.work; });
  // Backward: sequences longest-first (by their total work), and inside a
  // sequence its key tiles longest-first.  CTAs that run together then share
  // one sequence's Q, dO and dQ rows in L2 instead of streaming several
  // sequences' (the dQ accumulation is read-modify-write in L2); the tail is
  // still made of the shortest units of the shortest sequence.
  std::vector<long long> seq_work(s.nseq, 0);
  for (const BwdItem& b : bw) seq_work[b.seq] += b.work;
  std::stable_sort(bw.begin(), bw.end(), [&](const BwdItem& a, const BwdItem& b) {
    if (a.seq != b.seq) {
      if (seq_work[a.seq] != seq_work[b.seq]) return seq_work[a.seq] > seq_work[b.seq];
      return a.seq < b.seq;
    }
    return a.work > b.work;
  });
  // The last wave goes longest-first across sequences.  The block scheduler
  // hands out CTAs in grid order (item-major, hkv CTAs per item), so with
  // the tail in sequence order the last sequence's longest key tiles would
  // start last (the staircase replay's dK/dV: 148 -> 132 query tiles on the
  // busiest SM in a list schedule over 148 SMs).  The wave's few items span
  // two or three sequences, whose Q, dO and dQ rows still fit in L2.
  const size_t n_tail = std::min(bw.size(), size_t((kTailWaveCtas + s.hkv - 1) / s.hkv));
  std::stable_sort(bw.end() - std::ptrdiff_t(n_tail), bw.end(),
                   [](const BwdItem& a, const BwdItem& b) { return a.work > b.work; });
  // Split-forward units, in the forward items' (longest-first) order: each
  // item's key tiles cut into n_split nearly equal chunks of about split_c.
  DecItem* dec = reinterpret_cast<DecItem*>(out + plan_dec_offset(s, with_bwd));
  int n_dec = 0, n_parts = 0;
  for (size_t i = 0; i < fw.size(); ++i) {
    FwdItem& it = fw[i];
    it.n_split = s.split_c > 0 ? std::max(1, ceil_div(it.work, s.split_c)) : 1;
    it.part0 = it.n_split > 1 ? n_parts : -1;
    for (int c = 0; c < it.n_split; ++c) {
      DecItem& d = dec[n_dec++];
      d.item = int32_t(i);
      d.kt_lo = int32_t(int64_t(c) * it.work / it.n_split);
      d.kt_hi = int32_t(int64_t(c + 1) * it.work / it.n_split);
      d.part = it.n_split > 1 ? n_parts + c : -1;
    }
    if (it.n_split > 1) n_parts += it.n_split;
  }
  std::memcpy(out + kHeaderBytes, fw.data(), sizeof(FwdItem) * fw.size());
  std::memcpy(out + kHeaderBytes + sizeof(FwdItem) * fw.size(), bw.data(),
              sizeof(BwdItem) * bw.size());
}

long long count_pairs(const bda_problem* p, const bda_mask_desc* m, const Shape& s) {
  if (m->kind == BDA_MASK_STAIRCASE_MULTI) {
    // prefix rows: block-causal inside [0, P); a copy row: its group's
    // visible clean keys and its own B-token copy
    long long n = 0;
    for (int sq = 0; sq < s.nseq; ++sq) {
      const int P = m->prefix_len_host[sq];
      for (int i = 0; i < P; ++i) n += std::min(P, (i / s.B + 1) * s.B);
      for (int g = m->group_offsets_host[sq]; g < m->group_offsets_host[sq + 1]; ++g)
        n += (long long)m->group_copies_host[g] * s.B * (m->group_visible_host[g] + s.B);
    }
    return n;
  }
  long long n = 0;
  for (int sq = 0; sq < s.nseq; ++sq) {
    const int lq = p->cu_seqlens_q_host[sq + 1] - p->cu_seqlens_q_host[sq];
    const int lk = p->cu_seqlens_k_host[sq + 1] - p->cu_seqlens_k_host[sq];
    const int P = seq_prefix(m, sq, lk);
    for (int i = 0; i < lq; ++i) {
      const RowKeys r = row_keys(i + lk - lq, P, s.B, lk);
      n += r.a + (r.e - r.b);
    }
  }
  return n;
}

}  // namespace bda
