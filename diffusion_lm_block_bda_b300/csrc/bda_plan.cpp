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
  return m->kind == BDA_MASK_STAIRCASE ? m->prefix_len_host[s] : lk;
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
    int64_t nf = 0, nb = 0;
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
        int64_t tokens = 0;
        for (int32_t g = g0; g < g1; ++g) {
          const int64_t c = m->group_copies_host[g], v = m->group_visible_host[g];
          if (c < 0 || v < 0 || v > P) return BDA_ERR_INVALID_ARG;
          tokens += c * m->block_size;
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
    r.n_fwd = int(nf);
    r.n_bwd = int(nb);
  }
  *s = r;
  // The multi-block staircase is validated and counted; no kernel takes it yet.
  return multi && !count_only ? BDA_ERR_UNSUPPORTED : BDA_OK;
}

size_t plan_bytes(const Shape& s) {
  return kHeaderBytes + sizeof(FwdItem) * size_t(s.n_fwd) + sizeof(BwdItem) * size_t(s.n_bwd);
}

size_t ws_offset_D(const Shape& s) { return align256(plan_bytes(s)); }

size_t ws_offset_dqacc(const Shape& s) {
  return ws_offset_D(s) + align256(sizeof(float) * size_t(s.hq) * size_t(s.total_q));
}

size_t workspace_bytes(const Shape& s, bool with_bwd) {
  if (!with_bwd) return align256(plan_bytes(s));
  return ws_offset_dqacc(s) +
         align256(sizeof(float) * size_t(s.total_q) * size_t(s.hq) * size_t(s.d));
}

void build_plan(const bda_problem* p, const bda_mask_desc* m, const Shape& s, uint8_t* out) {
  std::memset(out, 0, plan_bytes(s));
  PlanHeader* h = reinterpret_cast<PlanHeader*>(out);
  h->status = 0;
  h->magic = kPlanMagic;
  h->n_fwd = s.n_fwd;
  h->n_bwd = s.n_bwd;
  h->hg = s.hg;
  h->tok = s.tok;
  h->total_q = int32_t(s.total_q);
  h->total_k = int32_t(s.total_k);
  std::vector<FwdItem> fw;
  std::vector<BwdItem> bw;
  fw.reserve(s.n_fwd);
  bw.reserve(s.n_bwd);
  const int B = s.B;
  for (int sq = 0; sq < s.nseq; ++sq) {
    const int q0 = p->cu_seqlens_q_host[sq], lq = p->cu_seqlens_q_host[sq + 1] - q0;
    const int k0 = p->cu_seqlens_k_host[sq], lk = p->cu_seqlens_k_host[sq + 1] - k0;
    const int P = seq_prefix(m, sq, lk);
    const int delta = lk - lq;
    // forward: query tiles of tok tokens
    for (int t0 = 0; t0 < lq; t0 += s.tok) {
      FwdItem it{};
      it.q_row = q0 + t0;
      it.q_len = std::min(s.tok, lq - t0);
      it.pos0 = t0 + delta;
      it.k_row = k0;
      it.lk = lk;
      it.prefix = P;
      it.seq = sq;
      const int p_lo = it.pos0, p_hi = it.pos0 + it.q_len - 1;
      // [0, a(p)) grows with p: tiles inside [0, a(p_lo)) are FULL for every row.
      const RowKeys lo = row_keys(p_lo, P, B, lk), hi = row_keys(p_hi, P, B, lk);
      it.n_full = lo.a / kTileN;
      it.r1_end = ceil_div(hi.a, kTileN);
      it.r2_begin = it.r2_end = 0;
      if (p_hi >= P) {  // copy rows: their own copies span [b(first copy row), e(p_hi))
        const RowKeys c = row_keys(std::max(p_lo, P), P, B, lk);
        int b0 = c.b / kTileN, b1 = ceil_div(hi.e, kTileN);
        if (b0 <= it.r1_end) {
          it.r1_end = std::max(it.r1_end, b1);
        } else {
          it.r2_begin = b0;
          it.r2_end = b1;
        }
      }
      it.work = it.r1_end + (it.r2_end - it.r2_begin);
      fw.push_back(it);
    }
    // backward: key tiles of 128 keys
    for (int kp = 0; kp < lk; kp += kTileN) {
      BwdItem it{};
      it.k_row = k0 + kp;
      it.k_len = std::min(kTileN, lk - kp);
      it.kpos0 = kp;
      it.q_row = q0;
      it.lq = lq;
      it.lk = lk;
      it.prefix = P;
      it.seq = sq;
      const KeyRows first = key_rows(kp, P, B, lk), last = key_rows(kp + it.k_len - 1, P, B, lk);
      const int hi = std::max(first.hi, last.hi);
      it.q_begin = std::max(0, first.lo - delta);
      it.q_end = std::min(lq, hi - delta);
      if (it.q_end < it.q_begin) it.q_end = it.q_begin;
      it.work = ceil_div(it.q_end - it.q_begin, s.tok) * (s.G / s.hg);
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
