// bda_fwd.cu -- forward block-causal / staircase attention for sm_103a.
//
// The forward of the attention the ORL announcement thread (24vids.com
// mirror), highlight 3, says was redesigned for block-causal masks, and the
// staircase replay of Insight 3 / the ORL paper card's Figure 3 caption.
// FlashAttention-style: per 128-row query tile the key tiles stream through
// shared memory and an online softmax keeps a running max and sum, so the
// L x L score matrix never exists.
//
// A work unit is (query tile, group of hg query heads); the tile is tok =
// 128/hg tokens x hg heads of one KV group, so the KV head's K/V tile feeds
// all 128 rows (GQA packing).  The kernel is persistent: one CTA per SM walks
// its share of the units (the planner's longest-first list, dealt out in
// snake order), and every pipeline (Q buffers, the K/V ring, S and P buffers)
// runs on across unit boundaries, so the next unit's loads and first S
// product overlap the current unit's last softmax and epilogue.  Roles:
//   warp 4        TMA producer of Q (two buffers) and K (NST-stage ring)
//   warp 7        TMA producer of V (NST-stage ring)
//   warp 6        tcgen05 issuer of S = Q K^T into TMEM (double buffered)
//   warp 5        tcgen05 issuer of O += P V, P read from TMEM
//   warps 0..3    softmax: thread r owns TMEM lane r = query row r; masks
//                 PARTIAL tiles from block indices, online max/sum, writes P
//                 as bf16 into TMEM, rescales O when the max grows by more
//                 than 2^8, and runs the epilogue (O / l, LSE).
// TMEM columns: S0 [0,128) S1 [128,256) O [256,256+D) P0 [384,448) P1 [448,512).
// S and P are both double buffered, so the softmax of tile n+1 overlaps the
// P V product of tile n; it waits for that product only to rescale O.
#include <cuda_bf16.h>

#include "bda_internal.h"
#include "bda_kernels.h"
#include "bda_ptx.cuh"

namespace bda {

namespace {

constexpr int kFwdThreads = 256;
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;  // P0 at kColP, P1 at kColP + 64
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only if the max grows by > 2^8

template <int D, int NST>
struct FwdLayout {
  static constexpr int CH = D / 64;              // 128-byte chunks of a head_dim row
  static constexpr uint32_t CHUNK = 128 * 128;   // one [128 rows][64 bf16] swizzled chunk
  static constexpr uint32_t TILE = CH * CHUNK;
  static constexpr uint32_t Q = 0;               // two buffers
  static constexpr uint32_t K = Q + 2 * TILE;
  static constexpr uint32_t V = K + NST * TILE;
  static constexpr uint32_t OSTG = V + NST * TILE;  // O staging for the TMA store
  static constexpr uint32_t BAR = OSTG + TILE;
  // q_full[2], q_empty[2], k_full[NST], v_full[NST], s_full[2], s_free[2],
  // p_full[2], o_done[2] (per P buffer), o_free[2] (per unit parity), drain.
  // Barriers that all softmax threads arrive on come in pairs: the S and P
  // buffers are double, so one softmax warp may finish tile g+1 before
  // another has finished tile g, and its arrivals must not count towards
  // tile g's phase (one p_full barrier let P V(g) start without the slow
  // warp's rows of P).  A warp reaches tile g+2 only after P V(g) completed,
  // which needs every warp's P(g), and the first P V of unit k+1 needs
  // every warp's o_free arrival for unit k, so two of each suffice.  With two K/V stages
  // and two S buffers, tile g uses stage g % 2 and buffer g % 2, so the
  // completion of S(g) frees K stage g % 2 and that of P V(g) frees V stage
  // g % 2: the producers wait on s_full / o_done (same phases) and the MMA
  // warp commits each product once (a commit costs the issuing lane tens of
  // cycles while the softmax warps move data through TMEM).
  static_assert(NST == 2, "K/V stages are released through the S and O barriers");
  static constexpr int B_QFULL = 0;
  static constexpr int B_QEMPTY = 2;
  static constexpr int B_KFULL = 4;
  static constexpr int B_VFULL = B_KFULL + NST;
  static constexpr int B_SFULL = B_VFULL + NST;
  static constexpr int B_SFREE = B_SFULL + 2;
  static constexpr int B_PFULL = B_SFREE + 2;
  static constexpr int B_ODONE = B_PFULL + 2;
  static constexpr int B_OFREE = B_ODONE + 2;
  static constexpr int B_DRAIN = B_OFREE + 2;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr uint32_t MISC = BAR + 8 * NBAR;
  static constexpr uint32_t BYTES = MISC + 16;
  static constexpr uint32_t ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
};

// Bounded wait that ignores the abort flag: used to let in-flight copies and
// MMAs land before a CTA leaves (normal path and abort path alike).
__device__ __forceinline__ bool drain_wait(WaitCtx w, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > w.timeout_ns) {
      atomicOr(w.status, kDeviceTimeoutCode);
      return false;
    }
  }
  return true;
}

// Bits of the columns [lo, hi) that fall in the 32-column word starting at w0.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int w0) {
  const int l = min(max(lo - w0, 0), 32), h = min(max(hi - w0, 0), 32);
  if (h <= l) return 0u;
  const uint32_t below_h = h == 32 ? 0xffffffffu : (1u << h) - 1u;
  const uint32_t below_l = l == 32 ? 0xffffffffu : (1u << l) - 1u;
  return below_h & ~below_l;
}

// The k-th unit (k = 0, 1, ...) of this CTA: units are dealt to the CTAs in
// snake order over the longest-first list (forward in even rounds, backward
// in odd ones), which evens out the CTAs' totals.  -1 past the end.
__device__ __forceinline__ int unit_of(int k, int n_units) {
  const int g = int(gridDim.x), c = int(blockIdx.x);
  const int u = k * g + ((k & 1) ? g - 1 - c : c);
  return u < n_units ? u : -1;
}

template <int D, int NST>
__global__ void __launch_bounds__(kFwdThreads, 1)
    bda_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdArgs a) {
  using L = FwdLayout<D, NST>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) -> uint32_t { return base + L::BAR + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::MISC + 4);
  const int n_units = a.n_units;

  if (tid == 0) {
    *abort_flag = 0;
    for (int q = 0; q < 2; ++q) {
      mbar_init(bar(L::B_QFULL + q), 1);
      mbar_init(bar(L::B_QEMPTY + q), 1);
    }
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(L::B_KFULL + s), 1);
      mbar_init(bar(L::B_VFULL + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::B_SFULL + b), 1);
      mbar_init(bar(L::B_SFREE + b), 128);
      mbar_init(bar(L::B_PFULL + b), 128);
      mbar_init(bar(L::B_ODONE + b), 1);
      mbar_init(bar(L::B_OFREE + b), 128);
    }
    mbar_init(bar(L::B_DRAIN), 2);  // one commit from each MMA issuer
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // Failure-detection testing: CTA 0 leaves its first Q load un-issued and
  // waits only fault_timeout_ns for it (a.fault is 0 in normal use).
  const bool fault_cta = a.fault != 0 && blockIdx.x == 0;
  const WaitCtx wc{abort_flag, a.status, fault_cta ? a.fault_timeout_ns : a.timeout_ns};

  // Unit u: work item, head group, and its key tiles.
  struct Unit {
    FwdItem it;
    int head0, kvh, n_tiles;
  };
  auto load_unit = [&](int u) -> Unit {
    Unit x;
    const int item_idx = u / a.n_groups;
    const int grp = u - item_idx * a.n_groups;
    x.it = a.items[item_idx];
    x.head0 = grp * a.hg;
    x.kvh = x.head0 / a.G;
    x.n_tiles = x.it.r1_end + (x.it.r2_end - x.it.r2_begin);
    return x;
  };
  auto key_tile = [](const FwdItem& it, int n) -> int {
    return n < it.r1_end ? n : it.r2_begin + (n - it.r1_end);
  };

  if (warp == 4 || warp == 7) {
    // ----------------------------------------------------------- producers
    // Warp 4 streams Q and K, warp 7 streams V.  With one producer, the load
    // of K(g+1) queued behind the wait for V(g)'s buffer, and the gate of
    // S(g+1) then waited on a late K.
    const bool kprod = warp == 4;
    if (lane == 0) {
      if (kprod) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
      } else {
        tma_prefetch_desc(&tm_v);
      }
      int nq[2] = {0, 0}, ncopy[NST];  // copies issued per barrier (abort drain)
      for (int s = 0; s < NST; ++s) ncopy[s] = 0;
      const int b_full = kprod ? L::B_KFULL : L::B_VFULL;
      // stage s of tile g is free once S(g - 2) (K) or P V(g - 2) (V) completed
      const int b_empty = kprod ? L::B_SFULL : L::B_ODONE;
      const CUtensorMap* tm = kprod ? &tm_k : &tm_v;
      const uint32_t ring = base + (kprod ? L::K : L::V);
      bool ok = true;
      int g = 0;  // key tiles streamed so far (all units)
      Unit nx{};  // the next unit's descriptor, fetched one unit ahead
      int u = unit_of(0, n_units);
      if (u >= 0) nx = load_unit(u);
      for (int k = 0; ok && u >= 0; ++k) {
        const Unit x = nx;
        u = unit_of(k + 1, n_units);
        if (u >= 0) nx = load_unit(u);
        if (kprod) {
          const int qb = k & 1;
          if (k >= 2 && !mbar_wait(wc, bar(L::B_QEMPTY + qb), uint32_t((k >> 1) - 1) & 1u)) {
            ok = false;
            break;
          }
          if (!(fault_cta && k == 0)) {
            mbar_arrive_expect_tx(bar(L::B_QFULL + qb), L::TILE);
            for (int c = 0; c < L::CH; ++c)
              tma_load_3d(base + L::Q + qb * L::TILE + c * L::CHUNK, &tm_q, bar(L::B_QFULL + qb),
                          c * 64, x.head0, x.it.q_row);
            ++nq[qb];
          }
        }
        for (int n = 0; n < x.n_tiles; ++n, ++g) {
          const int s = g % NST;
          const uint32_t ph = uint32_t(g / NST) & 1u;
          const int krow = x.it.k_row + key_tile(x.it, n) * kTileN;
          if (g >= NST && !mbar_wait(wc, bar(b_empty + s), ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(b_full + s), L::TILE);
          for (int c = 0; c < L::CH; ++c)
            tma_load_3d(ring + s * L::TILE + c * L::CHUNK, tm, bar(b_full + s), c * 64, x.kvh, krow);
          ++ncopy[s];
        }
      }
      if (!ok || *abort_flag) {
        // Let every copy already issued land before the CTA can exit.
        for (int q = 0; q < 2; ++q)
          if (nq[q]) drain_wait(wc, bar(L::B_QFULL + q), uint32_t(nq[q] - 1) & 1u);
        for (int s = 0; s < NST; ++s)
          if (ncopy[s]) drain_wait(wc, bar(b_full + s), uint32_t(ncopy[s] - 1) & 1u);
      }
    }
  } else if (warp == 5 || warp == 6) {
    // ----------------------------------------------------------------- MMA
    // Two issuers, each waiting on the mbarriers of its own products: warp 6
    // issues every S = Q K^T, warp 5 every O += P V (lane 0).  A tcgen05.mma
    // holds its issuing thread until the pipe accepts it, so with one issuer
    // S(g+1) could not start before all of P V(g-1) was issued, and that
    // chain (P out -> P V issue -> next S issue -> S done -> softmax) set the
    // tile period.  The two products share no operand (separate TMEM buffers,
    // K and V stages of their own) and each commit tracks only its own
    // thread's MMAs.
    const bool s_issuer = warp == 6;
    auto wt = [&](int b, uint32_t parity) -> bool { return mbar_wait_warp(wc, bar(b), parity); };
    auto wt2 = [&](int b1, uint32_t p1, int b2, uint32_t p2) -> bool {
      return mbar_wait2_warp(wc, bar(b1), p1, bar(b2), p2);
    };
    constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idO = idesc_bf16(128, D, false, true);
    // S(g) waits for K(g) and for the softmax to have read S(g-2) out of its buffer.
    auto s_ready = [&](int g) -> bool {
      const int s = g % NST, b = g & 1;
      return g < 2 ? wt(L::B_KFULL + s, uint32_t(g / NST) & 1u)
                   : wt2(L::B_SFREE + b, uint32_t((g >> 1) - 1) & 1u, L::B_KFULL + s,
                         uint32_t(g / NST) & 1u);
    };
    // The issuing lane shares its SM sub-partition with a softmax warp, so
    // each MMA is issued with as few instructions as possible: descriptors
    // are built from a 32-bit low word (the high word is one constant), each
    // K step adds a constant to it, and the accumulate flag is literal.
    // Same-box A/B on the packed replay: forward 0.97 -> 0.92 ms, dK/dV
    // 1.97 -> 1.85 ms against descriptors rebuilt per MMA.
    auto issue_s = [&](int g, int qb, bool last_of_unit) {
      const int s = g % NST, b = g & 1;
      const uint32_t ql = opaque(sdesc_lo(base + L::Q + qb * L::TILE, 16));
      const uint32_t kl = opaque(sdesc_lo(base + L::K + s * L::TILE, 16));
      const uint32_t dst = tbase + kColS + 128u * b;
      mma_ss_c<false>(dst, sdesc_of_lo(ql), sdesc_of_lo(kl), idS);
#pragma unroll
      for (int kk = 1; kk < D / 16; ++kk) {
        const uint32_t off = (uint32_t(kk >> 2) * L::CHUNK + uint32_t(kk & 3) * 32u) >> 4;
        mma_ss_c<true>(dst, sdesc_of_lo(ql + off), sdesc_of_lo(kl + off), idS);
      }
      mma_commit(bar(L::B_SFULL + b));  // also frees K stage s (s == b)
      if (last_of_unit) mma_commit(bar(L::B_QEMPTY + qb));
    };
    bool go = true;
    int g = 0;  // key tiles issued so far (all units)
    Unit nx{};  // the next unit's descriptor, fetched one unit ahead
    int u = unit_of(0, n_units);
    if (u >= 0) nx = load_unit(u);
    for (int k = 0; go && u >= 0; ++k) {
      const Unit x = nx;
      u = unit_of(k + 1, n_units);
      if (u >= 0) nx = load_unit(u);
      const int qb = k & 1;
      if (s_issuer) {
        // S(g) once its Q (first tile of a unit), its K and its S buffer are in
        for (int n = 0; n < x.n_tiles; ++n, ++g) {
          if (!(go = (n > 0 || wt(L::B_QFULL + qb, uint32_t(k >> 1) & 1u)) && s_ready(g))) break;
          tc_fence_after();
          if (lane == 0) issue_s(g, qb, n + 1 == x.n_tiles);
        }
      } else {
        // O += P V; the unit's first product overwrites O, so the previous
        // unit's epilogue must have read it out.
        for (int n = 0; n < x.n_tiles; ++n, ++g) {
          const int s = g % NST;
          if (!(go = wt2(L::B_VFULL + s, uint32_t(g / NST) & 1u, L::B_PFULL + (g & 1),
                         uint32_t(g >> 1) & 1u) &&
                     (n > 0 || k == 0 ||
                      wt(L::B_OFREE + ((k - 1) & 1), uint32_t((k - 1) >> 1) & 1u))))
            break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t vl = opaque(sdesc_lo(base + L::V + s * L::TILE, L::CHUNK));
            const uint32_t pa = tbase + kColP + 64u * (g & 1);
            mma_ts(tbase + kColO, pa, sdesc_of_lo(vl), idO, n > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 1; kk < kTileN / 16; ++kk)
              mma_ts_c<true>(tbase + kColO, pa + 8u * kk, sdesc_of_lo(vl + ((2048u * kk) >> 4)), idO);
            mma_commit(bar(L::B_ODONE + (g & 1)));  // also frees V stage s
          }
        }
      }
    }
    if (lane == 0) {
      // Every MMA this thread issued completes before TMEM can be released
      // (the drain barrier takes one commit from each issuer).
      mma_commit(bar(L::B_DRAIN));
      drain_wait(wc, bar(L::B_DRAIN), 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------- softmax
    const int r = tid;  // TMEM lane == query row of the tile
    const int t_local = r >> a.lg_hg;
    const int hh = r & (a.hg - 1);
    const uint32_t lane_addr = tbase + (uint32_t(warp * 32) << 16);
    const float sl2 = a.scale_log2;
    bool ok = true;
    int g = 0;  // key tiles consumed so far (all units)
    Unit nx{};  // the next unit's descriptor, fetched one unit ahead
    int u = unit_of(0, n_units);
    if (u >= 0) nx = load_unit(u);
    // A finished unit's epilogue: O out of TMEM (then the next unit's first
    // P V may overwrite it), O / l and LSE to global memory.  It runs after
    // the next unit's first P is out: by then its last P V has completed, and
    // the MMA warp has had that unit's first products to work on meanwhile.
    struct Pend {
      int head0, q_row, q_len, gl, k;  // the unit's head group, rows, last key tile, index
      float l, m;                      // its row sum and reference max
    };
    auto epilogue = [&](const Pend& pd) -> bool {
      if (!mbar_wait_warp(wc, bar(L::B_ODONE + (pd.gl & 1)), uint32_t(pd.gl >> 1) & 1u))
        return false;
        tc_fence_after();
        uint32_t ov[D / 32][32];
  #pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(lane_addr + kColO + 32u * c, ov[c]);
  #pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld_wait(ov[c]);
        tc_fence_before();
        mbar_arrive(bar(L::B_OFREE + (pd.k & 1)));
        const float inv_l = 1.f / pd.l;
        const bool row_valid = t_local < pd.q_len;
        if (pd.q_len == (kTileM >> a.lg_hg)) {
          // Whole tile: each warp's 32 rows (a quarter of the tile's tokens x
          // its hg heads) go to swizzled shared memory (conflict-free) and the
          // warp's lane 0 has the TMA write them (a store from each thread
          // would hit 32 rows per instruction).  The warp's previous store must
          // have read its part of the staging buffer first.
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
  #pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t pk[16];
  #pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[j] = pack_bf16x2(__uint_as_float(ov[c][2 * j]) * inv_l,
                                  __uint_as_float(ov[c][2 * j + 1]) * inv_l);
  #pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(gbase + L::OSTG + (c >> 1) * L::CHUNK +
                                        sw128_offset(r, 4 * (c & 1) + j)) =
                  make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int tok_w = kTileM >> (a.lg_hg + 2);  // tokens of one warp's 32 rows
            for (int c = 0; c < L::CH; ++c)
              tma_store_3d(&tm_o, base + L::OSTG + c * L::CHUNK + uint32_t(warp) * 4096u, 64 * c,
                           pd.head0, pd.q_row + warp * tok_w);
            bulk_commit();
          }
        } else if (row_valid) {
          // The sequence's last, partial tile: the box would spill into the
          // next sequence's rows, so each thread stores its own row.
          __nv_bfloat16* orow =
              a.o + (size_t(pd.q_row + t_local) * a.hq + size_t(pd.head0 + hh)) * size_t(D);
  #pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t pk[16];
  #pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[j] = pack_bf16x2(__uint_as_float(ov[c][2 * j]) * inv_l,
                                  __uint_as_float(ov[c][2 * j + 1]) * inv_l);
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
  #pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
        if (row_valid) {
          const float lse2 = pd.m + log2f(pd.l);
          a.lse[size_t(pd.head0 + hh) * size_t(a.total_q) + size_t(pd.q_row + t_local)] =
              lse2 * 0.69314718055994530942f;
        }
      return true;
    };
    Pend pend{};
    bool have_pend = false;
    for (int k = 0; ok && u >= 0; ++k) {
      const Unit x = nx;
      u = unit_of(k + 1, n_units);
      if (u >= 0) nx = load_unit(u);
      const FwdItem& it = x.it;
      const bool row_valid = t_local < it.q_len;
      const int p = it.pos0 + (row_valid ? t_local : it.q_len - 1);
      // Copy rows of a multi-block staircase see their group's clean keys.
      const RowKeys rk = row_keys_g(p, it.prefix, a.block, it.lk, a.cgroups + it.grp_off, it.n_grp);
      float m_ref = -INFINITY;  // running max of scale*log2(e)*S, the reference of P
      float l = 0.f;            // running sum of P (relative to m_ref)
      for (int n = 0; n < x.n_tiles; ++n, ++g) {
        const int b = g & 1;
        // S(g) and, for the P buffer b this tile writes, P V of tile g-2
        // (read out of b); one paired wait.
        const bool got = g < 2 ? mbar_wait_warp(wc, bar(L::B_SFULL + b), uint32_t(g >> 1) & 1u)
                               : mbar_wait2_warp(wc, bar(L::B_ODONE + b), uint32_t((g - 2) >> 1) & 1u,
                                                 bar(L::B_SFULL + b), uint32_t(g >> 1) & 1u);
        if (!got) { ok = false; break; }
        tc_fence_after();
        // All of S at once: four loads in flight, one wait.
        float sv[kTileN];
        {
          uint32_t rr[kTileN / 32][32];
#pragma unroll
          for (int c = 0; c < kTileN / 32; ++c)
            tmem_ld32(lane_addr + kColS + 128u * b + 32u * c, rr[c]);
#pragma unroll
          for (int c = 0; c < kTileN / 32; ++c) tmem_ld_wait(rr[c]);
#pragma unroll
          for (int c = 0; c < kTileN / 32; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j) sv[32 * c + j] = __uint_as_float(rr[c][j]);
        }
        tc_fence_before();
        mbar_arrive(bar(L::B_SFREE + b));
        if (n >= it.n_full) {  // PARTIAL tile: mask from block indices
          // Visible columns [0, ca) and [cb, ce) as four 32-bit masks, then
          // one bit test per score (a three-way compare per score cost as
          // much as the rest of the tile's softmax).
          const int k0 = key_tile(it, n) * kTileN;
          const int ca = rk.a - k0, cb = rk.b - k0, ce = rk.e - k0;
          uint32_t keep[kTileN / 32];
#pragma unroll
          for (int w = 0; w < kTileN / 32; ++w)
            keep[w] = range_bits(0, ca, 32 * w) | range_bits(cb, ce, 32 * w);
#pragma unroll
          for (int j = 0; j < kTileN; ++j)
            if (!(keep[j >> 5] & (1u << (j & 31)))) sv[j] = -INFINITY;
        }
        // Row max: three-input max in four independent chains (a single
        // chain would be 63 dependent steps).
        float mx4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) mx4[q] = fmaxf(sv[2 * q], sv[2 * q + 1]);
#pragma unroll
        for (int j = 8; j < kTileN; j += 8)
#pragma unroll
          for (int q = 0; q < 4; ++q) mx4[q] = max3f(mx4[q], sv[j + 2 * q], sv[j + 2 * q + 1]);
        const float mx = max3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
        const float m_cand = mx * sl2;
        float alpha = 1.f;
        if (m_cand > m_ref + kRescaleThreshold) {
          alpha = ex2(m_ref - m_cand);  // 0 on the first finite max
          m_ref = m_cand;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // A rescale needs O complete: wait for P V of the previous tile (rare
        // once the running max has settled).
        if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!mbar_wait_warp(wc, bar(L::B_ODONE + ((g - 1) & 1)), uint32_t((g - 1) >> 1) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(lane_addr + kColO + 32u * c, rr);
            tmem_ld_wait(rr);
#pragma unroll
            for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * alpha);
            tmem_st32(lane_addr + kColO + 32u * c, rr);
          }
        }
        // P = 2^(S*scale*log2(e) - m) on column pairs: the scaling FMA and the
        // row-sum adds run as packed fp32 pairs (two chains of pairs).
        const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(-m_use, -m_use);
        uint64_t rs2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < kTileN / 64; ++c) {
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(sv[64 * c + 2 * j], sv[64 * c + 2 * j + 1]), sl2x2, negm2),
                        x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            rs2[j & 1] = add_f32x2(rs2[j & 1], f32x2(p0, p1));
            pk[j] = pack_bf16x2(p0, p1);
          }
          tmem_st32(lane_addr + kColP + 64u * b + 32u * c, pk);
        }
        float r0, r1, r2, r3;
        f32x2_split(rs2[0], r0, r1);
        f32x2_split(rs2[1], r2, r3);
        l = l * alpha + ((r0 + r1) + (r2 + r3));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(L::B_PFULL + b));
        if (n == 0 && have_pend) {  // the previous unit's epilogue
          have_pend = false;
          if (!epilogue(pend)) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) break;
      pend = Pend{x.head0, it.q_row, it.q_len, g - 1, k, l, m_ref};
      have_pend = true;
    }
    if (ok && have_pend) ok = epilogue(pend);
    if (lane == 0) bulk_wait_all();  // the last O stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

int fwd_sm_count() {
  static int n = [] {
    int dev = 0, v = 148;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      return v;
    return 148;
  }();
  return n;
}

template <int D, int NST>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdArgs& a, int n_items, cudaStream_t stream) {
  using L = FwdLayout<D, NST>;
  static_assert(L::ALLOC <= 232448, "forward shared memory budget");
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = once_per_device(smem_set, [] {
    return cudaFuncSetAttribute(bda_fwd_kernel<D, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(L::ALLOC));
  });
  if (e != cudaSuccess) return e;
  FwdArgs args = a;
  args.n_units = n_items * a.n_groups;
  const int grid = args.n_units < fwd_sm_count() ? args.n_units : fwd_sm_count();
  bda_fwd_kernel<D, NST><<<unsigned(grid), kFwdThreads, L::ALLOC, stream>>>(tq, tk, tv, to, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& a, int n_items,
                       cudaStream_t stream) {
  if (n_items == 0) return cudaSuccess;
  if (head_dim == 128) return launch_fwd_t<128, 2>(tq, tk, tv, to, a, n_items, stream);
  return launch_fwd_t<64, 2>(tq, tk, tv, to, a, n_items, stream);
}

}  // namespace bda
