// bda_bwd.cu -- backward block-causal / staircase attention for sm_103a.
//
// The staircase kernel of the ORL announcement thread (24vids.com mirror),
// Insight 3, serves training ("up to 5.2x faster training"), so it needs the
// gradients.  Textbook softmax-attention backward with the forward's LSE:
//   P = exp(scale S - LSE), dV = P^T dO, dP = dO V^T, D = rowsum(dO o O),
//   dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
// Three stages:
//   1. bwd_preprocess: D (fp32 [hq][total_q]) and a zeroed fp32 dQ accumulator.
//   2. bwd_dkdv: one CTA per (128-key tile, KV head).  dK and dV accumulate in
//      TMEM over every query tile (tok tokens x hg heads of the group) that
//      sees the key tile; the mask comes from block indices.  Per query tile:
//        S^T  = K Q^T            (tcgen05, TMEM)
//        P^T  -> bf16 TMEM       (softmax warps, thread = key row; written over
//                                 the S^T columns already read)
//        dP^T = V dO^T           (tcgen05, TMEM)
//        dV  += P^T dO           (tcgen05, A = P^T from TMEM)
//        dS^T -> bf16 smem       (softmax warps)
//        dK  += dS^T Q           (tcgen05)
//        dQ_t = dS K             (tcgen05, A = the same dS^T buffer read MN-major)
//      and a second warpgroup moves the dQ partial TMEM -> smem, from where
//      the TMA adds it into the fp32 accumulator (bulk tensor reduce-add).
//   3. dq_convert: dQ = bf16(scale * accumulator).
// Roles of the dK/dV kernel (512 threads, four warpgroups):
//   warps 0..3   softmax, query columns [0, 64) of each tile: P^T and dS^T,
//                then the dK epilogue
//   warps 4..7   softmax, query columns [64, 128), then the dV epilogue
//   warps 8..11  dQ readout + staging for the TMA reduce
//   warp 12      producer: K/V once, then Q, dO (TMA) and LSE, D per query tile
//   warp 13      MMA issuer of dV, dQ and dK (one thread)
//   warp 14      MMA issuer of S^T and dP^T (one thread)
//   warp 15      idle
// P and dS are elementwise in (key, query) given LSE and D, so the two
// softmax warpgroups split each tile's columns with no exchange; two warps
// per SM sub-partition hide each other's latencies on the chain
// S^T -> P^T -> dV -> S^T of the next tile.  The warpgroups rebalance
// registers (setmaxnreg): launched at 128 each, the last warpgroup gives
// 64 up, the softmax warpgroups take 144 and the dQ warpgroup 160.
// TMEM columns: S^T / P^T [0,128) dP^T / dQ [128,256) dK [256,256+D) dV [384,384+D).
#include <cuda_bf16.h>

#include "bda_internal.h"
#include "bda_kernels.h"
// The dK/dV kernel's warpgroups run under different register budgets.
#define BDA_INLINE_SLOW_WAITS 1
#include "bda_ptx.cuh"

namespace bda {

namespace {

// ------------------------------------------------------------- preprocess
template <int D>
__global__ void __launch_bounds__(256) bda_bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                                 const __nv_bfloat16* __restrict__ dout,
                                                                 float* __restrict__ Dv,
                                                                 float* __restrict__ dq_acc,
                                                                 int64_t total_q, int hq) {
  // A row is D/8 lanes x 16 bytes; each warp loads NR rows of O and dO
  // before reducing any (one row at a time leaves the loads latency-bound).
  constexpr int LPR = D / 8, RPI = 32 / LPR, NR = 8, NI = NR / RPI;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, col = (lane % LPR) * 8;
  const int64_t rows = total_q * hq;
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r0 = warp0 * NR; r0 < rows; r0 += nwarps * NR) {
    uint4 xo[NI], xd[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int64_t row = r0 + i * RPI + sub;
      if (row < rows) {
        xo[i] = *reinterpret_cast<const uint4*>(o + row * D + col);
        xd[i] = *reinterpret_cast<const uint4*>(dout + row * D + col);
      }
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int64_t row = r0 + i * RPI + sub;
      float acc = 0.f;
      if (row < rows) {
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&xo[i]);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&xd[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 x = __bfloat1622float2(a2[j]), y = __bfloat1622float2(b2[j]);
          acc = fmaf(x.x, y.x, acc);
          acc = fmaf(x.y, y.y, acc);
        }
        float4* z = reinterpret_cast<float4*>(dq_acc + row * D + col);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (row < rows && lane % LPR == 0) {
        const int64_t t = row / hq, h = row - t * hq;
        Dv[h * total_q + t] = acc;
      }
    }
  }
}

// ---------------------------------------------------------------- convert
__global__ void __launch_bounds__(256) bda_dq_convert_kernel(const float* __restrict__ acc,
                                                             __nv_bfloat16* __restrict__ dq,
                                                             int64_t n8, float scale) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 out;
    out.x = pack_bf16x2(a.x * scale, a.y * scale);
    out.y = pack_bf16x2(a.z * scale, a.w * scale);
    out.z = pack_bf16x2(b.x * scale, b.y * scale);
    out.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = out;
  }
}

// ------------------------------------------------------------------ dK/dV
constexpr int kBwdThreads = 512;
// Per-thread registers after the rebalancing (multiples of 8); per SM
// sub-partition one warp of each warpgroup: 144 + 144 + 160 + 64 = 512
// registers x 32 lanes = the launch's 128 x 4 warps.
constexpr int kRegsSoftmax = 144, kRegsDq = 160, kRegsOther = 64, kRegsLaunch = 128;
static_assert(2 * kRegsSoftmax + kRegsDq + kRegsOther == 4 * kRegsLaunch, "register split");
constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 384;
constexpr uint32_t kDqBarrier = 1;  // named barrier of the dQ warpgroup (warps 4..7)

// Shared memory (D = 128): K | V | Q x2 | dO | dS^T | dQ staging x2 | LSE x2 |
// D x2 | barriers = 226.1 KB, so there is no slack to align the base by hand:
// the kernel checks that the dynamic shared memory starts 1024-byte aligned.
template <int D>
struct BwdLayout {
  static constexpr int CH = D / 64;
  static constexpr int NQC = D / 32;            // 32-float chunks of a dQ row
  static constexpr uint32_t CHUNK = 128 * 128;  // [128 rows][128 B], 128B-swizzled
  static constexpr uint32_t TILE = CH * CHUNK;  // a K, V, Q or dO tile
  static constexpr uint32_t K = 0;
  static constexpr uint32_t V = K + TILE;
  static constexpr uint32_t Q = V + TILE;          // 2 stages
  static constexpr uint32_t DO = Q + 2 * TILE;     // 1 stage
  static constexpr uint32_t DS = DO + TILE;        // dS^T [128 keys][128 query cols] bf16
  static constexpr uint32_t STG = DS + 2 * CHUNK;  // dQ staging: 2 x [128 rows][32 fp32]
  static constexpr uint32_t LSE = STG + 2 * CHUNK;  // float[2][128]: LSE * log2(e) per query col
  static constexpr uint32_t DD = LSE + 1024;        // float[2][128]: D per query col
  static constexpr uint32_t BAR = DD + 1024;
  enum {
    B_KV = 0, B_QFULL = 1 /* [2] */, B_QEMPTY = 3 /* [2] */, B_DOFULL = 5, B_SFULL, B_PFULL,
    B_DVDONE, B_DPFULL, B_DSFULL, B_DQFULL, B_DQFREE, B_DSCONS, B_ACC, NBAR
  };
  static constexpr uint32_t MISC = BAR + 8 * NBAR;
  static constexpr uint32_t BYTES = MISC + 16;
};
static_assert(BwdLayout<128>::BYTES <= 232448, "backward shared memory budget");

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

__device__ __forceinline__ void expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Per (128-key tile, KV head) CTA; loops over the query tiles i that see the
// key tile.  Two threads issue the MMAs, per query tile i:
//   warp 14 (what the P/dS warps consume):
//     S^T_i = K Q_i^T      after Q_i landed and dV_{i-1} read P^T_{i-1}    -> SFULL
//     dP^T_i = V dO_i^T    after dO_i landed and dQ_{i-1} left TMEM       -> DPFULL
//   warp 13 (the gradients):
//     dV   += P_i^T dO_i   A = P^T from TMEM, after P_i^T is stored       -> DVDONE
//     dQ_i  = dS_i K       after dS_i^T is in smem (dP^T_i read)          -> DQFULL
//     dK   += dS_i^T Q_i                                                   -> DSCONS, QEMPTY
// MMAs into different accumulators are not ordered by the hardware, so every
// reuse of a TMEM region or smem buffer waits for a commit of its readers.
// The dQ partial of each query tile leaves TMEM through shared memory and is
// added to the fp32 accumulator by TMA reduce-add (per-element atomic), so no
// thread issues global atomics.
// MULTI: the plan has copy groups (multi-block staircase), so a key is seen
// by up to two query intervals and a key tile by up to two query ranges;
// block-causal and single-block staircase plans run the one-interval code.
template <int D, bool MULTI>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bda_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* gbase = smem_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (base & 1023u) {  // uniform across the CTA: nothing has been touched yet
    if (tid == 0) atomicOr(a.status, kSmemAlignCode);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return base + L::BAR + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::MISC + 4);

  const int item_idx = blockIdx.x / a.hkv;
  const int kvh = blockIdx.x - item_idx * a.hkv;
  const BwdItem it = a.items[item_idx];
  const int n_sub = a.G / a.hg;
  const int n_iter = it.work;  // query tiles: token tiles x head sub-groups
  const int delta = it.lk - it.lq;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar(L::B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::B_QFULL + s), 32);
      mbar_init(bar(L::B_QEMPTY + s), 1);
    }
    mbar_init(bar(L::B_DOFULL), 1);
    mbar_init(bar(L::B_SFULL), 1);
    mbar_init(bar(L::B_PFULL), 256);
    mbar_init(bar(L::B_DVDONE), 1);
    mbar_init(bar(L::B_DPFULL), 1);
    mbar_init(bar(L::B_DSFULL), 256);
    mbar_init(bar(L::B_DQFULL), 1);
    mbar_init(bar(L::B_DQFREE), 128);
    mbar_init(bar(L::B_DSCONS), 1);
    mbar_init(bar(L::B_ACC), 2);  // one commit from each MMA issuer
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // Register rebalancing: every role starts by setting its warpgroup's
  // budget (the decrease of warps 12..15 frees what the increases take; the
  // launch holds exactly kRegsLaunch per thread) and runs to the end of the
  // kernel on its own, so no code is shared between budgets.
  auto finish = [&]() {
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
      tc_fence_after();
      tmem_dealloc(tbase, 512);
    }
  };
  // Failure-detection testing: CTA 0 leaves its first Q tile un-issued and
  // unannounced and waits only fault_timeout_ns for it (a.fault is 0 in
  // normal use).
  const bool fault_cta = a.fault != 0 && blockIdx.x == 0;
  const WaitCtx wc{abort_flag, a.status, fault_cta ? a.fault_timeout_ns : a.timeout_ns};
  // Query tile i: token tile t0 (local) and head sub-group.  Tiles are walked
  // from the end of the sequence down, so the CTAs of one sequence, which
  // start together, sweep the same query rows at the same time (L2 reuse of
  // Q, dO and the dQ accumulator).
  // The query tokens come in one or two ranges (the second for copy groups
  // that see the tile's clean keys past groups that do not).
  const int n_tok_tiles =
      MULTI ? it.n_tiles1 + (it.q2_end - it.q2_begin + a.tok - 1) / a.tok : it.n_tiles1;
  auto tile_t0 = [&](int i) -> int {
    const int m = n_tok_tiles - 1 - i / n_sub;
    if (!MULTI) return it.q_begin + m * a.tok;
    return m < it.n_tiles1 ? it.q_begin + m * a.tok : it.q2_begin + (m - it.n_tiles1) * a.tok;
  };
  auto tile_h0 = [&](int i) -> int { return kvh * a.G + (i % n_sub) * a.hg; };

  bool ok = true;
  if (warp >= 12) {
    // One decrease for the whole warpgroup (warps 12..15), then its roles.
    setmaxnreg_dec<kRegsOther>();
    if (warp == 12) {
      // ------------------------------------------------------------ producer
      int nq0 = 0, nq1 = 0, ndo = 0;  // copies issued per barrier (abort drain)
      if (n_iter > 0) {
        if (lane == 0) {
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_k);
          tma_prefetch_desc(&tm_v);
          tma_prefetch_desc(&tm_do);
          mbar_arrive_expect_tx(bar(L::B_KV), 2 * L::TILE);
          for (int c = 0; c < L::CH; ++c) {
            tma_load_3d(base + L::K + c * L::CHUNK, &tm_k, bar(L::B_KV), c * 64, kvh, it.k_row);
            tma_load_3d(base + L::V + c * L::CHUNK, &tm_v, bar(L::B_KV), c * 64, kvh, it.k_row);
          }
        }
        // LSE and D of a query tile are fetched one tile ahead, into registers.
        float lv[4], dv[4];
        auto fetch = [&](int i) {
          const int t0 = tile_t0(i), h0 = tile_h0(i);
  #pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int col = lane + 32 * k;
            const int tok = t0 + (col >> a.lg_hg);
            const int h = h0 + (col & (a.hg - 1));
            // negated, so the P/dS warps add them in packed fp32 pairs
            lv[k] = -INFINITY;
            dv[k] = 0.f;
            if (tok < it.lq) {
              const size_t idx = size_t(h) * size_t(a.total_q) + size_t(it.q_row + tok);
              lv[k] = -(a.lse[idx] * 1.4426950408889634f);
              dv[k] = -a.D[idx];
            }
          }
        };
        fetch(0);
        for (int i = 0; i < n_iter; ++i) {
          const int st = i & 1;
          if (i >= 2 &&
              !mbar_wait_warp(wc, bar(L::B_QEMPTY + st), uint32_t((i >> 1) - 1) & 1u)) {
            ok = false;
            break;
          }
          const int t0 = tile_t0(i), h0 = tile_h0(i);
          const bool skip = fault_cta && i == 0;
          if (lane == 0 && !skip) {
            expect_tx(bar(L::B_QFULL + st), L::TILE);
            for (int c = 0; c < L::CH; ++c)
              tma_load_3d(base + L::Q + st * L::TILE + c * L::CHUNK, &tm_q, bar(L::B_QFULL + st),
                          c * 64, h0, it.q_row + t0);
          }
          float* s_lse = reinterpret_cast<float*>(gbase + L::LSE) + 128 * st;
          float* s_D = reinterpret_cast<float*>(gbase + L::DD) + 128 * st;
  #pragma unroll
          for (int k = 0; k < 4; ++k) {
            s_lse[lane + 32 * k] = lv[k];
            s_D[lane + 32 * k] = dv[k];
          }
          if (!skip) {
            mbar_arrive(bar(L::B_QFULL + st));
            if (st == 0) ++nq0; else ++nq1;
          }
          if (i + 1 < n_iter) fetch(i + 1);
          // dO has one buffer: tile i's once dV and dP^T of tile i-1 have read it
          // (two threads issue them, so neither commit covers the other)
          if (i >= 1 && !mbar_wait2_warp(wc, bar(L::B_DVDONE), uint32_t(i - 1) & 1u, bar(L::B_DPFULL),
                                         uint32_t(i - 1) & 1u)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(L::B_DOFULL), L::TILE);
            for (int c = 0; c < L::CH; ++c)
              tma_load_3d(base + L::DO + c * L::CHUNK, &tm_do, bar(L::B_DOFULL), c * 64, h0,
                          it.q_row + t0);
          }
          ++ndo;
        }
        if ((!ok || *abort_flag) && lane == 0) {
          drain_wait(wc, bar(L::B_KV), 0);
          if (nq0) drain_wait(wc, bar(L::B_QFULL), uint32_t(nq0 - 1) & 1u);
          if (nq1) drain_wait(wc, bar(L::B_QFULL + 1), uint32_t(nq1 - 1) & 1u);
          if (ndo) drain_wait(wc, bar(L::B_DOFULL), uint32_t(ndo - 1) & 1u);
        }
      }
    } else if (warp == 13 || warp == 14) {
      // ----------------------------------------------------------------- MMA
      // Two issuers, each waiting on the mbarriers of its own products: warp
      // 14 issues what the P/dS warps consume (S^T, dP^T), warp 13 the
      // gradients (dV, dQ, dK), lane 0 each.  A tcgen05.mma holds its issuing
      // thread until the pipe accepts it, so a single issuer queued every
      // product behind the issue of the one before.  The two meet only through
      // mbarriers: the next S^T waits for dV to have read P^T out of its
      // columns, the next dP^T for the dQ read-out, dQ for dS^T (which also
      // means dP^T was read).  Each commit tracks its own thread's MMAs.
      const bool score_issuer = warp == 14;
      auto wt = [&](int b, uint32_t parity) -> bool { return mbar_wait_warp(wc, bar(b), parity); };
      auto wt2 = [&](int b1, uint32_t p1, int b2, uint32_t p2) -> bool {
        return mbar_wait2_warp(wc, bar(b1), p1, bar(b2), p2);
      };
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t idAcc = idesc_bf16(128, D, false, true);    // dV, dK
      constexpr uint32_t idDQ = idesc_bf16(128, D, true, true);      // dQ
      // Lean issue (one add per operand per MMA, literal accumulate flag):
      // the issuing lane shares its sub-partition with a P/dS warp.
      auto issue_s = [&](int i) {  // S_i^T = K Q_i^T
        const uint32_t kl = opaque(sdesc_lo(base + L::K, 16));
        const uint32_t ql = opaque(sdesc_lo(base + L::Q + (i & 1) * L::TILE, 16));
        mma_ss_c<false>(tbase + kColS, sdesc_of_lo(kl), sdesc_of_lo(ql), idSS);
  #pragma unroll
        for (int kk = 1; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t(kk >> 2) * L::CHUNK + uint32_t(kk & 3) * 32u) >> 4;
          mma_ss_c<true>(tbase + kColS, sdesc_of_lo(kl + off), sdesc_of_lo(ql + off), idSS);
        }
        mma_commit(bar(L::B_SFULL));
      };
      auto issue_dp = [&]() {  // dP^T = V dO^T
        const uint32_t vl = opaque(sdesc_lo(base + L::V, 16));
        const uint32_t ol = opaque(sdesc_lo(base + L::DO, 16));
        mma_ss_c<false>(tbase + kColDP, sdesc_of_lo(vl), sdesc_of_lo(ol), idSS);
  #pragma unroll
        for (int kk = 1; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t(kk >> 2) * L::CHUNK + uint32_t(kk & 3) * 32u) >> 4;
          mma_ss_c<true>(tbase + kColDP, sdesc_of_lo(vl + off), sdesc_of_lo(ol + off), idSS);
        }
        mma_commit(bar(L::B_DPFULL));
      };
      bool go = true;
      if (n_iter > 0) {
        if (score_issuer) {
          for (int i = 0; go && i < n_iter; ++i) {
            const uint32_t ph = uint32_t(i) & 1u;
            // S_i^T once Q_i is in and dV_{i-1} has read P^T out of the S^T columns
            if (!(go = i == 0 ? wt2(L::B_KV, 0, L::B_QFULL, 0)
                              : wt2(L::B_QFULL + (i & 1), uint32_t(i >> 1) & 1u, L::B_DVDONE, ph ^ 1u)))
              break;
            tc_fence_after();
            if (lane == 0) issue_s(i);
            // dP_i^T once dO_i is in and dQ_{i-1} has left the dP^T columns
            if (!(go = i == 0 ? wt(L::B_DOFULL, 0) : wt2(L::B_DOFULL, ph, L::B_DQFREE, ph ^ 1u)))
              break;
            tc_fence_after();
            if (lane == 0) issue_dp();
          }
        } else {
          for (int i = 0; go && i < n_iter; ++i) {
            const uint32_t ph = uint32_t(i) & 1u;
            const int st = i & 1;
            // dV += P^T dO, P^T (bf16 pairs) in the S^T columns, once dO_i landed
            // (the other issuer's dP^T_i no longer stands between them)
            if (!(go = wt2(L::B_PFULL, ph, L::B_DOFULL, ph))) break;
            tc_fence_after();
            if (lane == 0) {
              const uint32_t ol = opaque(sdesc_lo(base + L::DO, L::CHUNK));
              mma_ts(tbase + kColDV, tbase + kColS, sdesc_of_lo(ol), idAcc, i > 0 ? 1u : 0u);
  #pragma unroll
              for (int kk = 1; kk < kTileM / 16; ++kk)
                mma_ts_c<true>(tbase + kColDV, tbase + kColS + 8u * kk + (kk >= 4 ? 32u : 0u),
                               sdesc_of_lo(ol + ((2048u * kk) >> 4)), idAcc);
              mma_commit(bar(L::B_DVDONE));
            }
            // dQ = dS K into the dP^T columns, then dK += dS^T Q
            if (!(go = wt(L::B_DSFULL, ph))) break;
            tc_fence_after();
            if (lane == 0) {
              const uint32_t sl = opaque(sdesc_lo(base + L::DS, L::CHUNK));
              const uint32_t kl = opaque(sdesc_lo(base + L::K, L::CHUNK));
              mma_ss_c<false>(tbase + kColDP, sdesc_of_lo(sl), sdesc_of_lo(kl), idDQ);
  #pragma unroll
              for (int kk = 1; kk < kTileN / 16; ++kk)
                mma_ss_c<true>(tbase + kColDP, sdesc_of_lo(sl + ((2048u * kk) >> 4)),
                               sdesc_of_lo(kl + ((2048u * kk) >> 4)), idDQ);
              mma_commit(bar(L::B_DQFULL));
              const uint32_t tl = opaque(sdesc_lo(base + L::DS, 16));
              const uint32_t ql = opaque(sdesc_lo(base + L::Q + st * L::TILE, L::CHUNK));
              mma_ss(tbase + kColDK, sdesc_of_lo(tl), sdesc_of_lo(ql), idAcc, i > 0 ? 1u : 0u);
  #pragma unroll
              for (int kk = 1; kk < kTileM / 16; ++kk) {
                const uint32_t aoff = (uint32_t(kk >> 2) * L::CHUNK + uint32_t(kk & 3) * 32u) >> 4;
                mma_ss_c<true>(tbase + kColDK, sdesc_of_lo(tl + aoff),
                               sdesc_of_lo(ql + ((2048u * kk) >> 4)), idAcc);
              }
              mma_commit(bar(L::B_DSCONS));
              mma_commit(bar(L::B_QEMPTY + st));
            }
          }
        }
        ok = go;
        if (lane == 0) {
          // The accumulator barrier takes one commit from each issuer: every
          // MMA has completed once it flips.
          mma_commit(bar(L::B_ACC));
          drain_wait(wc, bar(L::B_ACC), 0);
        }
      }
    }  // warp 15: idle
    finish();
  } else if (warp < 8) {
    // ------------------------------------------------------------- softmax
    setmaxnreg_inc<kRegsSoftmax>();
    const int kr = tid & 127;  // TMEM lane == key row of the tile
    const int half = warp >> 2;  // query columns [64 half, 64 half + 64)
    const int c0 = 2 * half;     // its 32-column chunks c0, c0 + 1
    const bool key_valid = kr < it.k_len;
    // Query positions that see this key: [lo, hi) and [lo2, hi2).
    const KeyRows kq = MULTI ? key_rows(it.kpos0 + kr, it.prefix, a.block, it.lk,
                                        a.cgroups + it.grp_off, it.n_grp)
                             : key_rows(it.kpos0 + kr, it.prefix, a.block, it.lk);
    const int q_hi = min(kq.hi - delta, it.lq);  // local query tokens [kq.lo - delta, q_hi)
    const int q2_lo = kq.lo2 - delta, q2_hi = min(kq.hi2 - delta, it.lq);
    const uint32_t lane_addr = tbase + (uint32_t((warp & 3) * 32) << 16);
    const uint64_t sl2x2 = f32x2(a.scale_log2, a.scale_log2);
    uint8_t* dsb = gbase + L::DS;
    for (int i = 0; i < n_iter; ++i) {
      const uint32_t ph = uint32_t(i) & 1u;
      const int st = i & 1;
      const float4* s_lse4 = reinterpret_cast<const float4*>(gbase + L::LSE) + 32 * st;
      const float4* s_D4 = reinterpret_cast<const float4*>(gbase + L::DD) + 32 * st;
      const int t0 = tile_t0(i);
      const int lo_c = key_valid ? kq.lo - delta - t0 : 0;
      const int hi_c = key_valid ? q_hi - t0 : 0;
      // Visible query columns of this key row: [c_lo, c_hi) (column = token
      // * hg + head).  Warps whose rows all see the whole tile skip masking.
      const int c_lo = max(lo_c, 0) << a.lg_hg;
      const int c_hi = hi_c <= lo_c ? c_lo : min(hi_c, a.tok) << a.lg_hg;
      int c_lo2 = 0, c_hi2 = 0;
      if (MULTI) {
        const int lo2_c = key_valid ? q2_lo - t0 : 0;
        const int hi2_c = key_valid ? q2_hi - t0 : 0;
        c_lo2 = max(lo2_c, 0) << a.lg_hg;
        c_hi2 = hi2_c <= lo2_c ? c_lo2 : min(hi2_c, a.tok) << a.lg_hg;
      }
      // Warps whose rows all see this warpgroup's 64 columns skip masking.
      const int h_lo = 64 * half, h_hi = h_lo + 64;
      const bool warp_full = __all_sync(0xffffffffu, (c_lo <= h_lo && c_hi >= h_hi) ||
                                                         (MULTI && c_lo2 <= h_lo && c_hi2 >= h_hi));
      // QFULL publishes the producer's LSE / D staging to these threads.
      if (!mbar_wait2_warp(wc, bar(L::B_QFULL + st), uint32_t(i >> 1) & 1u, bar(L::B_SFULL), ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P^T = exp(scale S^T - LSE), masked, 32 query columns at a time; the
      // bf16 pairs go back into this warpgroup's S^T columns already read
      // (chunk c fills columns [16c + 32 half, +16)) for the dV MMA, and stay
      // in registers for dS.
      uint32_t pp[kTileM / 4];
      auto p_chunk = [&](int c, const uint32_t (&r)[32]) {
        uint32_t pk[16];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 nl = s_lse4[8 * c + q4];  // -LSE * log2(e)
          float x0, x1, x2, x3;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[4 * q4 + 0]), __uint_as_float(r[4 * q4 + 1])),
                                sl2x2, f32x2(nl.x, nl.y)),
                      x0, x1);
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3])),
                                sl2x2, f32x2(nl.z, nl.w)),
                      x2, x3);
          pk[2 * q4] = pack_bf16x2(ex2(x0), ex2(x1));
          pk[2 * q4 + 1] = pack_bf16x2(ex2(x2), ex2(x3));
        }
        // Masking clears the bf16 halves of hidden columns.  It sits apart
        // from the exponentials: a branch between them would keep the
        // scheduler from overlapping their latencies.
        if (!warp_full) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = 32 * c + 2 * j;
            const bool v0 = (col >= c_lo && col < c_hi) || (MULTI && col >= c_lo2 && col < c_hi2);
            const bool v1 = (col + 1 >= c_lo && col + 1 < c_hi) ||
                            (MULTI && col + 1 >= c_lo2 && col + 1 < c_hi2);
            pk[j] &= (v0 ? 0x0000ffffu : 0u) | (v1 ? 0xffff0000u : 0u);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) pp[16 * (c - c0) + j] = pk[j];
        tmem_st16(lane_addr + kColS + 16u * uint32_t(c) + 32u * uint32_t(half), pk);
      };
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(lane_addr + kColS + 32u * uint32_t(c0), ra);
        tmem_ld32(lane_addr + kColS + 32u * uint32_t(c0 + 1), rb);
        tmem_ld_wait(ra);
        p_chunk(c0, ra);
        tmem_ld_wait(rb);
        p_chunk(c0 + 1, rb);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(L::B_PFULL));
      // dS^T = P^T o (dP^T - D) -> bf16 smem (K-major for dK, read MN-major for dQ);
      // the dS^T buffer is free once dQ and dK of the previous tile ran
      const bool dp_ok = i == 0 ? mbar_wait_warp(wc, bar(L::B_DPFULL), ph)
                                : mbar_wait2_warp(wc, bar(L::B_DSCONS), uint32_t(i - 1) & 1u,
                                                  bar(L::B_DPFULL), ph);
      if (!dp_ok) { ok = false; break; }
      tc_fence_after();
      auto ds_chunk = [&](int c, const uint32_t (&r)[32]) {
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const float4 d0 = s_D4[8 * c + 2 * u4], d1 = s_D4[8 * c + 2 * u4 + 1];  // -D
          const uint64_t nd[4] = {f32x2(d0.x, d0.y), f32x2(d0.z, d0.w), f32x2(d1.x, d1.y),
                                  f32x2(d1.z, d1.w)};
          uint32_t pk[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // dP - D in fp32 (a packed pair), rounded to a bf16 pair, times
            // the bf16 pair of P in one packed multiply (dS is stored as bf16
            // anyway).
            const int cc = 8 * u4 + 2 * j;
            float e0, e1;
            f32x2_split(add_f32x2(f32x2(__uint_as_float(r[cc]), __uint_as_float(r[cc + 1])), nd[j]),
                        e0, e1);
            pk[j] = mul_bf16x2(pp[16 * (c - c0) + 4 * u4 + j], pack_bf16x2(e0, e1));
          }
          const int u = 4 * c + u4;
          *reinterpret_cast<uint4*>(dsb + (u >> 3) * L::CHUNK + sw128_offset(kr, u & 7)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      };
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(lane_addr + kColDP + 32u * uint32_t(c0), ra);
        tmem_ld32(lane_addr + kColDP + 32u * uint32_t(c0 + 1), rb);
        tmem_ld_wait(ra);
        ds_chunk(c0, ra);
        tmem_ld_wait(rb);
        ds_chunk(c0 + 1, rb);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar(L::B_DSFULL));
    }
    // ------------------------------------------- dK (warps 0-3), dV (4-7)
    {
    const int row = tid & 127;
    const bool is_dk = warp < 4;
    const uint32_t lane_addr = tbase + (uint32_t((warp & 3) * 32) << 16);
    const bool have = n_iter > 0 && ok && !*abort_flag;
    bool acc_ok = false;
    if (have) acc_ok = mbar_wait_warp(wc, bar(L::B_ACC), 0);
    if (have && acc_ok) tc_fence_after();
    if (n_iter == 0 || acc_ok) {
      __nv_bfloat16* dst = (is_dk ? a.dk : a.dv) +
                           (size_t(it.k_row + row) * size_t(a.hkv) + size_t(kvh)) * size_t(D);
      const float mul = is_dk ? a.scale : 1.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        if (n_iter > 0) {
          tmem_ld32(lane_addr + (is_dk ? kColDK : kColDV) + 32u * c, rr);
          tmem_ld_wait(rr);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) rr[j] = 0u;
        }
        if (row < it.k_len) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_bf16x2(__uint_as_float(rr[2 * j]) * mul, __uint_as_float(rr[2 * j + 1]) * mul);
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int j = 0; j < 4; ++j) d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
    }
    }
    finish();
  } else if (warp < 12) {
    // ------------------------------------------- dQ: TMEM -> smem -> TMA add
    setmaxnreg_inc<kRegsDq>();
    const int qc = tid - 256;  // TMEM lane == query row of the tile
    const bool leader = qc == 0;
    const uint32_t lane_addr = tbase + (uint32_t((warp - 8) * 32) << 16);
    uint32_t n_chunks = 0;  // staging buffers handed to the TMA so far
    for (int i = 0; i < n_iter; ++i) {
      // All four warps leave together, so none is left at a named barrier.
      bool good = mbar_wait_warp(wc, bar(L::B_DQFULL), uint32_t(i) & 1u);
      good = named_bar_and(kDqBarrier, 128, good);
      if (!good) { ok = false; break; }
      tc_fence_after();
      uint32_t rq[L::NQC][32];
#pragma unroll
      for (int c = 0; c < L::NQC; ++c) tmem_ld32(lane_addr + kColDP + 32u * c, rq[c]);
#pragma unroll
      for (int c = 0; c < L::NQC; ++c) tmem_ld_wait(rq[c]);
      tc_fence_before();
      mbar_arrive(bar(L::B_DQFREE));
      const int t0 = tile_t0(i), h0 = tile_h0(i);
#pragma unroll
      for (int c = 0; c < L::NQC; ++c) {
        const uint32_t b = n_chunks & 1u;
        if (n_chunks >= 2) {  // the reduce that used buffer b has read it
          if (leader) bulk_wait_read<1>();
          named_bar_sync(kDqBarrier, 128);
        }
        uint8_t* stg = gbase + L::STG + b * L::CHUNK;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(stg + sw128_offset(qc, u)) =
              make_uint4(rq[c][4 * u], rq[c][4 * u + 1], rq[c][4 * u + 2], rq[c][4 * u + 3]);
        fence_proxy_async_smem();
        named_bar_sync(kDqBarrier, 128);
        if (leader) {
          tma_reduce_add_3d(&tm_dq, base + L::STG + b * L::CHUNK, 32 * c, h0, it.q_row + t0);
          bulk_commit();
        }
        ++n_chunks;
      }
    }
    if (leader) bulk_wait_all();
    finish();
  }

}

template <int D, bool MULTI>
cudaError_t launch_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a,
                          int n_items, cudaStream_t stream) {
  using L = BwdLayout<D>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = once_per_device(smem_set, [] {
    return cudaFuncSetAttribute(bda_bwd_dkdv_kernel<D, MULTI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(L::BYTES));
  });
  if (e != cudaSuccess) return e;
  // The warpgroups' register increases take exactly what the decrease frees
  // from a launch of kRegsLaunch per thread; any other allocation would leave
  // an increase waiting, so refuse to launch then.
  static const int regs = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, bda_bwd_dkdv_kernel<D, MULTI>) == cudaSuccess ? fa.numRegs : -1;
  }();
  if (regs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  const unsigned grid = unsigned(n_items) * unsigned(a.hkv);
  bda_bwd_dkdv_kernel<D, MULTI><<<grid, kBwdThreads, L::BYTES, stream>>>(tq, tk, tv, tdo, tdq, a);
  return cudaGetLastError();
}

int sm_count() {
  static int n = [] {
    int dev = 0, v = 148;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      return v;
    return 148;
  }();
  return n;
}

}  // namespace

cudaError_t launch_bwd_preprocess(int head_dim, const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                  float* D, float* dq_acc, int64_t total_q, int hq,
                                  cudaStream_t stream) {
  const int64_t rows = total_q * hq;
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + 63) / 64;  // 8 warps per block, 8 rows per warp per pass
  const int64_t cap = int64_t(sm_count()) * 8;  // 64 warps per SM
  if (blocks > cap) blocks = cap;
  if (head_dim == 128)
    bda_bwd_preprocess_kernel<128><<<unsigned(blocks), 256, 0, stream>>>(o, dout, D, dq_acc, total_q, hq);
  else
    bda_bwd_preprocess_kernel<64><<<unsigned(blocks), 256, 0, stream>>>(o, dout, D, dq_acc, total_q, hq);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                            const BwdArgs& a, int n_items, cudaStream_t stream) {
  if (n_items == 0) return cudaSuccess;
  const bool multi = a.cgroups != nullptr;
  if (head_dim == 128)
    return multi ? launch_dkdv_t<128, true>(tq, tk, tv, tdo, tdq, a, n_items, stream)
                 : launch_dkdv_t<128, false>(tq, tk, tv, tdo, tdq, a, n_items, stream);
  return multi ? launch_dkdv_t<64, true>(tq, tk, tv, tdo, tdq, a, n_items, stream)
               : launch_dkdv_t<64, false>(tq, tk, tv, tdo, tdq, a, n_items, stream);
}

cudaError_t launch_dq_convert(int head_dim, const float* dq_acc, __nv_bfloat16* dq, int64_t total_q,
                              int hq, float scale, cudaStream_t stream) {
  const int64_t n8 = total_q * hq * head_dim / 8;
  if (n8 == 0) return cudaSuccess;
  int64_t blocks = (n8 + 255) / 256;
  const int64_t cap = int64_t(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  bda_dq_convert_kernel<<<unsigned(blocks), 256, 0, stream>>>(dq_acc, dq, n8, scale);
  return cudaGetLastError();
}

}  // namespace bda
