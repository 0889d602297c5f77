// bda_kernels.h -- launchers of the CUDA kernels (internal; the public surface
// is include/bda_attn.h).
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bda_host.h"
#include "bda_internal.h"

namespace bda {

// Runs `set` (a kernel attribute change) once per device for the call site
// that owns `done`: attributes persist, and changing one before every launch
// costs host time on each call.
template <typename F>
inline cudaError_t once_per_device(std::atomic<unsigned long long>& done, F set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  if ((e = set()) != cudaSuccess) return e;
  done.fetch_or(bit, std::memory_order_release);
  return cudaSuccess;
}

struct FwdArgs {
  const FwdItem* items;
  // Multi-block staircase: table of copy groups (x = first position of the
  // group in its sequence, y = clean keys its copies see); null otherwise.
  const int2* cgroups;
  __nv_bfloat16* o;
  float* lse;
  uint32_t* status;
  uint64_t timeout_ns;
  int n_groups;  // hq / hg: head groups per work item (a unit = item x group)
  int n_units;   // items x n_groups; set by launch_fwd
  int hg, lg_hg;
  int G;         // hq / hkv
  int hq;
  int total_q;
  int block;
  float scale_log2;  // softmax_scale * log2(e)
  // Failure-detection testing only (0 in normal use): when set, CTA 0 leaves
  // its first Q load un-issued, so the wait for it runs out after
  // fault_timeout_ns and the CTA takes its abort path.
  int fault;
  uint64_t fault_timeout_ns;
  // Split (decode) forward: its units, and the workspace's partial results
  // (null when the plan splits no item).
  const DecItem* dec;
  float* part_o;    // [n_parts * n_groups][D/4][128][4] fp32, normalised O of a chunk
  float* part_lse;  // [n_parts * n_groups][128] fp32, log2 LSE of a chunk
  // FP8 K/V: per-KV-head dequantisation scales (device, fp32 [hkv]).
  const float* k_scale;
  const float* v_scale;
};

struct BwdArgs {
  const BwdItem* items;
  const float* lse;      // [hq][total_q]
  const float* D;        // [hq][total_q]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  uint32_t* status;
  uint64_t timeout_ns;
  int hq, hkv, G;
  int hg, lg_hg, tok;
  int total_q;
  int block;
  float scale;       // softmax_scale
  float scale_log2;  // softmax_scale * log2(e)
  const int2* cgroups;  // as in FwdArgs
  int fault;           // as in FwdArgs (testing only)
  uint64_t fault_timeout_ns;
};

// Kernel arguments for a plan at `plan` (a workspace, or the no-alloc
// array) holding the items of `s` (with or without the backward items).
// Consumes a failure-detection test fault armed for that stage, if any.
FwdArgs make_fwd_args(const Shape& s, const uint8_t* plan, bool with_bwd, void* o, float* lse,
                      uint32_t* status, uint8_t* ws_parts = nullptr);
BwdArgs make_bwd_args(const Shape& s, const uint8_t* plan, const float* lse, const float* D,
                      void* dk, void* dv, uint32_t* status);

// to: map over O laid out like Q (box 64 x hg x tok / 4: one warp's 32 rows, 128-byte swizzle); whole
// query tiles are written through it.
cudaError_t launch_fwd(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& a, int n_items,
                       cudaStream_t stream);

// Split forward (one CTA per DecItem x head group; bf16 or e4m3 K/V) and,
// when `combine`, the merge of split items' partial results, launched as a
// programmatic dependent of the split kernel.
cudaError_t launch_decode(int head_dim, bool kv8, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const FwdArgs& a, int n_dec, int n_items,
                          bool combine, cudaStream_t stream);

// e4m3 codes of x / scale[h] (bf16 [rows][heads][d] -> bytes, same layout).
cudaError_t launch_quantize_fp8(const __nv_bfloat16* x, uint8_t* x8, const float* scale,
                                int64_t rows, int heads, int d, cudaStream_t stream);
// scale[h] = max |x[., h, .]| / 448 (1 for an all-zero head).
cudaError_t launch_fp8_scales(const __nv_bfloat16* x, float* scale, int64_t rows, int heads, int d,
                              cudaStream_t stream);

cudaError_t launch_bwd_preprocess(int head_dim, const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                  float* D, float* dq_acc, int64_t total_q, int hq,
                                  cudaStream_t stream);

// tdq: fp32 map over the dQ accumulator [total_q][hq][d] (unscaled sum of
// dS K), box 32 floats x hg heads x tok tokens, 128-byte swizzle.
cudaError_t launch_bwd_dkdv(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                            const BwdArgs& a, int n_items, cudaStream_t stream);

cudaError_t launch_dq_convert(int head_dim, const float* dq_acc, __nv_bfloat16* dq, int64_t total_q,
                              int hq, float scale, cudaStream_t stream);

}  // namespace bda
