// bda_api.cu -- the extern "C" entry points declared in include/bda_attn.h.
//
// Host side of every call: validate the problem (nothing is launched on an
// argument error), encode the TMA tensor maps over the caller's THD tensors,
// and launch the kernels on the caller's stream.  No device memory is
// allocated here; scratch lives in the caller's workspace.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/bda_attn.h"
#include "bda_host.h"
#include "bda_internal.h"
#include "bda_kernels.h"
#include "bda_ptx.cuh"

namespace bda {
namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // bounded device waits: 2 s

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bda_status check_ws(const Shape& s, const void* ws, size_t ws_bytes, bool with_bwd) {
  if (!ws || !aligned16(ws)) return BDA_ERR_INVALID_ARG;
  if (ws_bytes < workspace_bytes(s, with_bwd)) return BDA_ERR_WORKSPACE;
  return BDA_OK;
}

thread_local const char* g_last_cuda_error = "";

bda_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return BDA_OK;
  g_last_cuda_error = cudaGetErrorString(e);
  return BDA_ERR_CUDA;
}

bda_status tensor_map_error() {
  g_last_cuda_error = "cuTensorMapEncodeTiled failed";
  return BDA_ERR_CUDA;
}

const uint8_t* plan_ptr(const void* ws) { return static_cast<const uint8_t*>(ws); }

}  // namespace

void note_cuda_error(const char* text) { g_last_cuda_error = text; }

// 3-D map over a THD bf16 tensor [rows][heads][d]; box = 64 head-dim elements
// (128 bytes, 128B swizzle) x box_h heads x box_rows rows.
bool make_thd_map(void* map, const void* ptr, int d, int heads, int64_t rows, int box_h,
                  int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  CUtensorMap* m = static_cast<CUtensorMap*>(map);
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(d) * 2 * cuuint64_t(heads)};
  cuuint32_t box[3] = {64, cuuint32_t(box_h), cuuint32_t(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the fp32 dQ accumulator [rows][heads][d]; box = 32 floats
// (128 bytes, 128B swizzle) x box_h heads x box_rows rows.
bool make_f32_map(void* map, const void* ptr, int d, int heads, int64_t rows, int box_h,
                  int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  CUtensorMap* m = static_cast<CUtensorMap*>(map);
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(d) * 4, cuuint64_t(d) * 4 * cuuint64_t(heads)};
  cuuint32_t box[3] = {32, cuuint32_t(box_h), cuuint32_t(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One-shot failure-detection fault (testing only): stage 1 = forward,
// 2 = backward dK/dV; consumed by the next launch of that stage.
std::atomic<int> g_fault_stage{0};
std::atomic<uint64_t> g_fault_timeout_ns{0};

uint64_t take_fault(int stage) {
  int want = stage;
  if (!g_fault_stage.compare_exchange_strong(want, 0)) return 0;
  return g_fault_timeout_ns.load();
}

// Forward kernel choice, testing only: 0 = by the plan (the split kernel
// when the plan splits its items), 1 = always the persistent kernel, 2 =
// always the split kernel.
std::atomic<int> g_force_fwd{0};

FwdArgs make_fwd_args(const Shape& s, const uint8_t* plan, bool with_bwd, void* o, float* lse,
                      uint32_t* status, uint8_t* ws_parts) {
  FwdArgs a{};
  a.dec = reinterpret_cast<const DecItem*>(plan + plan_dec_offset(s, with_bwd));
  if (ws_parts && s.n_parts > 0) {
    a.part_o = reinterpret_cast<float*>(ws_parts + ws_offset_parts(s));
    a.part_lse = reinterpret_cast<float*>(ws_parts + ws_offset_part_lse(s));
  }
  a.items = reinterpret_cast<const FwdItem*>(plan + kHeaderBytes);
  a.cgroups = s.n_cgroups > 0 ? reinterpret_cast<const int2*>(plan + plan_group_offset(s, with_bwd))
                              : nullptr;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = status;
  a.timeout_ns = kTimeoutNs;
  a.n_groups = s.hq / s.hg;
  a.hg = s.hg;
  a.lg_hg = s.lg_hg;
  a.G = s.G;
  a.hq = s.hq;
  a.total_q = int(s.total_q);
  a.block = s.B;
  a.scale_log2 = s.scale * 1.4426950408889634f;
  a.fault_timeout_ns = take_fault(1);
  a.fault = a.fault_timeout_ns != 0;
  return a;
}

BwdArgs make_bwd_args(const Shape& s, const uint8_t* plan, const float* lse, const float* D,
                      void* dk, void* dv, uint32_t* status) {
  BwdArgs a{};
  a.items = reinterpret_cast<const BwdItem*>(plan + kHeaderBytes + sizeof(FwdItem) * size_t(s.n_fwd));
  a.cgroups = s.n_cgroups > 0 ? reinterpret_cast<const int2*>(plan + plan_group_offset(s, true))
                              : nullptr;
  a.lse = lse;
  a.D = D;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.status = status;
  a.timeout_ns = kTimeoutNs;
  a.hq = s.hq;
  a.hkv = s.hkv;
  a.G = s.G;
  a.hg = s.hg;
  a.lg_hg = s.lg_hg;
  a.tok = s.tok;
  a.total_q = int(s.total_q);
  a.block = s.B;
  a.scale = s.scale;
  a.scale_log2 = s.scale * 1.4426950408889634f;
  a.fault_timeout_ns = take_fault(2);
  a.fault = a.fault_timeout_ns != 0;
  return a;
}

// 3-D map over e4m3 codes [rows][heads][d] (bytes); box = d codes x 1 head x
// 128 rows, no swizzle (the split kernel's threads expand the tile).
bool make_fp8_map(void* map, const void* ptr, int d, int heads, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  CUtensorMap* m = static_cast<CUtensorMap*>(map);
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(d), cuuint64_t(d) * cuuint64_t(heads)};
  cuuint32_t box[3] = {cuuint32_t(d), 1, cuuint32_t(kTileN)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace bda

using namespace bda;

extern "C" {

size_t bda_attn_plan_size(const bda_problem* prob, const bda_mask_desc* mask) {
  Shape s;
  if (validate(prob, mask, &s) != BDA_OK) return 0;
  return plan_bytes(s);
}

size_t bda_attn_workspace_size(const bda_problem* prob, const bda_mask_desc* mask, int with_bwd) {
  Shape s;
  if (validate(prob, mask, &s) != BDA_OK) return 0;
  return workspace_bytes(s, with_bwd != 0);
}

long long bda_attn_count_pairs(const bda_problem* prob, const bda_mask_desc* mask) {
  Shape s;
  if (validate(prob, mask, &s, /*count_only=*/true) != BDA_OK) return -1;
  return count_pairs(prob, mask, s);
}

bda_status bda_attn_plan_host(const bda_problem* prob, const bda_mask_desc* mask, void* host_plan,
                              size_t host_plan_bytes) {
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  if (!host_plan) return BDA_ERR_INVALID_ARG;
  if (host_plan_bytes < plan_bytes(s)) return BDA_ERR_WORKSPACE;
  build_plan(prob, mask, s, static_cast<uint8_t*>(host_plan));
  return BDA_OK;
}

bda_status bda_attn_plan(const bda_problem* prob, const bda_mask_desc* mask, void* host_plan,
                         size_t host_plan_bytes, void* ws, size_t ws_bytes, bda_stream_t stream) {
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  if (!host_plan) return BDA_ERR_INVALID_ARG;
  if (host_plan_bytes < plan_bytes(s)) return BDA_ERR_WORKSPACE;
  if ((st = check_ws(s, ws, ws_bytes, false)) != BDA_OK) return st;
  build_plan(prob, mask, s, static_cast<uint8_t*>(host_plan));
  return cuda_status(cudaMemcpyAsync(ws, host_plan, plan_bytes(s), cudaMemcpyHostToDevice,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

bda_status bda_attn_fwd(const bda_problem* prob, const bda_mask_desc* mask, const void* q,
                        const void* k, const void* v, void* o, float* lse, void* ws,
                        size_t ws_bytes, bda_stream_t stream) {
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes, false)) != BDA_OK) return st;
  if (s.n_fwd == 0) return BDA_OK;
  if (!q || !k || !v || !o || !lse) return BDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return BDA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv, to;
  if (!make_thd_map(&tq, q, s.d, s.hq, s.total_q, s.hg, s.tok) ||
      !make_thd_map(&tk, k, s.d, s.hkv, s.total_k, 1, kTileN) ||
      !make_thd_map(&tv, v, s.d, s.hkv, s.total_k, 1, kTileN) ||
      !make_thd_map(&to, o, s.d, s.hq, s.total_q, s.hg, s.tok / 4))
    return tensor_map_error();
  const FwdArgs a = make_fwd_args(s, plan_ptr(ws), /*with_bwd=*/true, o, lse,
                                  reinterpret_cast<uint32_t*>(ws), static_cast<uint8_t*>(ws));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // Problems that fill few SMs (a decode step) take the split kernel; the
  // persistent kernel ignores the plan's split units and computes every item.
  const int force = g_force_fwd.load();
  if (force == 2 || (force == 0 && s.split_c > 0))
    return cuda_status(launch_decode(s.d, false, tq, tk, tv, a, s.n_dec, s.n_fwd, s.n_parts > 0, cs));
  return cuda_status(launch_fwd(s.d, tq, tk, tv, to, a, s.n_fwd, cs));
}

bda_status bda_attn_fwd_fp8kv(const bda_problem* prob, const bda_mask_desc* mask, const void* q,
                              const void* k8, const void* v8, const float* k_scale,
                              const float* v_scale, void* o, float* lse, void* ws, size_t ws_bytes,
                              bda_stream_t stream) {
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes, false)) != BDA_OK) return st;
  if (s.n_fwd == 0) return BDA_OK;
  if (!q || !k8 || !v8 || !k_scale || !v_scale || !o || !lse) return BDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k8) || !aligned16(v8) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return BDA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv;
  if (!make_thd_map(&tq, q, s.d, s.hq, s.total_q, s.hg, s.tok) ||
      !make_fp8_map(&tk, k8, s.d, s.hkv, s.total_k) || !make_fp8_map(&tv, v8, s.d, s.hkv, s.total_k))
    return tensor_map_error();
  FwdArgs a = make_fwd_args(s, plan_ptr(ws), /*with_bwd=*/true, o, lse,
                            reinterpret_cast<uint32_t*>(ws), static_cast<uint8_t*>(ws));
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return cuda_status(launch_decode(s.d, true, tq, tk, tv, a, s.n_dec, s.n_fwd, s.n_parts > 0,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

bda_status bda_kv_quantize_fp8(const void* x, void* x8, const float* scale, long long rows,
                               int heads, int head_dim, bda_stream_t stream) {
  if (rows < 0 || heads <= 0 || (head_dim != 64 && head_dim != 128)) return BDA_ERR_INVALID_ARG;
  if (rows == 0) return BDA_OK;
  if (!x || !x8 || !scale || !aligned16(x) || !aligned16(x8) ||
      (reinterpret_cast<uintptr_t>(scale) & 3u))
    return BDA_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_fp8(static_cast<const __nv_bfloat16*>(x),
                                         static_cast<uint8_t*>(x8), scale, rows, heads, head_dim,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

bda_status bda_kv_fp8_scales(const void* x, float* scale, long long rows, int heads, int head_dim,
                             bda_stream_t stream) {
  if (rows < 0 || heads <= 0 || heads > 4096 || (head_dim != 64 && head_dim != 128))
    return BDA_ERR_INVALID_ARG;
  if (!scale || (reinterpret_cast<uintptr_t>(scale) & 3u) || (rows > 0 && (!x || !aligned16(x))))
    return BDA_ERR_INVALID_ARG;
  return cuda_status(launch_fp8_scales(static_cast<const __nv_bfloat16*>(x), scale, rows, heads,
                                       head_dim, reinterpret_cast<cudaStream_t>(stream)));
}

bda_status bda_attn_bwd_preprocess(const bda_problem* prob, const bda_mask_desc* mask,
                                   const void* o, const void* dout, void* ws, size_t ws_bytes,
                                   bda_stream_t stream) {
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes, true)) != BDA_OK) return st;
  if (s.total_q == 0) return BDA_OK;
  if (!o || !dout || !aligned16(o) || !aligned16(dout)) return BDA_ERR_INVALID_ARG;
  uint8_t* w = static_cast<uint8_t*>(ws);
  return cuda_status(launch_bwd_preprocess(
      s.d, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
      reinterpret_cast<float*>(w + ws_offset_D(s)), reinterpret_cast<float*>(w + ws_offset_dqacc(s)),
      s.total_q, s.hq, reinterpret_cast<cudaStream_t>(stream)));
}

bda_status bda_attn_bwd_dkdv(const bda_problem* prob, const bda_mask_desc* mask, const void* q,
                             const void* k, const void* v, const float* lse, const void* dout,
                             void* dk, void* dv, void* ws, size_t ws_bytes, bda_stream_t stream) {
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes, true)) != BDA_OK) return st;
  if (s.n_bwd == 0) return BDA_OK;
  if (!k || !v || !dk || !dv) return BDA_ERR_INVALID_ARG;
  if (s.total_q > 0 && (!q || !lse || !dout)) return BDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dk) || !aligned16(dv))
    return BDA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv, tdo, tdq;
  uint8_t* w = static_cast<uint8_t*>(ws);
  // A problem without queries still launches (dK = dV = 0); point the query
  // maps at the key tensor and the workspace, they are never accessed.
  const int64_t rq = s.total_q > 0 ? s.total_q : 1;
  const void* qsrc = s.total_q > 0 ? q : k;
  const void* dsrc = s.total_q > 0 ? dout : k;
  const void* accsrc = s.total_q > 0 ? static_cast<const void*>(w + ws_offset_dqacc(s)) : ws;
  const int hq_map = s.total_q > 0 ? s.hq : s.hkv;
  const int hg_map = s.total_q > 0 ? s.hg : 1;
  if (!make_thd_map(&tq, qsrc, s.d, hq_map, rq, hg_map, s.tok) ||
      !make_thd_map(&tdo, dsrc, s.d, hq_map, rq, hg_map, s.tok) ||
      !make_thd_map(&tk, k, s.d, s.hkv, s.total_k, 1, kTileN) ||
      !make_thd_map(&tv, v, s.d, s.hkv, s.total_k, 1, kTileN) ||
      !make_f32_map(&tdq, accsrc, s.d, s.total_q > 0 ? s.hq : 1, rq, hg_map, s.tok))
    return tensor_map_error();
  const BwdArgs a = make_bwd_args(s, w, lse, reinterpret_cast<const float*>(w + ws_offset_D(s)),
                                  dk, dv, reinterpret_cast<uint32_t*>(ws));
  return cuda_status(launch_bwd_dkdv(s.d, tq, tk, tv, tdo, tdq, a, s.n_bwd,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

bda_status bda_attn_bwd_dq_convert(const bda_problem* prob, const bda_mask_desc* mask, void* dq,
                                   void* ws, size_t ws_bytes, bda_stream_t stream) {
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes, true)) != BDA_OK) return st;
  if (s.total_q == 0) return BDA_OK;
  if (!dq || !aligned16(dq)) return BDA_ERR_INVALID_ARG;
  uint8_t* w = static_cast<uint8_t*>(ws);
  return cuda_status(launch_dq_convert(s.d, reinterpret_cast<const float*>(w + ws_offset_dqacc(s)),
                                       static_cast<__nv_bfloat16*>(dq), s.total_q, s.hq, s.scale,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

bda_status bda_attn_bwd(const bda_problem* prob, const bda_mask_desc* mask, const void* q,
                        const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                        bda_stream_t stream) {
  // Every argument of all three stages is checked before the first launch.
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  if ((st = check_ws(s, ws, ws_bytes, true)) != BDA_OK) return st;
  const void* need_q[] = {q, o, lse, dout, dq};
  const void* need_k[] = {k, v, dk, dv};
  for (const void* p : need_q)
    if ((s.total_q > 0 && !p) || !aligned16(p)) return BDA_ERR_INVALID_ARG;
  for (const void* p : need_k)
    if ((s.total_k > 0 && !p) || !aligned16(p)) return BDA_ERR_INVALID_ARG;
  st = bda_attn_bwd_preprocess(prob, mask, o, dout, ws, ws_bytes, stream);
  if (st != BDA_OK) return st;
  st = bda_attn_bwd_dkdv(prob, mask, q, k, v, lse, dout, dk, dv, ws, ws_bytes, stream);
  if (st != BDA_OK) return st;
  return bda_attn_bwd_dq_convert(prob, mask, dq, ws, ws_bytes, stream);
}

bda_status bda_attn_check_status(void* ws, size_t ws_bytes, bda_stream_t stream) {
  if (!ws || ws_bytes < sizeof(uint32_t)) return BDA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  bda_status r;
  if ((r = cuda_status(cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st))) != BDA_OK)
    return r;
  if ((r = cuda_status(cudaStreamSynchronize(st))) != BDA_OK) return r;
  if (v == 0) return BDA_OK;
  if ((r = cuda_status(cudaMemsetAsync(ws, 0, sizeof(uint32_t), st))) != BDA_OK) return r;
  if ((r = cuda_status(cudaStreamSynchronize(st))) != BDA_OK) return r;
  return (v & kDeviceTimeoutCode) ? BDA_ERR_DEVICE_TIMEOUT : BDA_ERR_UNSUPPORTED;
}

bda_status bda_testing_arm_wait_timeout(int stage, unsigned long long timeout_ns) {
  if (stage == 0) {
    g_fault_stage.store(0);
    return BDA_OK;
  }
  if ((stage != 1 && stage != 2) || timeout_ns < 1000ull || timeout_ns > 1000000000ull)
    return BDA_ERR_INVALID_ARG;
  g_fault_timeout_ns.store(timeout_ns);
  g_fault_stage.store(stage);
  return BDA_OK;
}

bda_status bda_testing_force_forward_kernel(int which) {
  if (which < 0 || which > 2) return BDA_ERR_INVALID_ARG;
  g_force_fwd.store(which);
  return BDA_OK;
}

const char* bda_last_cuda_error(void) { return g_last_cuda_error; }

const char* bda_status_string(bda_status s) {
  switch (s) {
    case BDA_OK: return "ok";
    case BDA_ERR_INVALID_ARG: return "invalid argument";
    case BDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case BDA_ERR_WORKSPACE: return "workspace or plan buffer too small";
    case BDA_ERR_CUDA: return "CUDA error";
    case BDA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
