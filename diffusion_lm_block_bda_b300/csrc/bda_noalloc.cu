// bda_noalloc.cu -- bda_attn_fwd_noalloc: the forward without a workspace.
//
// Who needs it: callers that cannot call cudaMalloc (or hand out a
// workspace) at the point where they run attention -- for example a plugin
// inside an inference engine that owns every byte of device memory through
// its own pool and gives plugins none, or a decode loop that must not risk
// the device-wide synchronisation an allocation can cause.  The regular
// forward keeps its tile plan and status word in a caller-provided
// workspace; this variant keeps them in a fixed array compiled into the
// library instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (1 MiB): every GPU that loads the library holds it until the process
// exits.  Host code cannot use the array's name as a device address, so the
// first call on each device looks the address up with cudaGetSymbolAddress
// (with that device current) and caches it; make that first call before any
// stream capture begins on that device.  All calls share the one array and
// every call overwrites it (plan and a zeroed status word) before its kernel
// runs: calls whose work overlaps on the GPU -- on different streams, or from
// different host threads -- race on it and must be serialised by the caller.
#include <cstring>
#include <mutex>

#include "../../include/bda_attn.h"
#include "bda_host.h"
#include "bda_internal.h"
#include "bda_kernels.h"

namespace bda {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 2000000000ull;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Pageable staging copy of the plan: cudaMemcpyAsync returns once it has
// taken the bytes, so the buffer is free again when the call returns.
static uint8_t g_plan_staging[kNoAllocScratchBytes];
static std::mutex g_mu;
static void* g_scratch_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
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

bool thd_map(CUtensorMap* m, const void* ptr, int d, int heads, int64_t rows, int box_h,
             int box_rows) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(d) * 2 * cuuint64_t(heads)};
  cuuint32_t box[3] = {64, cuuint32_t(box_h), cuuint32_t(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bda_status fail_cuda(cudaError_t e) {
  note_cuda_error(cudaGetErrorString(e));
  return BDA_ERR_CUDA;
}

// Device address of g_noalloc_scratch on the current device (looked up once).
bda_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return BDA_ERR_UNSUPPORTED;
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e);
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return BDA_OK;
}

}  // namespace
}  // namespace bda

using namespace bda;

extern "C" {

bda_status bda_attn_fwd_noalloc(const bda_problem* prob, const bda_mask_desc* mask, const void* q,
                                const void* k, const void* v, void* o, float* lse,
                                bda_stream_t stream) {
  Shape s;
  bda_status st = validate(prob, mask, &s);
  if (st != BDA_OK) return st;
  const size_t need = plan_bytes(s);
  if (need > kNoAllocScratchBytes) return BDA_ERR_WORKSPACE;  // beyond the fixed 1 MiB
  if (s.n_fwd == 0) return BDA_OK;
  if (!q || !k || !v || !o || !lse) return BDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return BDA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv, to;
  if (!thd_map(&tq, q, s.d, s.hq, s.total_q, s.hg, s.tok) ||
      !thd_map(&tk, k, s.d, s.hkv, s.total_k, 1, kTileN) ||
      !thd_map(&tv, v, s.d, s.hkv, s.total_k, 1, kTileN) ||
      !thd_map(&to, o, s.d, s.hq, s.total_q, s.hg, s.tok)) {
    note_cuda_error("cuTensorMapEncodeTiled failed");
    return BDA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != BDA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // The plan (its header carries the zeroed status word) replaces whatever
  // the previous call left in the array.
  build_plan(prob, mask, s, g_plan_staging);
  cudaError_t e = cudaMemcpyAsync(scratch, g_plan_staging, need, cudaMemcpyHostToDevice, cs);
  if (e != cudaSuccess) return fail_cuda(e);
  FwdArgs a{};
  a.items = reinterpret_cast<const FwdItem*>(static_cast<uint8_t*>(scratch) + kHeaderBytes);
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = static_cast<uint32_t*>(scratch);
  a.timeout_ns = kTimeoutNs;
  a.n_groups = s.hq / s.hg;
  a.hg = s.hg;
  a.lg_hg = s.lg_hg;
  a.G = s.G;
  a.hq = s.hq;
  a.total_q = int(s.total_q);
  a.block = s.B;
  a.scale_log2 = s.scale * 1.4426950408889634f;
  e = launch_fwd(s.d, tq, tk, tv, to, a, s.n_fwd, cs);
  if (e != cudaSuccess) return fail_cuda(e);
  return BDA_OK;
}

}  // extern "C"
