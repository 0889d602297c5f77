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
// (with that device current) and caches it.  Each call writes the forward
// plan (with a zeroed status word) into the array through the parameters of
// a small copy kernel -- no host-to-device memcpy, so the call never waits
// for the stream's earlier work -- and then launches the forward.  All calls
// share the one array: calls whose work overlaps on the GPU (other streams,
// other host threads) race on it and must be serialised by the caller.  A
// stream that is being captured into a CUDA graph is refused.
#include <cstring>
#include <mutex>

#include "../../include/bda_attn.h"
#include "bda_host.h"
#include "bda_internal.h"
#include "bda_kernels.h"
#include "bda_ptx.cuh"

namespace bda {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Host staging of the plan; its bytes travel as kernel parameters, which the
// launch copies, so the buffer is free again as soon as a launch returns.
static uint8_t g_plan_staging[kNoAllocScratchBytes];
static std::mutex g_mu;
static void* g_scratch_dev[kMaxDevices];

// One launch carries up to kChunk16 16-byte units (the parameter space holds
// at most 32,764 bytes).
constexpr uint32_t kChunk16 = 1984;
struct PlanChunk {
  uint32_t offset16;  // destination offset in 16-byte units
  uint32_t n16;       // units in this chunk
  uint4 data[kChunk16];
};
static_assert(sizeof(PlanChunk) <= 32764, "kernel parameter space");

__global__ void __launch_bounds__(256) bda_plan_upload_kernel(const __grid_constant__ PlanChunk c) {
  uint4* dst = reinterpret_cast<uint4*>(g_noalloc_scratch) + c.offset16;
  for (uint32_t i = threadIdx.x; i < c.n16; i += blockDim.x) dst[i] = c.data[i];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bda_status fail_cuda(cudaError_t e) {
  note_cuda_error(cudaGetErrorString(e));
  return BDA_ERR_CUDA;
}

// Device address of g_noalloc_scratch on the current device (looked up once
// per device, with that device current).
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

// Refuses streams under capture: a captured call would bake this call's
// plan into the graph while the array it writes is shared with every other
// call.
bda_status refuse_capture(cudaStream_t cs) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(cs, &cap);
  if (e != cudaSuccess) return fail_cuda(e);
  return cap == cudaStreamCaptureStatusNone ? BDA_OK : BDA_ERR_UNSUPPORTED;
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
  const size_t need = plan_bytes(s, /*with_bwd=*/false);
  if (need > kNoAllocScratchBytes) return BDA_ERR_WORKSPACE;  // beyond the fixed 1 MiB
  if (s.n_fwd == 0) return BDA_OK;
  if (!q || !k || !v || !o || !lse) return BDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return BDA_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if ((st = refuse_capture(cs)) != BDA_OK) return st;
  CUtensorMap tq, tk, tv, to;
  if (!make_thd_map(&tq, q, s.d, s.hq, s.total_q, s.hg, s.tok) ||
      !make_thd_map(&tk, k, s.d, s.hkv, s.total_k, 1, kTileN) ||
      !make_thd_map(&tv, v, s.d, s.hkv, s.total_k, 1, kTileN) ||
      !make_thd_map(&to, o, s.d, s.hq, s.total_q, s.hg, s.tok / 4)) {
    note_cuda_error("cuTensorMapEncodeTiled failed");
    return BDA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != BDA_OK) return st;
  // The plan (its header carries the zeroed status word) replaces whatever
  // the previous call left in the array.
  build_plan(prob, mask, s, g_plan_staging, /*with_bwd=*/false);
  const size_t n16 = (need + 15) / 16;
  static PlanChunk chunk;  // guarded by g_mu; too large for the stack of some threads
  for (size_t u = 0; u < n16; u += kChunk16) {
    chunk.offset16 = uint32_t(u);
    chunk.n16 = uint32_t(n16 - u < kChunk16 ? n16 - u : kChunk16);
    std::memcpy(chunk.data, g_plan_staging + 16 * u, 16 * size_t(chunk.n16));
    bda_plan_upload_kernel<<<1, 256, 0, cs>>>(chunk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e);
  }
  FwdArgs a = make_fwd_args(s, static_cast<const uint8_t*>(scratch), /*with_bwd=*/false, o, lse,
                            static_cast<uint32_t*>(scratch));
  cudaError_t e = launch_fwd(s.d, tq, tk, tv, to, a, s.n_fwd, cs);
  if (e != cudaSuccess) return fail_cuda(e);
  return BDA_OK;
}

bda_status bda_attn_fwd_noalloc_check_status(bda_stream_t stream) {
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  bda_status st = refuse_capture(cs);
  if (st != BDA_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != BDA_OK) return st;
  cudaError_t e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return fail_cuda(e);
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_noalloc_scratch, sizeof(v), 0, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  if (v == 0) return BDA_OK;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail_cuda(e);
  return (v & kDeviceTimeoutCode) ? BDA_ERR_DEVICE_TIMEOUT : BDA_ERR_UNSUPPORTED;
}

}  // extern "C"
