// bda_fp8.cu -- FP8 (e4m3) KV cache: per-head scales and quantisation.
//
// The decode engine of the ORL paper card (thelatestinai.com, Table 11
// caption) runs its NVFP4 configurations with an FP8 KV cache.  The format
// here: K and V as e4m3 codes (OCP FP8: 1 sign, 4 exponent bits with bias 7,
// 3 mantissa bits; largest finite 448) with one fp32 dequantisation scale per
// KV head, value = code * scale[h].  Quantisation divides by the scale in
// fp32 (IEEE division) and rounds to the nearest e4m3 value, ties to even,
// saturating to +-448.  Both kernels are bound by HBM bandwidth.
#include <cuda_bf16.h>

#include "bda_kernels.h"
#include "bda_ptx.cuh"

namespace bda {
namespace {

// Eight bf16 -> eight e4m3 codes (bytes in element order).
__device__ __forceinline__ uint2 quantize8(uint4 x, float scale) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
    const float a = __fdiv_rn(lo, scale), b = __fdiv_rn(hi, scale);
    uint16_t c;
    // the first source lands in the upper byte: (b, a) puts a in the low byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(b), "f"(a));
    out[k >> 1] |= uint32_t(c) << (16 * (k & 1));
  }
  return make_uint2(out[0], out[1]);
}

__global__ void __launch_bounds__(256) bda_quantize_fp8_kernel(const uint4* __restrict__ x,
                                                               uint2* __restrict__ x8,
                                                               const float* __restrict__ scale,
                                                               int64_t n8, int heads, int d8) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const int h = int((i / d8) % heads);
    x8[i] = quantize8(x[i], scale[h]);
  }
}

__global__ void __launch_bounds__(32) bda_fp8_scales_init_kernel(float* scale, int heads) {
  for (int h = threadIdx.x; h < heads; h += 32) scale[h] = 0.f;
}

// max |x| per head into scale[] (as the bits of a non-negative float, whose
// integer order is the float order): each block reduces into shared memory,
// then adds one global atomic per head it saw.
__global__ void __launch_bounds__(256) bda_fp8_absmax_kernel(const uint4* __restrict__ x,
                                                             float* __restrict__ scale, int64_t n8,
                                                             int heads, int d8) {
  extern __shared__ unsigned int blk_max[];
  for (int h = threadIdx.x; h < heads; h += blockDim.x) blk_max[h] = 0u;
  __syncthreads();
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 v = x[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m = max(m, (w[k] << 16) & 0x7fffffffu);
      m = max(m, w[k] & 0x7fff0000u);
    }
    // NaN bits sort above every finite value; a NaN input yields a NaN scale
    if (m) atomicMax(blk_max + int((i / d8) % heads), m);
  }
  __syncthreads();
  for (int h = threadIdx.x; h < heads; h += blockDim.x)
    if (blk_max[h]) atomicMax(reinterpret_cast<unsigned int*>(scale) + h, blk_max[h]);
}

__global__ void __launch_bounds__(32) bda_fp8_scales_final_kernel(float* scale, int heads) {
  for (int h = threadIdx.x; h < heads; h += 32) {
    const float amax = scale[h];
    scale[h] = amax > 0.f ? amax / 448.f : (amax == 0.f ? 1.f : amax);
  }
}

int sm_count_fp8() {
  static int n = [] {
    int dev = 0, v = 148;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      return v;
    return 148;
  }();
  return n;
}

unsigned grid_for(int64_t n) {
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = int64_t(sm_count_fp8()) * 16;
  return unsigned(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_quantize_fp8(const __nv_bfloat16* x, uint8_t* x8, const float* scale,
                                int64_t rows, int heads, int d, cudaStream_t stream) {
  const int64_t n8 = rows * heads * d / 8;
  if (n8 == 0) return cudaSuccess;
  bda_quantize_fp8_kernel<<<grid_for(n8), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(x), reinterpret_cast<uint2*>(x8), scale, n8, heads, d / 8);
  return cudaGetLastError();
}

cudaError_t launch_fp8_scales(const __nv_bfloat16* x, float* scale, int64_t rows, int heads, int d,
                              cudaStream_t stream) {
  bda_fp8_scales_init_kernel<<<1, 32, 0, stream>>>(scale, heads);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n8 = rows * heads * d / 8;
  if (n8 > 0) {
    bda_fp8_absmax_kernel<<<grid_for(n8), 256, sizeof(unsigned int) * size_t(heads), stream>>>(
        reinterpret_cast<const uint4*>(x), scale, n8, heads, d / 8);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  bda_fp8_scales_final_kernel<<<1, 32, 0, stream>>>(scale, heads);
  return cudaGetLastError();
}

}  // namespace bda
