// bf16 -> e4m3 (fp8, 4 exponent bits, 3 mantissa bits, no infinities, largest
// finite 448), rounding to nearest even and saturating to +-448: the operand
// format of the estimator's fp8 path.  One thread converts 8 values (a
// 16-byte load, an 8-byte store) when the buffers allow it, else one value.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launchers.h"

namespace bsx {
namespace {

// two floats -> two e4m3 bytes, lo at the lower address
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(256) quantize8_kernel(const uint4* __restrict__ src,
                                                        uint2* __restrict__ dst, long long n8) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t b[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // a 32-bit word holds two bf16, the first in its low half
      const float f0 = __uint_as_float(w[e] << 16);
      const float f1 = __uint_as_float(w[e] & 0xFFFF0000u);
      b[e] = e4m3x2(f0, f1);
    }
    dst[i] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
  }
}

__global__ void __launch_bounds__(256) quantize1_kernel(const uint16_t* __restrict__ src,
                                                        uint8_t* __restrict__ dst, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = (uint8_t)(e4m3x2(__uint_as_float((uint32_t)src[i] << 16), 0.f) & 0xFFu);
}

}  // namespace

cudaError_t launch_quantize_e4m3(const void* src, uint8_t* dst, long long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool vec = n % 8 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dst) % 8 == 0;
  const long long units = vec ? n / 8 : n;
  long long blocks = (units + 255) / 256;
  if (blocks > (long long)sms * 16) blocks = (long long)sms * 16;  // grid-stride beyond
  if (vec)
    quantize8_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4*>(src),
                                                       reinterpret_cast<uint2*>(dst), units);
  else
    quantize1_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(src), dst,
                                                       units);
  return cudaGetLastError();
}

}  // namespace bsx
