// Device helpers shared by the kernels of the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bsx {

constexpr int kBlock = 128;  // BSA block size (fixed at 128 tokens)

// Error word layout: bits 0..7 kernel id, bits 8..15 wait site, bit 31 set.
enum ErrKernel : unsigned {
  kErrBsaTc = 1,
  kErrEstimateTc = 2,
  kErrFused = 3,  // the fused chunk step's waits for other CTAs' results
};
__device__ __forceinline__ void record_error(unsigned* err, unsigned kernel,
                                             unsigned site) {
  if (err) atomicCAS(err, 0u, 0x80000000u | (site << 8) | kernel);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// 16-byte vector of T elements.
template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  union {
    uint4 u;
    T e[N];
  };
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) as two two-input maxima.  (The three-input max.f32 of PTX was
// tried here and returned 0 for (-6.5, -inf, -inf) in one build of the
// attention kernel while the same source built differently got it right; a
// wrong row maximum only shifts the exponentials and stays within the output
// tolerance, so nothing would flag it.  Plain fmaxf is what the kernels use.)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  return fmaxf(fmaxf(a, b), c);
}

// LSE merge of two normalised partial attentions (nano-vllm optimization
// guide, "Online Softmax Merge"): the weights of (o1, o2) and the merged LSE
// from (lse1, lse2), and one merged element.  Written once with explicit
// rounding so that every kernel that merges produces the same bits.
struct MergeWeights {
  float w1, w2, lse;
};
__device__ __forceinline__ MergeWeights merge_weights(float l1, float l2) {
  const float m = fmaxf(l1, l2);
  MergeWeights r{0.f, 0.f, -INFINITY};
  if (m != -INFINITY) {
    // exp(-inf) = 0 for an empty partial; the differences are rounded on
    // their own, so that an LSE computed just before (not loaded) cannot fuse
    // into them
    r.w1 = __expf(__fsub_rn(l1, m));
    r.w2 = __expf(__fsub_rn(l2, m));
    const float den = __fadd_rn(r.w1, r.w2);
    r.lse = __fadd_rn(m, __logf(den));
    const float inv = __frcp_rn(den);
    r.w1 = __fmul_rn(r.w1, inv);
    r.w2 = __fmul_rn(r.w2, inv);
  }
  return r;
}
__device__ __forceinline__ float merge_element(const MergeWeights& w, float a, float c) {
  return __fmaf_rn(w.w1, a, __fmul_rn(w.w2, c));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace bsx
