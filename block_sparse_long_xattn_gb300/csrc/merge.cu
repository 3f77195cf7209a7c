// a6: LSE merge of two partial attentions, in place into (o1, lse1).
//
// nano-vllm optimization guide, "Online Softmax Merge - Triton Fused Kernel":
// m = max(lse1, lse2), w_i = exp(lse_i - m), o = (w1 o1 + w2 o2)/(w1 + w2),
// lse = m + ln(w1 + w2).  The pages use two kernels (LSE, then output); here
// one HBM-bound pass reads each o row once with 16-byte vectors and updates
// its LSE in the same warp.
#include "common.cuh"
#include "launchers.h"

namespace bsx {
namespace {

// One thread per 16-byte vector of o.  All VPR vectors of one (b, i, h) row
// lie in one warp (VPR = d * sizeof(T) / 16 <= 32), so the LSE of the row is
// read by the whole warp before one lane overwrites it.  Index arithmetic is
// 32-bit whenever the problem allows it (Idx), and the row of a vector is a
// shift (VPR is a template parameter): the kernel moves 48 bytes per thread,
// and 64-bit divisions by runtime values would cost more than the copy.
template <typename T, int VPR, typename Idx>
__global__ void __launch_bounds__(256) merge_kernel(
    Idx rows_total, unsigned Hq, unsigned q_len, T* __restrict__ o1,
    float* __restrict__ lse1, const T* __restrict__ o2,
    const float* __restrict__ lse2) {
  using V = Vec16<T>;
  const Idx gid = (Idx)blockIdx.x * blockDim.x + threadIdx.x;
  const bool active = gid < rows_total * VPR;
  const Idx row = active ? gid / VPR : 0;     // (b * q_len + i) * Hq + h
  const Idx bi = row / Hq;
  const unsigned h = (unsigned)(row - bi * Hq);
  const Idx b = bi / q_len;
  const unsigned i = (unsigned)(bi - b * q_len);
  const Idx lidx = (b * Hq + h) * q_len + i;
  // the o vectors are loaded first: they do not depend on the LSEs, so both
  // round trips to memory overlap instead of following one another
  V a, c;
  float l1 = -INFINITY, l2 = -INFINITY;
  if (active) {
    a.u = reinterpret_cast<const uint4*>(o1)[gid];
    c.u = reinterpret_cast<const uint4*>(o2)[gid];
    l1 = lse1[lidx];
    l2 = lse2[lidx];
  }
  __syncwarp();
  if (!active) return;
  const MergeWeights w = merge_weights(l1, l2);
#pragma unroll
  for (int e = 0; e < V::N; ++e)
    a.e[e] = from_f32<T>(merge_element(w, to_f32(a.e[e]), to_f32(c.e[e])));
  reinterpret_cast<uint4*>(o1)[gid] = a.u;
  if (gid % VPR == 0) lse1[lidx] = w.lse;
}

template <typename T, int VPR>
cudaError_t launch_vpr(const Problem& p, void* o1, float* lse1, const void* o2,
                       const float* lse2, cudaStream_t st) {
  const long long rows = (long long)p.B * p.q_len * p.Hq;
  const long long nvec = rows * VPR;
  const int threads = 256;
  const long long blocks = (nvec + threads - 1) / threads;
  // 32-bit indices while every index (vectors and LSE entries) fits
  if (blocks * threads < (1LL << 31))
    merge_kernel<T, VPR, uint32_t><<<(unsigned)blocks, threads, 0, st>>>(
        (uint32_t)rows, p.Hq, p.q_len, static_cast<T*>(o1), lse1, static_cast<const T*>(o2),
        lse2);
  else
    merge_kernel<T, VPR, uint64_t><<<(unsigned)blocks, threads, 0, st>>>(
        (uint64_t)rows, p.Hq, p.q_len, static_cast<T*>(o1), lse1, static_cast<const T*>(o2),
        lse2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const Problem& p, void* o1, float* lse1, const void* o2,
                         const float* lse2, cudaStream_t st) {
  if ((long long)p.B * p.q_len * p.Hq == 0) return cudaSuccess;
  // vectors per row: d * sizeof(element) / 16
  if (p.dtype == 1)
    return p.d == 128 ? launch_vpr<__nv_bfloat16, 16>(p, o1, lse1, o2, lse2, st)
                      : launch_vpr<__nv_bfloat16, 8>(p, o1, lse1, o2, lse2, st);
  return p.d == 128 ? launch_vpr<float, 32>(p, o1, lse1, o2, lse2, st)
                    : launch_vpr<float, 16>(p, o1, lse1, o2, lse2, st);
}

}  // namespace bsx
