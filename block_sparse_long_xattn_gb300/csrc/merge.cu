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

// One thread per 16-byte vector of o.  All vectors of one (b, i, h) row lie in
// one warp (d * sizeof(T) / 16 <= 32 for d <= 128), so the LSE of the row is
// read by the whole warp before one lane overwrites it.
template <typename T>
__global__ void __launch_bounds__(256) merge_kernel(
    int rows_total, int Hq, int q_len, int vec_per_row, T* __restrict__ o1,
    float* __restrict__ lse1, const T* __restrict__ o2,
    const float* __restrict__ lse2) {
  using V = Vec16<T>;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nvec = (long long)rows_total * vec_per_row;
  const bool active = gid < nvec;
  long long row = active ? gid / vec_per_row : 0;
  const int h = (int)(row % Hq);
  const long long bi = row / Hq;              // b * q_len + i
  const int i = (int)(bi % q_len);
  const long long b = bi / q_len;
  const long long lidx = (b * Hq + h) * q_len + i;
  float l1 = -INFINITY, l2 = -INFINITY;
  if (active) {
    l1 = lse1[lidx];
    l2 = lse2[lidx];
  }
  __syncwarp();
  if (!active) return;
  const float m = fmaxf(l1, l2);
  float w1 = 0.f, w2 = 0.f, lse = -INFINITY;
  if (m != -INFINITY) {
    w1 = __expf(l1 - m);   // exp(-inf) = 0 for an empty partial
    w2 = __expf(l2 - m);
    const float den = w1 + w2;
    lse = m + __logf(den);
    const float inv = 1.f / den;
    w1 *= inv;
    w2 *= inv;
  }
  V a, c;
  a.u = reinterpret_cast<const uint4*>(o1)[gid];
  c.u = reinterpret_cast<const uint4*>(o2)[gid];
#pragma unroll
  for (int e = 0; e < V::N; ++e)
    a.e[e] = from_f32<T>(w1 * to_f32(a.e[e]) + w2 * to_f32(c.e[e]));
  reinterpret_cast<uint4*>(o1)[gid] = a.u;
  if (gid % vec_per_row == 0) lse1[lidx] = lse;
}

}  // namespace

cudaError_t launch_merge(const Problem& p, void* o1, float* lse1, const void* o2,
                         const float* lse2, cudaStream_t st) {
  const int esize = p.dtype == 1 ? 2 : 4;
  const int vec_per_row = p.d * esize / 16;
  const long long rows = (long long)p.B * p.q_len * p.Hq;
  const long long nvec = rows * vec_per_row;
  if (nvec == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (nvec + threads - 1) / threads;
  if (p.dtype == 1)
    merge_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, st>>>(
        (int)rows, p.Hq, p.q_len, vec_per_row, (__nv_bfloat16*)o1, lse1,
        (const __nv_bfloat16*)o2, lse2);
  else
    merge_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(
        (int)rows, p.Hq, p.q_len, vec_per_row, (float*)o1, lse1,
        (const float*)o2, lse2);
  return cudaGetLastError();
}

}  // namespace bsx
