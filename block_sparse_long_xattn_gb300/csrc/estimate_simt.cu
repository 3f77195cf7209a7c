// a1-a2 partial on CUDA cores: per-(row, key block) log-sum-exp of the scaled
// antidiagonal scores.
//
// docs/xattention_algorithm_guide.md "Stride Reshape 详解" (inverse mode):
// s[I,J] = sum_{t<S} q[I*S+S-1-t] . k[J*S+t]; the row softmax is over J <= I
// (global reshaped indices, the chunk starting at reshaped row q_start_pos/S,
// xattn_bsa.py select_blocks Step 0) with scale 1/(sqrt(d)*S).  This kernel
// writes, for every reshaped row I of the chunk and every key block kb at or
// before the row's diagonal block,
//   lse_part[b][h][kb][I] = ln sum_{J in kb, J <= I} exp(s[I,J] / (sqrt(d) S)).
// One CTA per (b, h, q-block): the q-block's 128 query tokens and, in turn,
// each causal key block's 128 key tokens are staged in shared memory as fp32.
// This is the exact-fp32 path (fp32 inputs); bf16 inputs take the tcgen05
// kernel.
#include "common.cuh"
#include "launchers.h"

namespace bsx {
namespace {

constexpr int kEstThreads = 256;

template <typename T, int S>
__global__ void __launch_bounds__(kEstThreads) estimate_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k, int q_len, int Lk, int Hq,
    int Hkv, int d, int cur, float scale, float* __restrict__ lse_part) {
  constexpr int RB = kBlock / S;          // reshaped rows per block
  constexpr int CELLS = RB * RB;
  constexpr int PARTS = CELLS >= kEstThreads ? 1 : kEstThreads / CELLS;
  extern __shared__ __align__(16) float sm[];
  const int ld = d + 1;                   // padded row stride (floats)
  float* Qs = sm;                         // [128][ld]
  float* Ks = Qs + kBlock * ld;           // [128][ld]
  float* part = Ks + kBlock * ld;         // [PARTS][CELLS]

  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (Hq / Hkv);
  const int nkb = Lk / kBlock;
  const int R = q_len / S;
  const int diag = cur + qb;
  const int tid = threadIdx.x;

  for (int e = tid; e < kBlock * d; e += kEstThreads) {
    const int r = e / d, c = e % d;
    Qs[r * ld + c] = to_f32(q[(((long long)b * q_len + qb * kBlock + r) * Hq + h) * d + c]);
  }
  for (int kb = 0; kb <= diag; ++kb) {
    __syncthreads();
    for (int e = tid; e < kBlock * d; e += kEstThreads) {
      const int r = e / d, c = e % d;
      Ks[r * ld + c] = to_f32(k[(((long long)b * Lk + kb * kBlock + r) * Hkv + hk) * d + c]);
    }
    __syncthreads();
    for (int w = tid; w < CELLS * PARTS; w += kEstThreads) {
      const int cell = w % CELLS, pt = w / CELLS;
      const int i = cell / RB, j = cell % RB;
      float acc = 0.f;
      for (int t = pt; t < S; t += PARTS) {
        const float* qr = Qs + (i * S + S - 1 - t) * ld;
        const float* kr = Ks + (j * S + t) * ld;
        for (int c = 0; c < d; ++c) acc = fmaf(qr[c], kr[c], acc);
      }
      part[pt * CELLS + cell] = acc;
    }
    __syncthreads();
    if (tid < RB) {
      const int i = tid;
      const int Ig = cur * RB + qb * RB + i;   // global reshaped row
      float x[RB];
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        float sc = 0.f;
        for (int pt = 0; pt < PARTS; ++pt) sc += part[pt * CELLS + i * RB + j];
        const int Jg = kb * RB + j;
        x[j] = (Jg <= Ig) ? sc * scale : -INFINITY;
        m = fmaxf(m, x[j]);
      }
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < RB; ++j) l += expf(x[j] - m);
      lse_part[((((long long)b * Hq + h) * (R / RB) + qb) * nkb + kb) * RB + i] = m + logf(l);
    }
  }
}

template <typename T, int S>
cudaError_t launch_typed(const Problem& p, const void* q, const void* k,
                         float* lse_part, cudaStream_t st) {
  constexpr int RB = kBlock / S;
  constexpr int CELLS = RB * RB;
  constexpr int PARTS = CELLS >= kEstThreads ? 1 : kEstThreads / CELLS;
  const size_t smem = (size_t)(2 * kBlock * (p.d + 1) + PARTS * CELLS) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(estimate_simt_kernel<T, S>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const float scale = 1.0f / (sqrtf((float)p.d) * (float)S);
  dim3 grid(p.nqb, p.Hq, p.B);
  estimate_simt_kernel<T, S><<<grid, kEstThreads, smem, st>>>(
      (const T*)q, (const T*)k, p.q_len, p.Lk, p.Hq, p.Hkv, p.d,
      p.q_start_pos / kBlock, scale, lse_part);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_stride(const Problem& p, const void* q, const void* k, int stride,
                          float* lse_part, cudaStream_t st) {
  switch (stride) {
    case 4: return launch_typed<T, 4>(p, q, k, lse_part, st);
    case 8: return launch_typed<T, 8>(p, q, k, lse_part, st);
    case 16: return launch_typed<T, 16>(p, q, k, lse_part, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_estimate_simt(const Problem& p, const void* q, const void* k,
                                 int stride, float* lse_part, cudaStream_t st) {
  if (p.dtype == 1) return launch_stride<__nv_bfloat16>(p, q, k, stride, lse_part, st);
  return launch_stride<float>(p, q, k, stride, lse_part, st);
}

}  // namespace bsx
