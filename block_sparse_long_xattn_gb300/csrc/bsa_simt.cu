// a5 on CUDA cores: block-sparse causal attention with LSE, exact fp32 math.
//
// docs/xattention_algorithm_guide.md "BSA (Block Sparse Attention)": causal
// attention restricted to the selected 128x128 tiles of a per-head block
// mask; xattn_bsa.py compute_chunked_prefill takes O and LSE from each part.
// One CTA per (b, h, 128-row q-block), four threads per query row (each owns
// d/4 dimensions in an interleaved 16-byte pattern so a quad reads one
// contiguous 64-byte span of a shared-memory K/V row).  Key blocks outside
// [kb_begin, kb_end), after the diagonal, or not selected are skipped.  This
// is the fp32 path; bf16 inputs take the tcgen05 kernel.
#include "common.cuh"
#include "launchers.h"

namespace bsx {
namespace {

constexpr int kBsaThreads = 512;  // 128 rows x 4 threads
constexpr int kChunk = 16;        // keys scored before one softmax update

template <typename T, int D>
__global__ void __launch_bounds__(kBsaThreads) bsa_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const uint8_t* __restrict__ mask, int q_len, int Lk, int Hq, int Hkv,
    int cur, int kb_begin, int kb_end, float scale_log2, T* __restrict__ o,
    float* __restrict__ lse) {
  constexpr int DP = D / 4;      // dims per thread
  constexpr int NV4 = DP / 4;    // float4 groups per thread
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;                // [128][D]
  float* Vs = sm + kBlock * D;   // [128][D]

  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int nqb = gridDim.x;
  const int hk = h / (Hq / Hkv);
  const int nkb = Lk / kBlock;
  const int tid = threadIdx.x;
  const int row = tid >> 2, part = tid & 3;
  const int i_local = qb * kBlock + row;          // row within the chunk
  const int qpos = cur * kBlock + i_local;        // absolute query position
  const int diag = cur + qb;

  // this thread's dims: for g < NV4, e < 4: 16*g + 4*part + e
  float qr[DP], acc[DP];
  const T* qrow = q + (((long long)b * q_len + i_local) * Hq + h) * D;
#pragma unroll
  for (int g = 0; g < NV4; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qr[4 * g + e] = to_f32(qrow[16 * g + 4 * part + e]) * scale_log2;
      acc[4 * g + e] = 0.f;
    }
  float m = -INFINITY, l = 0.f;
  const uint8_t* mrow = mask + (((long long)b * Hq + h) * nqb + qb) * nkb;
  const int kb_last = min(kb_end, diag + 1);

  for (int kb = kb_begin; kb < kb_last; ++kb) {
    if (!mrow[kb]) continue;            // uniform across the CTA
    __syncthreads();
    for (int e = tid; e < kBlock * D; e += kBsaThreads) {
      const int r = e / D, c = e % D;
      const long long gi = (((long long)b * Lk + kb * kBlock + r) * Hkv + hk) * D + c;
      Ks[e] = to_f32(k[gi]);
      Vs[e] = to_f32(v[gi]);
    }
    __syncthreads();
    for (int j0 = 0; j0 < kBlock; j0 += kChunk) {
      float x[kChunk];
      float cmax = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < kChunk; ++jj) {
        const float4* kr = reinterpret_cast<const float4*>(Ks + (j0 + jj) * D) + part;
        float s = 0.f;
#pragma unroll
        for (int g = 0; g < NV4; ++g) {
          const float4 kv = kr[4 * g];
          s = fmaf(qr[4 * g + 0], kv.x, s);
          s = fmaf(qr[4 * g + 1], kv.y, s);
          s = fmaf(qr[4 * g + 2], kv.z, s);
          s = fmaf(qr[4 * g + 3], kv.w, s);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        const int kpos = kb * kBlock + j0 + jj;
        x[jj] = (kpos <= qpos) ? s : -INFINITY;
        cmax = fmaxf(cmax, x[jj]);
      }
      const float mnew = fmaxf(m, cmax);
      if (mnew != -INFINITY) {  // else nothing visible yet in this row
        const float alpha = exp2f(m - mnew);   // m = -inf -> 0
        l *= alpha;
#pragma unroll
        for (int c = 0; c < DP; ++c) acc[c] *= alpha;
        m = mnew;
      }
#pragma unroll
      for (int jj = 0; jj < kChunk; ++jj) {
        if (x[jj] == -INFINITY) continue;
        const float p = exp2f(x[jj] - m);
        l += p;
        const float4* vr = reinterpret_cast<const float4*>(Vs + (j0 + jj) * D) + part;
#pragma unroll
        for (int g = 0; g < NV4; ++g) {
          const float4 vv = vr[4 * g];
          acc[4 * g + 0] = fmaf(p, vv.x, acc[4 * g + 0]);
          acc[4 * g + 1] = fmaf(p, vv.y, acc[4 * g + 1]);
          acc[4 * g + 2] = fmaf(p, vv.z, acc[4 * g + 2]);
          acc[4 * g + 3] = fmaf(p, vv.w, acc[4 * g + 3]);
        }
      }
    }
  }
  T* orow = o + (((long long)b * q_len + i_local) * Hq + h) * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int g = 0; g < NV4; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) orow[16 * g + 4 * part + e] = from_f32<T>(acc[4 * g + e] * inv);
  if (part == 0)
    lse[((long long)b * Hq + h) * q_len + i_local] =
        l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
}

template <typename T, int D>
cudaError_t launch_typed(const Problem& p, const void* q, const void* k, const void* v,
                         const uint8_t* mask, int kb_begin, int kb_end, void* o,
                         float* lse, cudaStream_t st) {
  const size_t smem = (size_t)2 * kBlock * D * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bsa_simt_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  dim3 grid(p.nqb, p.Hq, p.B);
  bsa_simt_kernel<T, D><<<grid, kBsaThreads, smem, st>>>(
      (const T*)q, (const T*)k, (const T*)v, mask, p.q_len, p.Lk, p.Hq, p.Hkv,
      p.q_start_pos / kBlock, kb_begin, kb_end, scale_log2, (T*)o, lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bsa_simt(const Problem& p, const void* q, const void* k,
                            const void* v, const uint8_t* mask, int kb_begin,
                            int kb_end, void* o, float* lse, cudaStream_t st) {
  if (p.dtype == 1) {
    if (p.d == 64) return launch_typed<__nv_bfloat16, 64>(p, q, k, v, mask, kb_begin, kb_end, o, lse, st);
    return launch_typed<__nv_bfloat16, 128>(p, q, k, v, mask, kb_begin, kb_end, o, lse, st);
  }
  if (p.d == 64) return launch_typed<float, 64>(p, q, k, v, mask, kb_begin, kb_end, o, lse, st);
  return launch_typed<float, 128>(p, q, k, v, mask, kb_begin, kb_end, o, lse, st);
}

}  // namespace bsx
