// a2-a4: row normalisation, block sums and threshold block selection.
//
// Input: lse_part[b][h][qb][kb][r] = ln sum_{J in kb, J <= I} exp(s[I,J] / (sqrt(d) S))
// for the reshaped query rows I = q_start_pos/S + qb * 128/S + r of the chunk
// (written by the estimate kernels): one query block's partials are one
// contiguous run of nkb * 128/S floats.
// Then for one query block qb with rows I in qb:
//   LSE_I   = ln sum_kb exp(lse_part[kb][I])                 (row softmax denominator)
//   A[kb]   = sum_{I in qb} exp(lse_part[kb][I] - LSE_I)      (block sum of probabilities)
// which is the attn_sum of docs/xattention_algorithm_guide.md ("Triton Kernels
// 详解", softmax_fuse_block_sum) computed without materialising the scores.
//
// Selection ("块选择算法 (find_blocks_chunked)"): blocks 0 and the diagonal are
// forced; the others are sorted by descending A (ties: lower kb first) and
// taken while the cumulative mass, forced mass included, is below
// threshold * sum(A).  The crossing block is kept (the section's worked
// example); threshold >= 1 keeps every causal block.  One CTA per (b, h, qb):
// rows of at most 1024 key blocks take select_cta_kernel (everything in
// registers, warp shuffles and a few shared-memory stages); longer rows take
// select_kernel (a bitonic sort of packed (A, kb) keys in shared memory, then
// a block-wide exclusive scan of the sorted masses).
#include "common.cuh"
#include "launchers.h"

namespace bsx {
namespace {

constexpr int kSelThreads = 256;

__device__ __forceinline__ float block_reduce_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < 32) {
    t = (threadIdx.x < kSelThreads / 32) ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  return red[0];
}

template <int RB>  // reshaped rows per 128-token block, 128 / stride
__global__ void __launch_bounds__(kSelThreads) select_kernel(
    const float* __restrict__ lse_part, int Hq, int nkb, int cur,
    float threshold, uint8_t* __restrict__ mask, float* __restrict__ block_sums,
    int n_pad) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem_raw);  // n_pad
  float* sA = reinterpret_cast<float*>(keys + n_pad);                          // nkb
  uint8_t* sel = reinterpret_cast<uint8_t*>(sA + nkb);                         // nkb
  __shared__ float red_rows[kSelThreads / 32][RB];
  __shared__ float row_lse[RB];
  __shared__ float red[32];
  __shared__ float scan_tot[kSelThreads];

  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int nqb = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int diag = cur + qb;
  const int ncausal = diag + 1;
  const float* base = lse_part + ((long long)(b * Hq + h) * gridDim.x + qb) * nkb * RB;

  // ---- row maxima over key blocks ----
  float acc[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) acc[i] = -INFINITY;
  for (int kb = tid; kb < ncausal; kb += kSelThreads) {
    const float4* p = reinterpret_cast<const float4*>(base + (long long)kb * RB);
#pragma unroll
    for (int c = 0; c < RB / 4; ++c) {
      const float4 v = __ldg(p + c);
      acc[4 * c + 0] = fmaxf(acc[4 * c + 0], v.x);
      acc[4 * c + 1] = fmaxf(acc[4 * c + 1], v.y);
      acc[4 * c + 2] = fmaxf(acc[4 * c + 2], v.z);
      acc[4 * c + 3] = fmaxf(acc[4 * c + 3], v.w);
    }
  }
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    const float m = warp_max(acc[i]);
    if (lane == 0) red_rows[warp][i] = m;
  }
  __syncthreads();
  if (tid < RB) {
    float m = -INFINITY;
    for (int w = 0; w < kSelThreads / 32; ++w) m = fmaxf(m, red_rows[w][tid]);
    row_lse[tid] = m;  // row max for now
  }
  __syncthreads();
  float rmax[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) rmax[i] = row_lse[i];

  // ---- row sums -> row LSE ----
#pragma unroll
  for (int i = 0; i < RB; ++i) acc[i] = 0.f;
  for (int kb = tid; kb < ncausal; kb += kSelThreads) {
    const float4* p = reinterpret_cast<const float4*>(base + (long long)kb * RB);
#pragma unroll
    for (int c = 0; c < RB / 4; ++c) {
      const float4 v = __ldg(p + c);
      acc[4 * c + 0] += __expf(v.x - rmax[4 * c + 0]);
      acc[4 * c + 1] += __expf(v.y - rmax[4 * c + 1]);
      acc[4 * c + 2] += __expf(v.z - rmax[4 * c + 2]);
      acc[4 * c + 3] += __expf(v.w - rmax[4 * c + 3]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    const float s = warp_sum(acc[i]);
    if (lane == 0) red_rows[warp][i] = s;
  }
  __syncthreads();
  if (tid < RB) {
    float s = 0.f;
    for (int w = 0; w < kSelThreads / 32; ++w) s += red_rows[w][tid];
    row_lse[tid] += logf(s);  // it still holds the row max
  }
  __syncthreads();
  float rlse[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) rlse[i] = row_lse[i];

  // ---- block sums A[kb] ----
  float part_total = 0.f;
  for (int kb = tid; kb < nkb; kb += kSelThreads) {
    float a = 0.f;
    if (kb < ncausal) {
      const float4* p = reinterpret_cast<const float4*>(base + (long long)kb * RB);
#pragma unroll
      for (int c = 0; c < RB / 4; ++c) {
        const float4 v = __ldg(p + c);
        a += __expf(v.x - rlse[4 * c + 0]) + __expf(v.y - rlse[4 * c + 1]) +
             __expf(v.z - rlse[4 * c + 2]) + __expf(v.w - rlse[4 * c + 3]);
      }
    }
    sA[kb] = a;
    sel[kb] = 0;
    part_total += a;
    if (block_sums) block_sums[(((long long)b * Hq + h) * nqb + qb) * nkb + kb] = a;
  }
  const float total = block_reduce_sum(part_total, red);  // also syncs sA/sel

  uint8_t* mrow = mask + (((long long)b * Hq + h) * nqb + qb) * nkb;
  if (threshold >= 1.0f) {
    for (int kb = tid; kb < nkb; kb += kSelThreads) mrow[kb] = kb < ncausal ? 1 : 0;
    return;
  }

  // ---- sort candidates by (A desc, kb asc) ----
  for (int i = tid; i < n_pad; i += kSelThreads) {
    unsigned long long key = 0ull;
    if (i < ncausal && i != 0 && i != diag)
      key = ((unsigned long long)__float_as_uint(sA[i]) << 32) |
            (unsigned long long)(0xFFFFFFFFu - (unsigned)i);
    keys[i] = key;
  }
  __syncthreads();
  for (int k = 2; k <= n_pad; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < n_pad; i += kSelThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], c = keys[ixj];
          const bool first_half = (i & k) == 0;
          if (first_half ? (a < c) : (a > c)) {
            keys[i] = c;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- exclusive scan of sorted masses; keep while below the target ----
  const int nforced = diag == 0 ? 1 : 2;
  const int ncand = ncausal - nforced;
  const float forced_mass = sA[0] + (diag != 0 ? sA[diag] : 0.f);
  const float target = threshold * total;
  const int per = (n_pad + kSelThreads - 1) / kSelThreads;
  const int i0 = tid * per;
  float seg = 0.f;
  for (int e = 0; e < per; ++e) {
    const int i = i0 + e;
    if (i < ncand) seg += __uint_as_float((unsigned)(keys[i] >> 32));
  }
  // block exclusive scan of seg
  float incl = seg;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  if (tid < 32) {
    float w = tid < kSelThreads / 32 ? red[tid] : 0.f;
    float wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, wi, o);
      if (tid >= o) wi += n;
    }
    if (tid < kSelThreads / 32) scan_tot[tid] = wi - w;  // exclusive over warps
  }
  __syncthreads();
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  float run = scan_tot[warp] + excl;  // exclusive prefix before this segment
  for (int e = 0; e < per; ++e) {
    const int i = i0 + e;
    if (i < ncand) {
      const unsigned long long key = keys[i];
      const float v = __uint_as_float((unsigned)(key >> 32));
      if (forced_mass + run < target) sel[0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull)] = 1;
      run += v;
    }
  }
  __syncthreads();
  for (int kb = tid; kb < nkb; kb += kSelThreads) {
    uint8_t s = sel[kb];
    if (kb == 0 || kb == diag) s = 1;
    mrow[kb] = kb < ncausal ? s : 0;
  }
}

// ---------------------------------------------------------------------------
// The same computation for rows of at most 256 * E key blocks, one CTA of 256
// threads per (b, h, qb) row, with no phase that runs on a single warp:
//  1. every thread loads the partials of its key blocks kb = e * 256 + tid
//     (128/S consecutive floats each, all loads in flight at once) and
//     stores them transposed, vals[i][kb], in shared memory;
//  2. each reshaped row i is reduced by 256/RB threads (a max, then a sum of
//     exponentials written back over the partials, each followed by a
//     shuffle reduction inside the group): row_inv[i] = 1 / sum;
//  3. each thread sums its key blocks' probabilities over the rows: A[kb];
//     one block reduction gives the row total T;
//  4. a bitonic sort of packed (A, ~kb) 64-bit keys, descending, position
//     p = tid * E + e: partner distances below E are register swaps, below
//     32 E warp shuffles, the others go through shared memory (two buffers,
//     one barrier per stage);
//  5. an exclusive scan of the sorted masses (per thread, then per warp by
//     shuffles, then across warps), and every candidate whose exclusive mass
//     plus the forced mass is below threshold * T is selected.
template <int RB, int E>
__global__ void __launch_bounds__(kSelThreads) select_cta_kernel(
    const float* __restrict__ lse_part, int Hq, int nqb, int nkb, int cur,
    float threshold, uint8_t* __restrict__ mask, float* __restrict__ block_sums) {
  constexpr int NT = kSelThreads;
  constexpr int N = NT * E;                  // padded row length (a power of two)
  constexpr int GR = NT / RB;                // threads per row in step 2 (8, 16 or 32)
  constexpr int LD = N + (GR < 32 ? GR : 0);  // row stride: the row groups of a warp
                                              // read disjoint banks
  constexpr int NW = NT / 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* vals = reinterpret_cast<float*>(smem_raw);                              // [RB][LD]
  unsigned long long* kbuf = reinterpret_cast<unsigned long long*>(vals + RB * LD);  // [2][N]
  uint8_t* sel = reinterpret_cast<uint8_t*>(kbuf + 2 * N);                       // [N]
  __shared__ float row_inv[RB];
  __shared__ float red[NW];
  __shared__ float forced[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qb = blockIdx.x % nqb, h = blockIdx.x / nqb, b = blockIdx.y;
  const int diag = cur + qb;
  const int ncausal = diag + 1;
  const float* base = lse_part + ((long long)(b * Hq + h) * nqb + qb) * nkb * RB;

  // ---- 1. partials, transposed into shared memory ----
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int kb = e * NT + tid;
    float4 v[RB / 4];
    const float4* src = reinterpret_cast<const float4*>(base + (long long)kb * RB);
#pragma unroll
    for (int c = 0; c < RB / 4; ++c)
      v[c] = kb < ncausal ? __ldg(src + c) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
    for (int c = 0; c < RB / 4; ++c) {
      vals[(4 * c + 0) * LD + kb] = v[c].x;
      vals[(4 * c + 1) * LD + kb] = v[c].y;
      vals[(4 * c + 2) * LD + kb] = v[c].z;
      vals[(4 * c + 3) * LD + kb] = v[c].w;
    }
    sel[kb] = 0;
  }
  __syncthreads();

  // ---- 2. row softmax: GR threads per row; each exponential exp(x - m) is
  // written back over its partial, and the row keeps 1 / sum ----
  {
    const int i = tid / GR, j = tid % GR;
    float* rowp = vals + i * LD;
    float m = -INFINITY;
#pragma unroll
    for (int c = j; c < N; c += GR) m = fmaxf(m, rowp[c]);
#pragma unroll
    for (int o = GR / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int c = j; c < N; c += GR) {
      const float e = __expf(rowp[c] - m);
      rowp[c] = e;
      sum += e;
    }
#pragma unroll
    for (int o = GR / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (j == 0) row_inv[i] = 1.f / sum;
  }
  __syncthreads();

  // ---- 3. block sums A[kb] = sum_i exp(x - m_i) / sum_i, and the row total ----
  float a[E];
  float part = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int kb = e * NT + tid;
    float x = 0.f;
    if (kb < ncausal) {
#pragma unroll
      for (int i = 0; i < RB; ++i) x = fmaf(vals[i * LD + kb], row_inv[i], x);
    }
    a[e] = x;
    part += x;
    if (block_sums && kb < nkb) block_sums[(((long long)b * Hq + h) * nqb + qb) * nkb + kb] = x;
    if (kb == 0) forced[0] = x;
    if (kb == diag) forced[1] = x;
  }
  part = warp_sum(part);
  if (lane == 0) red[warp] = part;
  __syncthreads();
  float total = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) total += red[w];

  uint8_t* mrow = mask + (((long long)b * Hq + h) * nqb + qb) * nkb;
  if (threshold >= 1.0f) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int kb = e * NT + tid;
      if (kb < nkb) mrow[kb] = kb < ncausal ? 1 : 0;
    }
    return;
  }

  // ---- 4. bitonic sort of (A, kb) keys, descending (ties: lower kb first) ----
  unsigned long long key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int kb = e * NT + tid;
    key[e] = (kb < ncausal && kb != 0 && kb != diag)
                 ? ((unsigned long long)__float_as_uint(a[e]) << 32) |
                       (unsigned long long)(0xFFFFFFFFu - (unsigned)kb)
                 : 0ull;
  }
  int buf = 0;
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & j) == 0) {
            const int p = tid * E + e;  // lower position of the pair
            const bool desc = (p & k) == 0;
            const unsigned long long x = key[e], y = key[e | j];
            const bool swap = desc ? (x < y) : (x > y);
            key[e] = swap ? y : x;
            key[e | j] = swap ? x : y;
          }
        }
      } else if (j < 32 * E) {
        const bool lower = (tid & (j / E)) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int p = tid * E + e;
          const bool desc = (p & k) == 0;
          const unsigned long long y = __shfl_xor_sync(0xffffffffu, key[e], j / E);
          const unsigned long long x = key[e];
          key[e] = (lower == desc) ? (x > y ? x : y) : (x < y ? x : y);
        }
      } else {
        unsigned long long* kb_ = kbuf + buf * N;
#pragma unroll
        for (int e = 0; e < E; ++e) kb_[tid * E + e] = key[e];
        __syncthreads();
        const bool lower = (tid & (j / E)) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int p = tid * E + e;
          const bool desc = (p & k) == 0;
          const unsigned long long y = kb_[p ^ j];
          const unsigned long long x = key[e];
          key[e] = (lower == desc) ? (x > y ? x : y) : (x < y ? x : y);
        }
        buf ^= 1;
      }
    }
  }

  // ---- 5. exclusive scan of the sorted masses; keep while below the target ----
  float pre[E];
  float tsum = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    pre[e] = tsum;
    tsum += __uint_as_float((unsigned)(key[e] >> 32));
  }
  float incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();  // every thread is past its reads of red[]
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  float before = incl - tsum;  // exclusive within the warp
#pragma unroll
  for (int w = 0; w < NW; ++w)
    if (w < warp) before += red[w];
  const float forced_mass = forced[0] + (diag != 0 ? forced[1] : 0.f);
  const float target = threshold * total;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (key[e] != 0ull && forced_mass + (before + pre[e]) < target)
      sel[0xFFFFFFFFu - (unsigned)(key[e] & 0xFFFFFFFFull)] = 1;
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int kb = e * NT + tid;
    if (kb < nkb) mrow[kb] = (kb < ncausal && (kb == 0 || kb == diag || sel[kb])) ? 1 : 0;
  }
}

template <int RB, int E>
cudaError_t launch_cta(const Problem& p, float threshold, const float* lse_part,
                       uint8_t* mask, float* block_sums, cudaStream_t st) {
  constexpr int N = kSelThreads * E;
  constexpr int GR = kSelThreads / RB;
  constexpr int LD = N + (GR < 32 ? GR : 0);
  const size_t smem = (size_t)RB * LD * 4 + (size_t)2 * N * 8 + N;
  cudaError_t e = cudaFuncSetAttribute(select_cta_kernel<RB, E>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Hq * p.nqb, p.B);
  select_cta_kernel<RB, E><<<grid, kSelThreads, smem, st>>>(
      lse_part, p.Hq, p.nqb, p.nkb, p.q_start_pos / kBlock, threshold, mask, block_sums);
  return cudaGetLastError();
}

template <int RB>
cudaError_t launch_rb(const Problem& p, float threshold, const float* lse_part,
                      uint8_t* mask, float* block_sums, cudaStream_t st) {
  if (p.nkb <= 256) return launch_cta<RB, 1>(p, threshold, lse_part, mask, block_sums, st);
  if (p.nkb <= 512) return launch_cta<RB, 2>(p, threshold, lse_part, mask, block_sums, st);
  if (p.nkb <= 1024) return launch_cta<RB, 4>(p, threshold, lse_part, mask, block_sums, st);
  int n_pad = 1;
  while (n_pad < p.nkb) n_pad <<= 1;
  const size_t smem = (size_t)n_pad * 8 + (size_t)p.nkb * 4 + (size_t)p.nkb + 16;
  cudaError_t e = cudaFuncSetAttribute(select_kernel<RB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.nqb, p.Hq, p.B);
  select_kernel<RB><<<grid, kSelThreads, smem, st>>>(
      lse_part, p.Hq, p.nkb, p.q_start_pos / kBlock, threshold, mask,
      block_sums, n_pad);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(const Problem& p, int stride, float threshold,
                          const float* lse_part, uint8_t* mask, float* block_sums,
                          cudaStream_t st) {
  switch (stride) {
    case 4: return launch_rb<32>(p, threshold, lse_part, mask, block_sums, st);
    case 8: return launch_rb<16>(p, threshold, lse_part, mask, block_sums, st);
    case 16: return launch_rb<8>(p, threshold, lse_part, mask, block_sums, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace bsx
