// a2-a4: row normalisation, block sums and threshold block selection.
//
// Input: lse_part[b][h][kb][I] = ln sum_{J in kb, J <= I} exp(s[I,J] / (sqrt(d) S))
// for the reshaped query rows I of the chunk (written by the estimate kernels).
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
// a bitonic sort of packed (A, kb) keys in shared memory, then a block-wide
// exclusive scan of the sorted masses.  Rows of at most 1024 key blocks take
// select_warp_kernel instead: one warp per (b, h, qb), everything in
// registers and warp shuffles.
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
    const float* __restrict__ lse_part, int Hq, int nkb, int R, int cur,
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
  const float* base = lse_part + ((long long)(b * Hq + h) * nkb) * R + qb * RB;

  // ---- row maxima over key blocks ----
  float acc[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) acc[i] = -INFINITY;
  for (int kb = tid; kb < ncausal; kb += kSelThreads) {
    const float4* p = reinterpret_cast<const float4*>(base + (long long)kb * R);
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
    const float4* p = reinterpret_cast<const float4*>(base + (long long)kb * R);
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
      const float4* p = reinterpret_cast<const float4*>(base + (long long)kb * R);
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
// The same computation with one warp per (b, h, qb) row, for rows of at most
// 32 * KPL key blocks.  Element i of the row (key block i before sorting,
// sorted position i after) lives in lane i % 32, register i / 32, so every
// compare-exchange of the bitonic network is either a warp shuffle (partner
// distance below 32) or a swap between two registers of one lane; no block
// barrier is needed anywhere.
constexpr int kWarpsPerCta = 4;

// One bitonic stage between registers t and t + TJ of every lane (element
// i = t * 32 + lane; partner distance 32 * TJ); descending runs where
// (i & k) == 0.
template <int KPL, int TJ>
__device__ __forceinline__ void bitonic_regs(unsigned long long (&key)[KPL], int k, int lane) {
  if constexpr (TJ < KPL) {
#pragma unroll
    for (int t = 0; t < KPL; ++t) {
      if ((t & TJ) == 0) {
        const int i = t * 32 + lane;  // lower index of the pair
        const bool desc = (i & k) == 0;
        const unsigned long long x = key[t], y = key[t | TJ];
        const bool swap = desc ? (x < y) : (x > y);
        key[t] = swap ? y : x;
        key[t | TJ] = swap ? x : y;
      }
    }
  }
}

template <int RB, int KPL>
__global__ void __launch_bounds__(32 * kWarpsPerCta, (KPL <= 8 && RB <= 16) ? 4 : 2) select_warp_kernel(
    const float* __restrict__ lse_part, int Hq, int nqb, int nkb, int R, int cur,
    float threshold, uint8_t* __restrict__ mask, float* __restrict__ block_sums) {
  constexpr int N = 32 * KPL;  // padded row length (a power of two)
  __shared__ __align__(16) uint8_t sel_all[kWarpsPerCta][N];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int row_id = blockIdx.x * kWarpsPerCta + wid;  // (h, qb) flattened
  if (row_id >= Hq * nqb) return;
  const int qb = row_id % nqb;
  const int h = row_id / nqb;
  const int b = blockIdx.y;
  uint8_t* sel = sel_all[wid];
  const int diag = cur + qb;
  const int ncausal = diag + 1;
  const float* base = lse_part + ((long long)(b * Hq + h) * nkb) * R + qb * RB;

  // ---- row maxima, then row sums -> row LSE ----
  float acc[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) acc[i] = -INFINITY;
#pragma unroll 4
  for (int kb = lane; kb < ncausal; kb += 32) {
    const float4* q = reinterpret_cast<const float4*>(base + (long long)kb * R);
#pragma unroll
    for (int c = 0; c < RB / 4; ++c) {
      const float4 v = __ldg(q + c);
      acc[4 * c + 0] = fmaxf(acc[4 * c + 0], v.x);
      acc[4 * c + 1] = fmaxf(acc[4 * c + 1], v.y);
      acc[4 * c + 2] = fmaxf(acc[4 * c + 2], v.z);
      acc[4 * c + 3] = fmaxf(acc[4 * c + 3], v.w);
    }
  }
  float rmax[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    rmax[i] = warp_max(acc[i]);
    acc[i] = 0.f;
  }
#pragma unroll 4
  for (int kb = lane; kb < ncausal; kb += 32) {
    const float4* q = reinterpret_cast<const float4*>(base + (long long)kb * R);
#pragma unroll
    for (int c = 0; c < RB / 4; ++c) {
      const float4 v = __ldg(q + c);
      acc[4 * c + 0] += __expf(v.x - rmax[4 * c + 0]);
      acc[4 * c + 1] += __expf(v.y - rmax[4 * c + 1]);
      acc[4 * c + 2] += __expf(v.z - rmax[4 * c + 2]);
      acc[4 * c + 3] += __expf(v.w - rmax[4 * c + 3]);
    }
  }
  float rlse[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) rlse[i] = rmax[i] + logf(warp_sum(acc[i]));

  // ---- block sums A[kb], kb = t * 32 + lane ----
  float a[KPL];
  float part = 0.f;
#pragma unroll
  for (int t = 0; t < KPL; ++t) {
    const int kb = t * 32 + lane;
    float v = 0.f;
    if (kb < ncausal) {
      const float4* q = reinterpret_cast<const float4*>(base + (long long)kb * R);
#pragma unroll
      for (int c = 0; c < RB / 4; ++c) {
        const float4 w = __ldg(q + c);
        v += __expf(w.x - rlse[4 * c + 0]) + __expf(w.y - rlse[4 * c + 1]) +
             __expf(w.z - rlse[4 * c + 2]) + __expf(w.w - rlse[4 * c + 3]);
      }
    }
    a[t] = v;
    part += v;
    if (block_sums && kb < nkb) block_sums[(((long long)b * Hq + h) * nqb + qb) * nkb + kb] = v;
  }
  const float total = warp_sum(part);

  uint8_t* mrow = mask + (((long long)b * Hq + h) * nqb + qb) * nkb;
  if (threshold >= 1.0f) {
    for (int kb = lane; kb < nkb; kb += 32) mrow[kb] = kb < ncausal ? 1 : 0;
    return;
  }

  // ---- bitonic sort of (A, kb) keys, descending (ties: lower kb first) ----
  unsigned long long key[KPL];
#pragma unroll
  for (int t = 0; t < KPL; ++t) {
    const int kb = t * 32 + lane;
    key[t] = (kb < ncausal && kb != 0 && kb != diag)
                 ? ((unsigned long long)__float_as_uint(a[t]) << 32) |
                       (unsigned long long)(0xFFFFFFFFu - (unsigned)kb)
                 : 0ull;
  }
  // For 1024-key rows the stage loops stay rolled and only the per-register
  // work is unrolled: their fully unrolled network overflows the instruction
  // cache.  Register distances (partner 32 or more elements away) dispatch
  // to bodies with a compile-time distance, so no register is indexed at
  // run time; for 256-key rows everything unrolls.
  auto stage = [&](int k, int j) {
    if (j >= 32) {
      switch (j >> 5) {
        case 1: bitonic_regs<KPL, 1>(key, k, lane); break;
        case 2: bitonic_regs<KPL, 2>(key, k, lane); break;
        case 4: bitonic_regs<KPL, 4>(key, k, lane); break;
        case 8: bitonic_regs<KPL, 8>(key, k, lane); break;
        default: bitonic_regs<KPL, 16>(key, k, lane); break;
      }
    } else {
      const bool lower = (lane & j) == 0;
#pragma unroll
      for (int t = 0; t < KPL; ++t) {
        const int i = t * 32 + lane;
        const bool desc = (i & k) == 0;
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, key[t], j);
        const unsigned long long x = key[t];
        // the lower index keeps the larger key in a descending run
        const bool take_max = (lower == desc);
        key[t] = take_max ? (x > y ? x : y) : (x < y ? x : y);
      }
    }
  };
  if constexpr (KPL <= 8) {
#pragma unroll
    for (int k = 2; k <= N; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) stage(k, j);
  } else {
#pragma unroll 1
    for (int k = 2; k <= N; k <<= 1)
#pragma unroll 1
      for (int j = k >> 1; j > 0; j >>= 1) stage(k, j);
  }

  // ---- exclusive scan of the sorted masses; keep while below the target ----
  const int nforced = diag == 0 ? 1 : 2;
  const int ncand = ncausal - nforced;
  // A of the diagonal block, recomputed by every lane the way its owner did
  // (selecting it from the owner's registers would need a runtime index)
  float a_diag = 0.f;
  {
    const float4* q = reinterpret_cast<const float4*>(base + (long long)diag * R);
#pragma unroll
    for (int c = 0; c < RB / 4; ++c) {
      const float4 w = __ldg(q + c);
      a_diag += __expf(w.x - rlse[4 * c + 0]) + __expf(w.y - rlse[4 * c + 1]) +
                __expf(w.z - rlse[4 * c + 2]) + __expf(w.w - rlse[4 * c + 3]);
    }
  }
  const float forced_mass = __shfl_sync(0xffffffffu, a[0], 0) + (diag != 0 ? a_diag : 0.f);
  const float target = threshold * total;
  for (int kb = lane; kb < N; kb += 32) sel[kb] = 0;
  __syncwarp();
  float carry = 0.f;  // mass of the sorted positions before register t
#pragma unroll
  for (int t = 0; t < KPL; ++t) {
    const int i = t * 32 + lane;
    const float v = i < ncand ? __uint_as_float((unsigned)(key[t] >> 32)) : 0.f;
    float incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const float excl = carry + incl - v;
    if (i < ncand && forced_mass + excl < target)
      sel[0xFFFFFFFFu - (unsigned)(key[t] & 0xFFFFFFFFull)] = 1;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
  for (int kb = lane; kb < nkb; kb += 32) {
    uint8_t m = sel[kb];
    if (kb == 0 || kb == diag) m = 1;
    mrow[kb] = kb < ncausal ? m : 0;
  }
}

template <int RB>
cudaError_t launch_rb(const Problem& p, float threshold, const float* lse_part,
                      uint8_t* mask, float* block_sums, cudaStream_t st) {
  const int R = p.q_len / (kBlock / RB);
  const int rows = p.B * p.Hq * p.nqb;
  if (p.nkb <= 1024) {
    dim3 grid((rows / p.B + kWarpsPerCta - 1) / kWarpsPerCta, p.B);
    if (p.nkb <= 256)
      select_warp_kernel<RB, 8><<<grid, 32 * kWarpsPerCta, 0, st>>>(
          lse_part, p.Hq, p.nqb, p.nkb, R, p.q_start_pos / kBlock, threshold, mask, block_sums);
    else
      select_warp_kernel<RB, 32><<<grid, 32 * kWarpsPerCta, 0, st>>>(
          lse_part, p.Hq, p.nqb, p.nkb, R, p.q_start_pos / kBlock, threshold, mask, block_sums);
    return cudaGetLastError();
  }
  int n_pad = 1;
  while (n_pad < p.nkb) n_pad <<= 1;
  const size_t smem = (size_t)n_pad * 8 + (size_t)p.nkb * 4 + (size_t)p.nkb + 16;
  cudaError_t e = cudaFuncSetAttribute(select_kernel<RB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.nqb, p.Hq, p.B);
  select_kernel<RB><<<grid, kSelThreads, smem, st>>>(
      lse_part, p.Hq, p.nkb, R, p.q_start_pos / kBlock, threshold, mask,
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
