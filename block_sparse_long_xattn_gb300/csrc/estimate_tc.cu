// a1-a2 partial on tcgen05 tensor cores (bf16, or e4m3 Q and K): per-(row,
// key block) log-sum-exp of the scaled antidiagonal scores.
//
// docs/xattention_algorithm_guide.md "Stride Reshape 详解" and "Triton Kernels
// 详解" (flat_group_gemm_fuse_reshape): the scores are Q_r K_r^T with
//   Q_r[i] = [q[i*S+S-1], q[i*S+S-2], ..., q[i*S]],  K_r[j] = [k[j*S], ..., k[j*S+S-1]],
// a GEMM with reduction length S*d.  Here the reshape is never materialised:
// the reduction runs over S*d/64 chunks (phase t, 64 features), and for each
// chunk a 5-D TMA view of Q (features, head, phase, reshaped row, batch)
// fetches the rows q[i*S + S-1-t] and one of K fetches k[j*S + t], both
// already in the 128-byte-swizzled K-major layout the MMA reads.
//
// Tile = 128 reshaped query rows x 256 reshaped keys, accumulated in TMEM
// (two accumulators, so the epilogue of one tile overlaps the MMAs of the
// next).  Epilogue, one row per thread: scale by log2(e)/(sqrt(d) S), apply
// the causal rule J <= I (global reshaped indices, the chunk starting at row
// q_start_pos/S; xattn_bsa.py select_blocks Step 0), and for every key block
// (128/S consecutive keys) at or before the row's diagonal write
//   lse_part[b][h][qb][kb][r] = ln sum_{J in kb, J <= I} exp(s[I,J] / (sqrt(d) S))
// for row I = q_start_pos/S + qb * (128/S) + r.
// The selection kernel turns these into the softmax block sums.
//
// Persistent CTAs (one per SM) walk tiles (b, h, row tile, key tile) in
// order, each CTA taking every gridDim-th tile, so the CTAs resident together
// work on the key tiles of one or two heads and share them through L2.  Every
// CTA loads its own Q and key tiles with plain TMA copies.
// Warp 0: TMA producer (4-stage ring); warp 1: MMA issuer; warps 2..5:
// epilogue.  Every wait is bounded and records the device error word.
#include <algorithm>

#include "launchers.h"
#include "tc_common.cuh"

namespace bsx {
namespace {

using namespace tc;

constexpr int kThreads = 192;
constexpr int kStages = 4;
constexpr int kM = 128;                  // reshaped query rows per tile
constexpr int kN = 256;                  // reshaped keys per tile
constexpr int kABytes = kM * 128;        // 128 rows x 64 bf16 features
constexpr int kBBytes = kN * 128;        // 256 rows x 64 bf16 features
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kMiscOff = kBarOff + 8 * 16;
constexpr int kSmemBytes = kMiscOff + 64;
constexpr uint32_t kTmemCols = 512;      // two 128 x 256 fp32 accumulators

enum Site : unsigned { kSiteEmpty = 1, kSiteFull, kSiteAccEmpty, kSiteAccFull };

// Work units are (b, h, row tile, key tile): 128 reshaped rows against 256
// reshaped keys, in that order (key tiles fastest).
struct Tiles {
  int Hq, R, p_s, n_rt, per_bh, total;
};

// Key tiles needed by row tile rt: every 256-key tile holding a key J <= the
// largest reshaped row of the tile.
__device__ __host__ __forceinline__ int key_tiles(const Tiles& T, int rt) {
  const int i_max = min(rt * kM + kM - 1, T.R - 1);
  return (T.p_s + i_max) / kN + 1;
}

__device__ __forceinline__ void tile_coords(const Tiles& T, int t, int& b, int& h, int& rt,
                                            int& kt) {
  const int bh = t / T.per_bh;
  int rem = t - bh * T.per_bh;
  b = bh / T.Hq;
  h = bh - b * T.Hq;
  rt = 0;
  while (rt < T.n_rt - 1) {
    const int n = key_tiles(T, rt);
    if (rem < n) break;
    rem -= n;
    ++rt;
  }
  kt = rem;
}

// F8: Q and K are e4m3 bytes (kind::f8f6f4 MMAs); otherwise bf16.  Either way
// a TMA row is 128 bytes: 64 bf16 or 128 e4m3 features.
template <int S, int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1) estimate_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    Tiles T, int Hkv, int nkb, float scale_log2, float* __restrict__ lse_part, unsigned* err) {
  constexpr int RB = kBlock / S;          // reshaped keys (and rows) per 128-token block
  constexpr int CW = F8 ? 128 : 64;      // features per 128-byte chunk
  constexpr int FCH = D / CW;             // chunks per token
  constexpr int NCH = S * FCH;            // reduction chunks per tile
  constexpr int GPC = 32 / RB;            // key blocks per 32-column TMEM load
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + kBarOff;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto empty = [&](int s) { return bar0 + 8 * (kStages + s); };
  auto acc_full = [&](int s) { return bar0 + 8 * (2 * kStages + s); };
  auto acc_empty = [&](int s) { return bar0 + 8 * (2 * kStages + 2 + s); };
  const uint32_t mma_final = bar0 + 8 * (2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = T.Hq / Hkv;
  const int cl = (int)blockIdx.x, ncl = (int)gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(acc_full(s), 1);
      mbar_init(acc_empty(s), 128);
    }
    mbar_init(mma_final, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      int it = 0;
      bool ok = true;
      for (int t = cl; ok && t < T.total; t += ncl) {
        int b, h, rt, kt;
        tile_coords(T, t, b, h, rt, kt);
        const int hk = h / G;
        for (int ch = 0; ch < NCH; ++ch, ++it) {
          const int s = it % kStages;
          if (it >= kStages &&
              !mbar_wait(empty(s), ((it / kStages) - 1) & 1, abort_flag, err, kErrEstimateTc,
                         kSiteEmpty)) {
            ok = false;
            break;
          }
          const int phase = ch / FCH, c0 = (ch % FCH) * CW;
          const uint32_t a_dst = sb + s * kStageBytes;
          mbar_arrive_expect_tx(full(s), kStageBytes);
          tma_load_5d(a_dst, &tm_q, full(s), c0, h, S - 1 - phase, rt * kM, b);
          tma_load_5d(a_dst + kABytes, &tm_k, full(s), c0, hk, phase, kt * kN, b);
        }
      }
      for (int s = 0; s < kStages && s < it; ++s)
        drain_wait(full(s), ((it - 1 - s) / kStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    // The whole warp runs the loop (warp-uniform slot addresses and
    // descriptors, formed by adding offsets to one base descriptor: the
    // start-address field is address >> 4 in the low bits, and shared
    // addresses are below 256 KB); one elected lane issues.  A single-lane
    // issuer sharing its scheduler with the ALU-bound epilogue warps cannot
    // keep the tensor pipe fed.  Every lane keeps its own wait result over the
    // same trip count, so a timed-out wait needs no warp vote.
    constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(kM, kN) : idesc_bf16_f32(kM, kN, 0, 0);
    const bool leader = elect_one_sync();
    const uint64_t d_base = smem_desc_sw128(sb, 16, 1024);
    int it = 0, ti = 0;
    bool ok = true;
    bool seen = false;  // the current stage was already seen full
    for (int t = cl; t < T.total; t += ncl, ++ti) {
      const int buf = ti & 1;
      if (ti >= 2)
        ok = ok && mbar_wait(acc_empty(buf), ((ti >> 1) - 1) & 1, abort_flag, err,
                             kErrEstimateTc, kSiteAccEmpty);
      tc_fence_after();
      const uint32_t acc = tmem + buf * kN;
      for (int ch = 0; ch < NCH; ++ch, ++it) {
        const int s = it % kStages;
        if (!seen)
          ok = ok && mbar_wait(full(s), (it / kStages) & 1, abort_flag, err, kErrEstimateTc,
                               kSiteFull);
        tc_fence_after();
        // Test the next stage now, without blocking: its answer is needed only
        // at the next stage, and the probe's latency then overlaps this
        // stage's MMAs instead of sitting between two batches (the tensor
        // pipe queues about one MMA ahead).  If it is not there yet the next
        // stage waits as usual.
        seen = ok && mbar_test_wait(full((it + 1) % kStages), ((it + 1) / kStages) & 1);
        if (leader && ok) {
          const uint64_t da = d_base + (uint64_t)((s * kStageBytes) >> 4);
          const uint64_t db = da + (uint64_t)(kABytes >> 4);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 32 bytes along the row per MMA
            if constexpr (F8)
              mma_f8(acc, da + 2 * k, db + 2 * k, idesc, (ch > 0 || k > 0) ? 1u : 0u);
            else
              mma_bf16(acc, da + 2 * k, db + 2 * k, idesc, (ch > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(empty(s));
        }
        __syncwarp();
      }
      if (leader && ok) mma_commit(acc_full(buf));
      __syncwarp();
    }
    if (leader) mma_commit(mma_final);
    __syncwarp();
    drain_wait(mma_final, 0);
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int ti = 0;
    for (int t = cl; t < T.total; t += ncl, ++ti) {
      const int buf = ti & 1;
      if (!mbar_wait_warp(acc_full(buf), (ti >> 1) & 1, abort_flag, err, kErrEstimateTc,
                          kSiteAccFull))
        break;
      tc_fence_after();
      int b, h, rt, kt;
      tile_coords(T, t, b, h, rt, kt);
      const int i = rt * kM + row;              // reshaped row within the chunk
      const int Ig = T.p_s + i;                 // global reshaped row
      const bool valid = i < T.R;
      // lse_part[b][h][qb][kb][r] for row i = qb * RB + r: the RB rows of a
      // query block are contiguous per key block, and a query block's rows
      // for all key blocks form one contiguous run that selection reads
      float* out = lse_part +
                   ((long long)(b * T.Hq + h) * (T.R / RB) + i / RB) * nkb * RB + (i % RB);
#pragma unroll 1
      for (int cc = 0; cc < kN / 32; ++cc) {
        float v[32];
        tmem_ld32(tmem + lane_base + buf * kN + cc * 32, v);
        const int J0 = kt * kN + cc * 32;
#pragma unroll
        for (int g = 0; g < GPC; ++g) {
          const int Jg = J0 + g * RB;
          if (valid && Jg <= Ig) {
            float m = -INFINITY;
#pragma unroll
            for (int e = 0; e < RB; ++e) {
              const float x = (Jg + e <= Ig) ? v[g * RB + e] * scale_log2 : -INFINITY;
              v[g * RB + e] = x;
              m = fmaxf(m, x);
            }
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < RB; ++e) sum += fast_exp2(v[g * RB + e] - m);
            out[Jg] = (m + __log2f(sum)) * 0.69314718055994531f;  // (Jg / RB) * RB
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty(buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int S, int D, bool F8>
cudaError_t launch_sd(const Problem& p, const void* q, const void* k, float* lse_part,
                      unsigned* err, cudaStream_t st) {
  const int R = p.q_len / S, Ck = p.Lk / S;
  constexpr uint64_t es = F8 ? 1 : 2;          // bytes per element
  constexpr uint32_t cw = F8 ? 128 : 64;       // features per 128-byte TMA row
  auto encode = F8 ? encode_tmap_u8 : encode_tmap_bf16;
  CUtensorMap mq, mk;
  {
    const uint64_t dims[5] = {(uint64_t)D, (uint64_t)p.Hq, (uint64_t)S, (uint64_t)R,
                              (uint64_t)p.B};
    const uint64_t strides[4] = {(uint64_t)D * es, (uint64_t)p.Hq * D * es,
                                 (uint64_t)S * p.Hq * D * es, (uint64_t)p.q_len * p.Hq * D * es};
    const uint32_t box[5] = {cw, 1, 1, (uint32_t)kM, 1};
    if (!encode(&mq, q, 5, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[5] = {(uint64_t)D, (uint64_t)p.Hkv, (uint64_t)S, (uint64_t)Ck,
                              (uint64_t)p.B};
    const uint64_t strides[4] = {(uint64_t)D * es, (uint64_t)p.Hkv * D * es,
                                 (uint64_t)S * p.Hkv * D * es, (uint64_t)p.Lk * p.Hkv * D * es};
    const uint32_t box[5] = {cw, 1, 1, (uint32_t)kN, 1};
    if (!encode(&mk, k, 5, dims, strides, box)) return cudaErrorInvalidValue;
  }
  Tiles T;
  T.Hq = p.Hq;
  T.R = R;
  T.p_s = p.q_start_pos / S;
  T.n_rt = (R + kM - 1) / kM;
  T.per_bh = 0;
  for (int rt = 0; rt < T.n_rt; ++rt) T.per_bh += key_tiles(T, rt);
  T.total = p.B * p.Hq * T.per_bh;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const size_t smem = kSmemBytes + 1024;
  e = cudaFuncSetAttribute(estimate_tc_kernel<S, D, F8>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / (sqrtf((float)D) * (float)S);
  // persistent: one CTA per SM (the kernel's shared memory allows no more)
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, estimate_tc_kernel<S, D, F8>,
                                                    kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int grid = std::min(sms * per_sm, T.total);
  estimate_tc_kernel<S, D, F8><<<grid, kThreads, smem, st>>>(mq, mk, T, p.Hkv, p.nkb,
                                                             scale_log2, lse_part, err);
  return cudaGetLastError();
}

template <int S>
cudaError_t launch_s(const Problem& p, const void* q, const void* k, float* lse_part,
                     unsigned* err, cudaStream_t st) {
  if (p.dtype == 2) {  // e4m3: d = 128 (one 128-byte row per token)
    if (p.d == 128) return launch_sd<S, 128, true>(p, q, k, lse_part, err, st);
    return cudaErrorInvalidValue;
  }
  if (p.d == 64) return launch_sd<S, 64, false>(p, q, k, lse_part, err, st);
  if (p.d == 128) return launch_sd<S, 128, false>(p, q, k, lse_part, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_estimate_tc(const Problem& p, const void* q, const void* k, int stride,
                               float* lse_part, unsigned* err, cudaStream_t st) {
  if (p.dtype != 1 && p.dtype != 2) return cudaErrorInvalidValue;
  switch (stride) {
    case 4: return launch_s<4>(p, q, k, lse_part, err, st);
    case 8: return launch_s<8>(p, q, k, lse_part, err, st);
    case 16: return launch_s<16>(p, q, k, lse_part, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace bsx
