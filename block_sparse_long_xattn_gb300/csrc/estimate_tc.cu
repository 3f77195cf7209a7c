// a1-a2 partial on tcgen05 tensor cores (bf16, or e4m3 Q and K): per-(row,
// key block) log-sum-exp of the scaled antidiagonal scores.  The method, the
// tile and the layout of the partials are described in estimate_tc.cuh.
//
// Persistent CTAs (one per SM) walk tiles (b, h, row tile, key tile) in
// order, each CTA taking every gridDim-th tile, so the CTAs resident together
// work on the key tiles of one or two heads and share them through L2.  Every
// CTA loads its own Q and key tiles with plain TMA copies.
// Warp 0: TMA producer (4-stage ring); warp 1: MMA issuer; warps 2..5:
// epilogue.  Every wait is bounded and records the device error word.
#include <algorithm>

#include "estimate_tc.cuh"
#include "launchers.h"

namespace bsx {
namespace {

using namespace tc;
using namespace est;

constexpr int kThreads = 192;
constexpr int kBarOff = kRingBytes;
constexpr int kMiscOff = kBarOff + 8 * 16;
constexpr int kSmemBytes = kMiscOff + 64;
static_assert(kNumBars <= 16, "barrier area");

template <int S, int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1) estimate_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    Tiles T, int Hkv, int nkb, float scale_log2, float* __restrict__ lse_part, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const Bars B{sb + kBarOff};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = T.Hq / Hkv;
  const int cl = (int)blockIdx.x, ncl = (int)gridDim.x;

  if (tid == 0) {
    B.init();
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
      for (int t = cl; t < T.total; t += ncl)
        if (!produce_tile<S, D, F8>(&tm_q, &tm_k, sb, B, T, G, t, it, abort_flag, err)) break;
      drain_stages(B, it);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    const bool leader = elect_one_sync();
    int it = 0, ti = 0;
    bool ok = true;
    bool seen = false;  // the current stage was already seen full
    for (int t = cl; t < T.total; t += ncl, ++ti)
      mma_tile<S, D, F8>(sb, B, tmem, ti, it, seen, ok, leader, abort_flag, err);
    mma_finish(B, leader);
  } else {
    // ------------------------------ epilogue ------------------------------
    int ti = 0;
    for (int t = cl; t < T.total; t += ncl, ++ti)
      if (!epilogue_tile<S, D, F8>(T, nkb, scale_log2, lse_part, tmem, B, t, ti, warp, lane,
                                   abort_flag, err))
        break;
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
