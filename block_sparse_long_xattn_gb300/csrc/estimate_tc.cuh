// a1-a2 partial on tcgen05 tensor cores: the per-tile pieces of the
// estimator (TMA producer, MMA issuer, epilogue), shared by the stand-alone
// estimator kernel and the fused chunk-step kernel.
//
// docs/xattention_algorithm_guide.md "Stride Reshape 详解" and "Triton Kernels
// 详解" (flat_group_gemm_fuse_reshape): the scores are Q_r K_r^T with
//   Q_r[i] = [q[i*S+S-1], q[i*S+S-2], ..., q[i*S]],  K_r[j] = [k[j*S], ..., k[j*S+S-1]],
// a GEMM with reduction length S*d.  The reshape is never materialised: the
// reduction runs over S*d/64 chunks (phase t, 64 features), and for each
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
#pragma once

#include "tc_common.cuh"

namespace bsx {
namespace est {

using namespace tc;

constexpr int kStages = 4;
constexpr int kM = 128;                  // reshaped query rows per tile
constexpr int kN = 256;                  // reshaped keys per tile
constexpr int kABytes = kM * 128;        // 128 rows x 64 bf16 features
constexpr int kBBytes = kN * 128;        // 256 rows x 64 bf16 features
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kRingBytes = kStages * kStageBytes;
constexpr uint32_t kTmemCols = 512;      // two 128 x 256 fp32 accumulators
constexpr int kNumBars = 2 * kStages + 5;  // full, empty, acc_full x2, acc_empty x2, final

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

__device__ __host__ __forceinline__ void tile_coords(const Tiles& T, int t, int& b, int& h,
                                                     int& rt, int& kt) {
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

// Barrier addresses of the pipeline (kNumBars mbarriers of 8 bytes at bar0).
struct Bars {
  uint32_t bar0;
  __device__ __forceinline__ uint32_t full(int s) const { return bar0 + 8 * s; }
  __device__ __forceinline__ uint32_t empty(int s) const { return bar0 + 8 * (kStages + s); }
  __device__ __forceinline__ uint32_t acc_full(int s) const {
    return bar0 + 8 * (2 * kStages + s);
  }
  __device__ __forceinline__ uint32_t acc_empty(int s) const {
    return bar0 + 8 * (2 * kStages + 2 + s);
  }
  __device__ __forceinline__ uint32_t mma_final() const { return bar0 + 8 * (2 * kStages + 4); }
  __device__ __forceinline__ void init() const {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(acc_full(s), 1);
      mbar_init(acc_empty(s), 128);
    }
    mbar_init(mma_final(), 1);
  }
};

// Compile-time shape of one tile's reduction.  F8: Q and K are e4m3 bytes
// (kind::f8f6f4 MMAs); otherwise bf16.  Either way a TMA row is 128 bytes:
// 64 bf16 or 128 e4m3 features.
template <int S, int D, bool F8>
struct Cfg {
  static constexpr int RB = kBlock / S;   // reshaped keys (and rows) per 128-token block
  static constexpr int CW = F8 ? 128 : 64;  // features per 128-byte chunk
  static constexpr int FCH = D / CW;      // chunks per token
  static constexpr int NCH = S * FCH;     // reduction chunks per tile
  static constexpr int GPC = 32 / RB;     // key blocks per 32-column TMEM load
};

// Producer (one lane): the NCH chunk copies of tile t into the stage ring;
// `it` counts chunks over the CTA's life.  False if a wait for a free stage
// gave up.
template <int S, int D, bool F8>
__device__ __forceinline__ bool produce_tile(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                             uint32_t sb, const Bars& B, const Tiles& T, int G,
                                             int t, int& it, volatile int* abort,
                                             unsigned* err) {
  using C = Cfg<S, D, F8>;
  int b, h, rt, kt;
  tile_coords(T, t, b, h, rt, kt);
  const int hk = h / G;
  for (int ch = 0; ch < C::NCH; ++ch, ++it) {
    const int s = it % kStages;
    if (it >= kStages && !mbar_wait(B.empty(s), ((it / kStages) - 1) & 1, abort, err,
                                    kErrEstimateTc, kSiteEmpty))
      return false;
    const int phase = ch / C::FCH, c0 = (ch % C::FCH) * C::CW;
    const uint32_t a_dst = sb + s * kStageBytes;
    mbar_arrive_expect_tx(B.full(s), kStageBytes);
    tma_load_5d(a_dst, tm_q, B.full(s), c0, h, S - 1 - phase, rt * kM, b);
    tma_load_5d(a_dst + kABytes, tm_k, B.full(s), c0, hk, phase, kt * kN, b);
  }
  return true;
}

// Copies still in flight must land before the CTA may exit.
__device__ __forceinline__ void drain_stages(const Bars& B, int it) {
  for (int s = 0; s < kStages && s < it; ++s)
    drain_wait(B.full(s), ((it - 1 - s) / kStages) & 1);
}

// MMA issuer (whole warp; `leader` issues): the CTA's ti-th tile into
// accumulator ti & 1.  The whole warp runs the loop (warp-uniform slot
// addresses and descriptors, formed by adding offsets to one base
// descriptor: the start-address field is address >> 4 in the low bits, and
// shared addresses are below 256 KB).  A single-lane issuer sharing its
// scheduler with the ALU-bound epilogue warps cannot keep the tensor pipe
// fed.  Every lane keeps its own wait result over the same trip count, so a
// timed-out wait needs no warp vote.  `it` counts chunks and `seen` carries
// the probe of the next stage across tiles.
template <int S, int D, bool F8>
__device__ __forceinline__ void mma_tile(uint32_t sb, const Bars& B, uint32_t tmem, int ti,
                                         int& it, bool& seen, bool& ok, bool leader,
                                         volatile int* abort, unsigned* err) {
  using C = Cfg<S, D, F8>;
  constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(kM, kN) : idesc_bf16_f32(kM, kN, 0, 0);
  const uint64_t d_base = smem_desc_sw128(sb, 16, 1024);
  const int buf = ti & 1;
  if (ti >= 2)
    ok = ok && mbar_wait(B.acc_empty(buf), ((ti >> 1) - 1) & 1, abort, err, kErrEstimateTc,
                         kSiteAccEmpty);
  tc_fence_after();
  const uint32_t acc = tmem + buf * kN;
  for (int ch = 0; ch < C::NCH; ++ch, ++it) {
    const int s = it % kStages;
    if (!seen)
      ok = ok && mbar_wait(B.full(s), (it / kStages) & 1, abort, err, kErrEstimateTc, kSiteFull);
    tc_fence_after();
    // Test the next stage now, without blocking: its answer is needed only at
    // the next stage, and the probe's latency then overlaps this stage's MMAs
    // instead of sitting between two batches (the tensor pipe queues about
    // one MMA ahead).  If it is not there yet the next stage waits as usual.
    seen = ok && mbar_test_wait(B.full((it + 1) % kStages), ((it + 1) / kStages) & 1);
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
      mma_commit(B.empty(s));
    }
    __syncwarp();
  }
  if (leader && ok) mma_commit(B.acc_full(buf));
  __syncwarp();
}

// Every MMA issued completes before TMEM is released.
__device__ __forceinline__ void mma_finish(const Bars& B, bool leader) {
  if (leader) mma_commit(B.mma_final());
  __syncwarp();
  drain_wait(B.mma_final(), 0);
}

// Epilogue (one warp of four; warp w reads TMEM lanes 32 (w % 4) ...): the
// CTA's ti-th tile t from accumulator ti & 1 into lse_part.  With a
// non-null tile_lse it also writes, for each row I of the tile, the
// log-sum-exp over all the tile's keys J <= I (the log-sum-exp of the row's
// block partials of this tile; -inf where the tile holds no such key):
//   tile_lse[b][h][kt][i], kt < n_kt (the key tiles of the last row tile).
// False if the wait for the accumulator gave up.
template <int S, int D, bool F8>
__device__ __forceinline__ bool epilogue_tile(const Tiles& T, int nkb, float scale_log2,
                                              float* __restrict__ lse_part, uint32_t tmem,
                                              const Bars& B, int t, int ti, int warp, int lane,
                                              volatile int* abort, unsigned* err,
                                              float* __restrict__ tile_lse = nullptr,
                                              int n_kt = 0) {
  using C = Cfg<S, D, F8>;
  constexpr int RB = C::RB, GPC = C::GPC;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const int buf = ti & 1;
  if (!mbar_wait_warp(B.acc_full(buf), (ti >> 1) & 1, abort, err, kErrEstimateTc, kSiteAccFull))
    return false;
  tc_fence_after();
  int b, h, rt, kt;
  tile_coords(T, t, b, h, rt, kt);
  const int i = rt * kM + row;              // reshaped row within the chunk
  const int Ig = T.p_s + i;                 // global reshaped row
  const bool valid = i < T.R;
  // lse_part[b][h][qb][kb][r] for row i = qb * RB + r: the RB rows of a
  // query block are contiguous per key block, and a query block's rows for
  // all key blocks form one contiguous run that selection reads
  float* out = lse_part + ((long long)(b * T.Hq + h) * (T.R / RB) + i / RB) * nkb * RB + (i % RB);
  float tm = -INFINITY, ts = 0.f;  // the tile's running max and sum (log2 domain)
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
        if (tile_lse) {  // fold the block's (m, sum) into the tile's
          if (m > tm) {
            ts = ts * fast_exp2(tm - m) + sum;
            tm = m;
          } else {
            ts += sum * fast_exp2(m - tm);
          }
        }
      }
    }
  }
  if (tile_lse && valid)
    tile_lse[((long long)(b * T.Hq + h) * n_kt + kt) * T.R + i] =
        ts > 0.f ? (tm + __log2f(ts)) * 0.69314718055994531f : -INFINITY;
  tc_fence_before();
  mbar_arrive(B.acc_empty(buf));
  return true;
}

}  // namespace est
}  // namespace bsx
