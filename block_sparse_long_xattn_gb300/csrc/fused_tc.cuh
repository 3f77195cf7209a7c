// f1: one chunk step -- estimate, block selection and block-sparse attention
// over every key block -- in a single kernel launch (bf16).  The kernel and
// its launcher template; fused_tc.cu dispatches, fused_d*_e*.cu instantiate.
//
// docs/xattention_algorithm_guide.md "算法流程": the estimate (Phases 1-2),
// the selection (Phase 3, "块选择算法") and the attention ("BSA") run in
// sequence for one chunk; xattn_bsa.py compute_chunked_prefill.  The
// arithmetic of each stage is that of the stand-alone kernels
// (estimate_tc.cuh, bsa_tc.cuh; the selection as in select.cu); what this
// kernel adds is the hand-over between the stages inside one launch.
//
// Every CTA takes a ticket (an atomic counter) when it starts, and its role
// follows from the ticket, not from blockIdx:
//   tickets [0, W)   workers, W = min(#SMs, estimate tiles).  Warps 0-5 run
//                    the estimator's pipeline (producer, MMA issuer, four
//                    epilogue warps) on estimate tiles taken from a second
//                    counter; each epilogue warp counts its finished part of
//                    a tile in tiles_done[b][h][row tile].  Warps 6-9 take
//                    selection rows (b, h, qb) from a third counter, wait
//                    until every tile of the row's row tile is counted, and
//                    write the row's mask, then set row_ready[b][h][qb].
//                    Once the counter has no estimate tile left, the four
//                    epilogue warps become a second selection group (the
//                    idle stage ring is their scratch).
//   tickets [W, W+n) one attention CTA per (b, h, qb), n = B Hq nqb, in the
//                    order of the stand-alone attention kernel; it waits for
//                    its row's ready flag before its first read of the mask.
//                    As the pages' chunk step (two ranges), the CTA attends
//                    to the history (key blocks below q_start_pos/128) and
//                    to the current chunk as two ranges and merges the two
//                    results by LSE itself (bsa_tc.cuh), and the selection
//                    also writes the CPU-block keep flags of each row's
//                    history blocks.
// Every wait points at work held by a smaller ticket or at work that a
// running worker will take: a CTA with a ticket has started, a worker never
// waits on an attention CTA, and workers keep taking estimate tiles and rows
// while any are left.  So the launch cannot deadlock, whatever number of
// CTAs the GPU keeps resident.  Every wait is bounded; one that gives up
// records the device error word and sets a shared abort flag that ends the
// others' waits.
//
// The control block (counters, tiles_done, row_ready) sits in the caller's
// workspace after the estimate partials and is zeroed on the stream before
// the launch.
#pragma once

#include <algorithm>

#include "bsa_tc.cuh"
#include "estimate_tc.cuh"
#include "launchers.h"

namespace bsx {
namespace fused {

using namespace tc;

constexpr int kThreads = bsa::kThreads;  // 10 warps in either role
constexpr int kSelThreads = 128;         // a selection group: four warps
constexpr int kSelWarps = kSelThreads / 32;

// control block: [0] ticket, [1] next estimate tile, [2] next selection row,
// [3] abort, then tiles_done[B*Hq*n_rt] and row_ready[n_rows] (n_rows =
// B*Hq*nqb; all zeroed before each launch); then, 256-byte aligned,
// tile_lse[B*Hq][n_ktm][R] (every value read is written first in the same
// launch)
constexpr int kCtlHead = 4;

// worker shared memory
constexpr int kWBars = est::kRingBytes;                        // est bars, then tile-id ring
constexpr int kWMisc = kWBars + 8 * 32;                        // tmem slot, flags, tile ids
constexpr int kWSel = kWMisc + 64;                             // selection scratch
constexpr unsigned kSiteTileRing = 3;                          // kErrFused site

template <int RB, int E>
struct SelLayout {
  static constexpr int N = kSelThreads * E;  // sorted keys per row (a power of two)
  static constexpr int kKeys = 0;            // [2][N] u64
  static constexpr int kSel = kKeys + 2 * N * 8;
  static constexpr int kStat = kSel + N;     // [warps][RB] fp32
  static constexpr int kRowM = kStat + kSelWarps * RB * 4;   // [warps][RB] fp32
  static constexpr int kRowLse = kRowM + kSelWarps * RB * 4;
  static constexpr int kRed = kRowLse + RB * 4;
  static constexpr int kForced = kRed + kSelWarps * 4;
  static constexpr int kBytes = kForced + 16;
};

struct FusedParams {
  est::Tiles T;
  int B, Hq, Hkv, nqb, nkb, q_len, Lk, cur;
  int n_workers, n_rows, skip_row;
  float scale_est, scale_bsa, threshold;
  float* lse_part;
  float* tile_lse;  // [b][h][kt][i]: each row's log-sum-exp over one key tile
  int n_ktm;        // key tiles of the last row tile (the most any row tile has)
  uint8_t* mask;
  __nv_bfloat16* o;  // the result (with two ranges: merged)
  float* lse;
  bool two;          // false: one range over every key block; true: history + current chunk
  __nv_bfloat16* o_scratch;  // two ranges: the history's O on its way to the merge
  uint8_t* keep;     // CPU-block keep flags [B][n_cpu], or nullptr
  int n_cpu, cpu_kb;  // CPU blocks of the history, key blocks per CPU block
  unsigned* ctl;
  unsigned* err;
};

// One selection row on a group of 128 threads (stid = 0..127, synchronised
// by named barrier `bar`), from the estimate partials lse_part[kb][r] of the
// row's RB reshaped rows and their per-key-tile log-sum-exps tile_lse[kt][r]
// (stride R, n_kt tiles; read from L2: other CTAs of this launch wrote
// them).  The same steps as the stand-alone selection (select.cu): row
// softmax over the key blocks, block masses, a bitonic sort of (mass, ~kb)
// keys descending, an exclusive scan, and the threshold rule with blocks 0
// and diag forced.  The row's normaliser comes from the n_kt tile values
// instead of a pass over all its partials.
template <int RB, int E>
__device__ __forceinline__ void select_row(const float* __restrict__ base,
                                           const float* __restrict__ tile_lse, int n_kt, int R,
                                           int nkb, int diag, float threshold,
                                           uint8_t* __restrict__ mrow, uint8_t* sm, int stid,
                                           int bar) {
  using SL = SelLayout<RB, E>;
  constexpr int NT = kSelThreads, N = SL::N;
  unsigned long long* kbuf = reinterpret_cast<unsigned long long*>(sm + SL::kKeys);
  uint8_t* sel = sm + SL::kSel;
  float* stat = reinterpret_cast<float*>(sm + SL::kStat);
  float* row_m = reinterpret_cast<float*>(sm + SL::kRowM);  // per-warp running sums
  float* row_lse = reinterpret_cast<float*>(sm + SL::kRowLse);
  float* red = reinterpret_cast<float*>(sm + SL::kRed);
  float* forced = reinterpret_cast<float*>(sm + SL::kForced);
  const int lane = stid & 31, w = stid >> 5;
  const int ncausal = diag + 1;
  auto sel_sync = [&] { named_barrier_sync(bar, NT); };

  // ---- 1. each reshaped row's log-sum-exp over its causal keys, from the
  // estimator's per-(row, key tile) log-sum-exps: thread (ii, g) folds key
  // tiles g, g + G, ... of row ii into a running (max, sum) in one pass,
  // four loads in flight; the lanes of a warp with the same ii, then the
  // warps (through shared memory), merge their pairs ----
  constexpr int G = NT / RB;
  const int ii = stid % RB, g = stid / RB;
  const float* tl = tile_lse + ii;  // + kt * R
  float m = -INFINITY, s = 0.f;
#pragma unroll 4
  for (int kt = g; kt < n_kt; kt += G) {
    const float x = __ldcg(tl + (long long)kt * R);  // -inf: no key of the tile is causal
    if (x > m) {
      s = s * __expf(m - x) + 1.f;
      m = x;
    } else if (x != -INFINITY) {
      s += __expf(x - m);
    }
  }
  auto merge = [](float& m1, float& s1, float m2, float s2) {
    const float mm = fmaxf(m1, m2);
    if (mm == -INFINITY) return;  // both empty
    s1 = s1 * __expf(m1 - mm) + s2 * __expf(m2 - mm);
    m1 = mm;
  };
#pragma unroll
  for (int o = 16; o >= RB; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge(m, s, m2, s2);
  }
  if (lane < RB) {  // then ii == lane
    stat[w * RB + ii] = m;
    row_m[w * RB + ii] = s;
  }
  for (int kb = stid; kb < N; kb += NT) sel[kb] = 0;
  sel_sync();
  if (stid < RB) {
    float mt = stat[stid], st = row_m[stid];
#pragma unroll
    for (int v = 1; v < kSelWarps; ++v) merge(mt, st, stat[v * RB + stid], row_m[v * RB + stid]);
    row_lse[stid] = mt + __logf(st);
  }
  sel_sync();

  // ---- 2. block masses A[kb] = sum_i exp(x_i - lse_i).  The row's partials
  // are swept as consecutive 16-byte columns (coalesced, eight loads in
  // flight per thread); the Q4 columns of one key block sit in adjacent
  // lanes and combine by shuffles; the masses meet in shared memory (the
  // sort's buffer, free until the sort) ----
  constexpr int Q4 = RB / 4;
  float* mass = reinterpret_cast<float*>(kbuf);  // [N]
  {
    const int c = stid % Q4;  // this thread's column in every sweep step
    const float4 lc = make_float4(row_lse[4 * c], row_lse[4 * c + 1], row_lse[4 * c + 2],
                                  row_lse[4 * c + 3]);
    const float4* b4 = reinterpret_cast<const float4*>(base);
    const int n4 = ncausal * Q4;
    for (int f0 = 0; f0 < n4; f0 += 8 * NT) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int f = f0 + u * NT + stid;
        v[u] = f < n4 ? __ldcg(b4 + f) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int f = f0 + u * NT + stid;
        float x = (__expf(v[u].x - lc.x) + __expf(v[u].y - lc.y)) +
                  (__expf(v[u].z - lc.z) + __expf(v[u].w - lc.w));
#pragma unroll
        for (int o = 1; o < Q4; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (c == 0 && f < n4) mass[f / Q4] = x;
      }
    }
    for (int kb = ncausal + stid; kb < N; kb += NT) mass[kb] = 0.f;
  }
  sel_sync();
  float a[E];
  float part = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    a[e] = mass[e * NT + stid];
    part += a[e];
  }
  if (stid == 0) {
    forced[0] = mass[0];
    forced[1] = mass[diag];
  }
  part = warp_sum(part);
  if (lane == 0) red[w] = part;
  sel_sync();  // also: every read of mass[] is done before the sort reuses it
  float total = 0.f;
#pragma unroll
  for (int v = 0; v < kSelWarps; ++v) total += red[v];

  if (threshold >= 1.0f) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int kb = e * NT + stid;
      if (kb < nkb) mrow[kb] = sel[kb] = kb < ncausal ? 1 : 0;
    }
    return;
  }

  // ---- 3. bitonic sort of (A, kb) keys, descending (ties: lower kb first),
  // position p = stid * E + e.  The stage loops stay rolled (the kernel holds
  // this code twice, next to the estimator's and the attention's); partner
  // distances j >= E are shuffles or shared memory, those below E swaps
  // inside a thread's own keys, unrolled ----
  unsigned long long key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int kb = e * NT + stid;
    key[e] = (kb < ncausal && kb != 0 && kb != diag)
                 ? ((unsigned long long)__float_as_uint(a[e]) << 32) |
                       (unsigned long long)(0xFFFFFFFFu - (unsigned)kb)
                 : 0ull;
  }
  int buf = 0;
#pragma unroll 1
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j >= E; j >>= 1) {
      const bool lower = (stid & (j / E)) == 0;
      if (j < 32 * E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int p = stid * E + e;
          const bool desc = (p & k) == 0;
          const unsigned long long y = __shfl_xor_sync(0xffffffffu, key[e], j / E);
          const unsigned long long x = key[e];
          key[e] = (lower == desc) ? (x > y ? x : y) : (x < y ? x : y);
        }
      } else {
        unsigned long long* kb_ = kbuf + buf * N;
#pragma unroll
        for (int e = 0; e < E; ++e) kb_[stid * E + e] = key[e];
        sel_sync();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int p = stid * E + e;
          const bool desc = (p & k) == 0;
          const unsigned long long y = kb_[p ^ j];
          const unsigned long long x = key[e];
          key[e] = (lower == desc) ? (x > y ? x : y) : (x < y ? x : y);
        }
        buf ^= 1;
      }
    }
#pragma unroll
    for (int j = E / 2; j > 0; j >>= 1) {
      if (j < k) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & j) == 0) {
            const int p = stid * E + e;  // lower position of the pair
            const bool desc = (p & k) == 0;
            const unsigned long long x = key[e], y = key[e | j];
            const bool swap = desc ? (x < y) : (x > y);
            key[e] = swap ? y : x;
            key[e | j] = swap ? x : y;
          }
        }
      }
    }
  }

  // ---- 4. exclusive scan of the sorted masses; keep while below the target ----
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
  sel_sync();  // every thread is past its reads of red[]
  if (lane == 31) red[w] = incl;
  sel_sync();
  float before = incl - tsum;  // exclusive within the warp
#pragma unroll
  for (int v = 0; v < kSelWarps; ++v)
    if (v < w) before += red[v];
  const float forced_mass = forced[0] + (diag != 0 ? forced[1] : 0.f);
  const float target = threshold * total;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (key[e] != 0ull && forced_mass + (before + pre[e]) < target)
      sel[0xFFFFFFFFu - (unsigned)(key[e] & 0xFFFFFFFFull)] = 1;
  }
  sel_sync();
  // the row's mask, also left in sel[] (each thread rewrites only the
  // entries it reads) for the CPU-block flags
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int kb = e * NT + stid;
    if (kb < nkb) mrow[kb] = sel[kb] = (kb < ncausal && (kb == 0 || kb == diag || sel[kb])) ? 1 : 0;
  }
}

// A selection group (128 threads, stid 0..127, named barrier `bar`; s_row and
// s_ok two words of shared memory of its own): takes rows (b, h, qb) in
// order from the counter, each once its row tile's estimate tiles are all
// counted (four epilogue warps per tile), until none are left.
template <int RB, int E>
__device__ __forceinline__ void select_rows(const FusedParams& P, uint8_t* sm, int stid, int bar,
                                            volatile int* s_row, volatile int* s_ok) {
  const est::Tiles& T = P.T;
  unsigned* ctl = P.ctl;
  unsigned* gabort = ctl + 3;
  unsigned* tiles_done = ctl + kCtlHead;
  unsigned* row_ready = tiles_done + P.B * P.Hq * T.n_rt;
  for (;;) {
    if (stid == 0) {
      int r = (int)atomicAdd(ctl + 2, 1u);
      if (r >= P.n_rows || ld_acquire_gpu(gabort) != 0) r = -1;
      int ok = 0;
      if (r >= 0) {
        const int qb = r % P.nqb, bh = r / P.nqb;
        const int rt = qb * RB / est::kM;
        ok = wait_counter(tiles_done + bh * T.n_rt + rt, 4u * (unsigned)est::key_tiles(T, rt),
                          gabort, P.err, kErrFused, bsa::kSiteTilesDone)
                 ? 1
                 : 0;
      }
      *s_row = r;
      *s_ok = ok;
    }
    named_barrier_sync(bar, kSelThreads);
    const int r = *s_row;
    const bool ok = *s_ok != 0;
    named_barrier_sync(bar, kSelThreads);  // every thread has read s_row before it is rewritten
    if (r < 0) break;
    if (ok) {
      const int qb = r % P.nqb, bh = r / P.nqb;
      const int rt = qb * RB / est::kM;
      const float* base = P.lse_part + (long long)r * P.nkb * RB;
      const float* tl = P.tile_lse + (long long)bh * P.n_ktm * T.R + qb * RB;
      uint8_t* mrow = P.mask + ((long long)bh * P.nqb + qb) * P.nkb;
      select_row<RB, E>(base, tl, est::key_tiles(T, rt), T.R, P.nkb, P.cur + qb, P.threshold,
                        mrow, sm, stid, bar);
      // the row's mask is written; one thread makes it visible GPU-wide and
      // then marks the row ready
      named_barrier_sync(bar, kSelThreads);
      if (P.keep) {
        // the CPU-block map (xattn_bsa.py select_blocks Step 6): a history
        // CPU block is kept when any of its key blocks is selected in any
        // row; every row sets the flags of its own blocks (the same value
        // from every writer; the flags are zeroed before the launch)
        // (read from the copy of the row's mask that the selection left in
        // shared memory: a re-read of the row from global memory made the
        // workers finish 3-5 us later)
        const int b = bh / P.Hq;
        const uint8_t* srow = sm + SelLayout<RB, E>::kSel;
        for (int c = stid; c < P.n_cpu; c += kSelThreads) {
          bool any = false;
          for (int u = 0; u < P.cpu_kb; ++u) any = any || srow[c * P.cpu_kb + u] != 0;
          if (any) P.keep[(long long)b * P.n_cpu + c] = 1;
        }
      }
      if (stid == 0) {
        __threadfence();
        if (r != P.skip_row) st_release_gpu(row_ready + r, 1u);
      }
    }
  }
}

template <int S, int D, int E>
__device__ __forceinline__ void worker(const FusedParams& P, const CUtensorMap* tm_q,
                                       const CUtensorMap* tm_k, uint8_t* smem) {
  constexpr int RB = kBlock / S;
  const est::Tiles& T = P.T;
  const uint32_t sb = smem_u32(smem);
  const est::Bars B{sb + kWBars};
  const uint32_t ring0 = sb + kWBars + 8 * est::kNumBars;
  auto tid_full = [&](int s) { return ring0 + 8 * s; };        // tile id published
  auto tid_empty = [&](int s) { return ring0 + 8 * (4 + s); };  // read by MMA + 4 epilogue warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kWMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kWMisc + 4);
  volatile int* tile_ids = reinterpret_cast<volatile int*>(smem + kWMisc + 8);  // [4]
  volatile int* s_row = reinterpret_cast<volatile int*>(smem + kWMisc + 24);
  volatile int* s_ok = reinterpret_cast<volatile int*>(smem + kWMisc + 28);
  unsigned* ctl = P.ctl;
  unsigned* gabort = ctl + 3;
  unsigned* tiles_done = ctl + kCtlHead;
  unsigned* err = P.err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.Hq / P.Hkv;

  if (tid == 0) {
    B.init();
    for (int s = 0; s < 4; ++s) {
      mbar_init(tid_full(s), 1);
      mbar_init(tid_empty(s), 5);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), est::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- producer: takes estimate tiles and publishes each tile's id in a
    // four-entry ring before copying its chunks; -1 ends the sequence ----
    if (lane == 0) {
      tma_prefetch_map(tm_q);
      tma_prefetch_map(tm_k);
      int it = 0;
      unsigned t_next = atomicAdd(ctl + 1, 1u);
      for (int ti = 0;; ++ti) {
        const int slot = ti & 3;
        if (ti >= 4 && !mbar_wait(tid_empty(slot), ((ti >> 2) - 1) & 1, abort_flag, err,
                                  kErrFused, kSiteTileRing))
          break;
        const int t = (t_next < (unsigned)T.total && ld_acquire_gpu(gabort) == 0) ? (int)t_next
                                                                                    : -1;
        tile_ids[slot] = t;
        mbar_arrive(tid_full(slot));
        if (t < 0) break;
        t_next = atomicAdd(ctl + 1, 1u);  // the next tile, taken while this one loads
        if (!est::produce_tile<S, D, false>(tm_q, tm_k, sb, B, T, G, t, it, abort_flag, err))
          break;
      }
      est::drain_stages(B, it);
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    const bool leader = elect_one_sync();
    int it = 0;
    bool ok = true, seen = false;
    for (int ti = 0;; ++ti) {
      const int slot = ti & 3;
      ok = ok && mbar_wait(tid_full(slot), (ti >> 2) & 1, abort_flag, err, kErrFused,
                           kSiteTileRing);
      // lane 0's view decides for the warp, so that every lane runs the same
      // number of tiles
      const int t = __shfl_sync(0xffffffffu, ok ? tile_ids[slot] : -1, 0);
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(tid_empty(slot));
      if (t < 0) break;
      est::mma_tile<S, D, false>(sb, B, tmem, ti, it, seen, ok, leader, abort_flag, err);
    }
    est::mma_finish(B, leader);
  } else if (warp < 6) {
    // ---- epilogue: partials of each tile, then this warp's share counted ----
    for (int ti = 0;; ++ti) {
      const int slot = ti & 3;
      if (!mbar_wait_warp(tid_full(slot), (ti >> 2) & 1, abort_flag, err, kErrFused,
                          kSiteTileRing))
        break;
      const int t = tile_ids[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(tid_empty(slot));
      if (t < 0) break;
      if (!est::epilogue_tile<S, D, false>(T, P.nkb, P.scale_est, P.lse_part, tmem, B, t, ti,
                                           warp, lane, abort_flag, err, P.tile_lse, P.n_ktm))
        break;
      // the warp's partials of tile t are written; one lane makes them
      // visible GPU-wide and then counts them
      __syncwarp();
      if (lane == 0) {
        int b, h, rt, kt;
        est::tile_coords(T, t, b, h, rt, kt);
        __threadfence();
        atomicAdd(tiles_done + (b * P.Hq + h) * T.n_rt + rt, 1u);
      }
    }
    // the estimate tiles are done and the stage ring is idle: these four warps
    // become a second selection group, with the ring as scratch
    select_rows<RB, E>(P, smem, tid - 2 * 32, 2, s_row + 2, s_ok + 2);
  } else {
    select_rows<RB, E>(P, smem + kWSel, tid - 6 * 32, 1, s_row, s_ok);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, est::kTmemCols);
  }
  // a wait of this CTA that gave up ends the other CTAs' waits too
  if (tid == 0 && *abort_flag) atomicExch(gabort, 1u);
}

template <int S, int D, int E, bool kTwo>
__global__ void __launch_bounds__(kThreads, 1) fused_step_kernel(
    const __grid_constant__ CUtensorMap tm_qe, const __grid_constant__ CUtensorMap tm_ke,
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
    const FusedParams P) {
  __shared__ int s_ticket;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (threadIdx.x == 0) s_ticket = (int)atomicAdd(P.ctl, 1u);
  __syncthreads();
  const int ticket = s_ticket;
  if (ticket < P.n_workers) {
    worker<S, D, E>(P, &tm_qe, &tm_ke, smem);
    return;
  }
  // attention CTA u: batch, heads, then query tiles last-first (the order
  // of the stand-alone attention kernel), which is also the order in which
  // the workers finish the rows of the early heads
  const int u = ticket - P.n_workers;
  const int nqb = P.nqb;
  const int b = u / (nqb * P.Hq);
  const int r2 = u - b * (nqb * P.Hq);
  const int h = r2 / nqb;
  const int qb = nqb - 1 - (r2 - h * nqb);
  const int r = (b * P.Hq + h) * nqb + qb;
  unsigned* row_ready = P.ctl + kCtlHead + P.B * P.Hq * P.T.n_rt;
  const bsa::BsaArgs a{&tm_q, &tm_k, &tm_v, P.mask, P.q_len, P.Lk, P.Hq, P.Hkv,
                       nqb,   P.cur, P.scale_bsa, P.err};
  const bsa::BsaTile tile{b,     h,          qb,          0,     P.two ? P.cur : P.nkb,
                          P.nkb, P.o,        P.lse,       &tm_o, P.o_scratch,
                          false, -1,         row_ready + r, P.ctl + 3};
  bsa::bsa_cta<D, true, kTwo>(a, tile, smem);
}

template <int S, int D, int E, bool kTwo>
cudaError_t launch_sde(const Problem& p, const void* q, const void* k, const void* v,
                       float threshold, float* lse_part, unsigned* ctl, size_t ctl_bytes,
                       const FusedOut& out, unsigned* err, int skip_row, cudaStream_t st) {
  const int R = p.q_len / S, Ck = p.Lk / S;
  const bool split = out.o_curr != nullptr;
  if (split != kTwo) return cudaErrorInvalidValue;
  CUtensorMap mqe, mke, mq, mk, mv, mo;
  {  // the estimator's 5-D views (features, head, phase, reshaped row, batch)
    const uint64_t dims[5] = {(uint64_t)D, (uint64_t)p.Hq, (uint64_t)S, (uint64_t)R,
                              (uint64_t)p.B};
    const uint64_t strides[4] = {(uint64_t)D * 2, (uint64_t)p.Hq * D * 2,
                                 (uint64_t)S * p.Hq * D * 2, (uint64_t)p.q_len * p.Hq * D * 2};
    const uint32_t box[5] = {64, 1, 1, (uint32_t)est::kM, 1};
    if (!encode_tmap_bf16(&mqe, q, 5, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[5] = {(uint64_t)D, (uint64_t)p.Hkv, (uint64_t)S, (uint64_t)Ck,
                              (uint64_t)p.B};
    const uint64_t strides[4] = {(uint64_t)D * 2, (uint64_t)p.Hkv * D * 2,
                                 (uint64_t)S * p.Hkv * D * 2, (uint64_t)p.Lk * p.Hkv * D * 2};
    const uint32_t box[5] = {64, 1, 1, (uint32_t)est::kN, 1};
    if (!encode_tmap_bf16(&mke, k, 5, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {  // the attention's 4-D views (features, head, token, batch), 128-token boxes
    const uint32_t box[4] = {64, 1, 128, 1};
    const uint64_t dq[4] = {(uint64_t)D, (uint64_t)p.Hq, (uint64_t)p.q_len, (uint64_t)p.B};
    const uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)p.Hq * D * 2,
                            (uint64_t)p.q_len * p.Hq * D * 2};
    if (!encode_tmap_bf16(&mq, q, 4, dq, sq, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&mo, out.o, 4, dq, sq, box)) return cudaErrorInvalidValue;
    const uint64_t dk[4] = {(uint64_t)D, (uint64_t)p.Hkv, (uint64_t)p.Lk, (uint64_t)p.B};
    const uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)p.Hkv * D * 2,
                            (uint64_t)p.Lk * p.Hkv * D * 2};
    if (!encode_tmap_bf16(&mk, k, 4, dk, sk, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&mv, v, 4, dk, sk, box)) return cudaErrorInvalidValue;
  }
  FusedParams P;
  P.T.Hq = p.Hq;
  P.T.R = R;
  P.T.p_s = p.q_start_pos / S;
  P.T.n_rt = (R + est::kM - 1) / est::kM;
  P.T.per_bh = 0;
  for (int rt = 0; rt < P.T.n_rt; ++rt) P.T.per_bh += est::key_tiles(P.T, rt);
  P.T.total = p.B * p.Hq * P.T.per_bh;
  P.B = p.B;
  P.Hq = p.Hq;
  P.Hkv = p.Hkv;
  P.nqb = p.nqb;
  P.nkb = p.nkb;
  P.q_len = p.q_len;
  P.Lk = p.Lk;
  P.cur = p.q_start_pos / kBlock;
  P.n_rows = p.B * p.Hq * p.nqb;
  P.skip_row = skip_row;
  P.scale_est = 1.4426950408889634f / (sqrtf((float)D) * (float)S);
  P.scale_bsa = 1.4426950408889634f / sqrtf((float)D);
  P.threshold = threshold;
  P.lse_part = lse_part;
  P.mask = out.mask;
  P.o = static_cast<__nv_bfloat16*>(out.o);
  P.lse = out.lse;
  P.two = split;
  P.o_scratch = static_cast<__nv_bfloat16*>(out.o_curr);
  P.keep = out.keep;
  P.n_cpu = out.keep ? p.q_start_pos / out.cpu_block_tokens : 0;
  P.cpu_kb = out.keep ? out.cpu_block_tokens / kBlock : 1;
  P.ctl = ctl;
  P.err = err;
  P.n_ktm = est::key_tiles(P.T, P.T.n_rt - 1);
  P.tile_lse = reinterpret_cast<float*>(reinterpret_cast<char*>(ctl) +
                                        fused_ctl_words_bytes(p, S));
  if (fused_ctl_bytes(p, S) > ctl_bytes) return cudaErrorInvalidValue;

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  P.n_workers = std::max(1, std::min(sms, P.T.total));
  constexpr int kWorkerBytes = kWSel + SelLayout<kBlock / S, E>::kBytes;
  // an attention CTA keeps its copy of the mask row (at most 1024 bytes)
  // after the attention's own layout
  constexpr int kBytes = std::max(kWorkerBytes, bsa::Layout<D>::kBytes + 1024);
  const size_t smem = kBytes + 1024;
  e = cudaFuncSetAttribute(fused_step_kernel<S, D, E, kTwo>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(ctl, 0, fused_ctl_words_bytes(p, S), st);  // the counters and flags
  if (e != cudaSuccess) return e;
  if (P.n_cpu > 0) {
    e = cudaMemsetAsync(P.keep, 0, (size_t)p.B * P.n_cpu, st);
    if (e != cudaSuccess) return e;
  }
  const int grid = P.n_workers + P.n_rows;
  fused_step_kernel<S, D, E, kTwo><<<grid, kThreads, smem, st>>>(mqe, mke, mq, mk, mv, mo, P);
  return cudaGetLastError();
}

}  // namespace fused
}  // namespace bsx

// One host launcher per (d, E, ranges): the kernels of the three strides.
// Each fused_*.cu translation unit defines one, so that they compile in
// parallel.
#define BSX_FUSED_LAUNCHER(NAME, D, E, TWO)                                                  \
  cudaError_t NAME(const Problem& p, const void* q, const void* k, const void* v, int stride, \
                   float threshold, float* lse_part, unsigned* ctl, size_t ctl_bytes,         \
                   const FusedOut& out, unsigned* err, int skip_row, cudaStream_t st) {       \
    switch (stride) {                                                                         \
      case 4:                                                                                 \
        return fused::launch_sde<4, D, E, TWO>(p, q, k, v, threshold, lse_part, ctl,          \
                                               ctl_bytes, out, err, skip_row, st);            \
      case 8:                                                                                 \
        return fused::launch_sde<8, D, E, TWO>(p, q, k, v, threshold, lse_part, ctl,          \
                                               ctl_bytes, out, err, skip_row, st);            \
      case 16:                                                                                \
        return fused::launch_sde<16, D, E, TWO>(p, q, k, v, threshold, lse_part, ctl,         \
                                                ctl_bytes, out, err, skip_row, st);           \
      default:                                                                                \
        return cudaErrorInvalidValue;                                                         \
    }                                                                                         \
  }
