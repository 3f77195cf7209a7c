// a5 on tcgen05 tensor cores: block-sparse causal attention with LSE (bf16).
//
// docs/xattention_algorithm_guide.md "BSA (Block Sparse Attention)": causal
// FlashAttention restricted to the selected 128x128 tiles of a per-head block
// mask (block size fixed at 128); xattn_bsa.py compute_chunked_prefill takes O
// and LSE from the history part and the current-chunk part and merges them.
//
// One CTA per (128-row q-tile, q-head, batch), the body below (bsa_cta) shared
// by the stand-alone attention kernel and the fused chunk-step kernel; 10
// warps with fixed roles:
//   warp 0      TMA producer: Q and the first selected K tile (both copied
//               before the block count), then the K and V tiles of every selected
//               key block, found by scanning the mask row, into a ring of
//               tile-sized slots in the order the MMAs consume them (K_0, K_1,
//               V_0, K_2, V_1, ...).  A K slot is freed as soon as its S MMA
//               completes and a V slot after its P V MMA.
//   warp 1      tcgen05 issuer (one elected lane): S(j) = Q K_j^T into TMEM
//               buffer j % 2, and O_{j%2} += P(j) V_j with P(j) read from that
//               same buffer.
//   warps 2..9  two softmax groups of four warps; group g takes the blocks
//               j = g, g + 2, ... with one query row per thread (TMEM lane =
//               row): read S, mask the diagonal block causally, P =
//               exp2(x - m) as bf16 pairs written back over the consumed S
//               columns, row sums; the running max m is raised (and O_g
//               rescaled) only on a group's first block and when a block's
//               row sum would exceed 2^32.  At the end the two partial
//               results (O_g, m_g, l_g) are merged per row; LSE goes to
//               global memory directly, O through the finished Q buffer and
//               one TMA store per 64-feature region.
// Each group's chain S(j) -> softmax -> P V(j) -> S(j + 2) interleaves with
// the other group's on the tensor pipe, and no per-block exchange between
// warps is needed.  TMEM: S/P buffers in columns 0-255, O_0 and O_1 after.
// Two ranges (the fused chunk step, a separate instantiation): the blocks of
// the history and then of the current chunk run as one sequence; at the
// boundary the groups finish the history range (its O to a scratch buffer,
// its LSE in registers) and restart their statistics, and the final
// epilogue merges the two results as bsx_merge_attn does.
// Every wait is bounded (2 s of wall time); on expiry the CTA records the wait
// in the device error word, drains its in-flight copies and MMAs, frees TMEM
// and exits.
#pragma once

#include "tc_common.cuh"

namespace bsx {
namespace bsa {

using namespace tc;

constexpr int kThreads = 320;   // producer, MMA issuer, 8 softmax warps
constexpr int kRegion = 128 * 128;  // bytes of one 128-row x 64-feature bf16 tile
// Largest row sum of one block's P accepted without raising the running max
// first (2^32: P and the fp32 sums stay far from overflow).
constexpr float kMaxBlockSum = 4294967296.0f;

enum Site : unsigned {
  kSiteKvEmpty = 1, kSiteQFull, kSiteKvFull, kSitePFull, kSiteSFull, kSiteODoneFinal,
  kSiteXchg, kSiteStage, kSiteRangeDone
};

template <int D>
struct Layout {
  static constexpr int kRegions = D / 64;
  static constexpr int kTile = kRegions * kRegion;        // Q, K or V tile bytes
  static constexpr int kSlots = D == 128 ? 5 : 8;         // K/V ring slots of kTile bytes
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + kTile;
  static constexpr int kBars = kRing + kSlots * kTile;    // mbarriers (8 B each)
  static constexpr int kNumBars = 32;
  static constexpr int kMisc = kBars + 8 * kNumBars;      // tmem slot, n, flags
  static constexpr int kXchg = kMisc + 64;  // [2 ranges][2 groups][m, l][128 rows] fp32
  static constexpr int kBytes = kXchg + 2 * 2 * 2 * 128 * 4;
  static constexpr uint32_t kTmemCols = 512;              // S/P 0, S/P 1, O_0, O_1
};

// Mask bytes.  Stand-alone, the row was written by an earlier launch and is
// read through the read-only path.  In the fused step another CTA of the
// same launch wrote it: the first read (thread 0's search for K_0, right
// after the ready flag) goes to L2, never to a possibly stale L1 line, and
// then the CTA copies the row (from L2) into shared memory and reads it there.
template <bool kFused>
__device__ __forceinline__ uint8_t mask_first(const uint8_t* p) {
  if constexpr (kFused) return __ldcg(p); else return __ldg(p);
}
template <bool kFused>
__device__ __forceinline__ uint8_t mask_scan(const uint8_t* p) {
  if constexpr (kFused) return *p; else return __ldg(p);
}

// What every CTA of a launch shares.
struct BsaArgs {
  const CUtensorMap *tm_q, *tm_k, *tm_v;
  const uint8_t* mask;
  int q_len, Lk, Hq, Hkv, nqb;
  int cur;  // q_start_pos / 128
  float scale_log2;
  unsigned* err;
};

// One CTA's tile: query block qb of head h, batch b, over key blocks
// [kb_begin, kb_end), into o / lse (the TMA store goes through tm_o).
// kb_split < kb_end (fused chunk step only): [kb_begin, kb_split) and
// [kb_split, kb_end) are two ranges (the history and the current chunk),
// each attended on its own; this CTA then merges the two results by LSE into
// o / lse exactly as bsx_merge_attn merges the results of separate launches
// (both rounded to the stored precision first).  The first range's O goes
// through o_scratch (same layout as o) on the way.  kb_split == kb_end: one
// range.
// `ready` (fused step only): the row's mask is complete once *ready != 0;
// `ready_wait` waits for that, bounded, and gives up early once *gabort is
// set.
struct BsaTile {
  int b, h, qb, kb_begin, kb_split, kb_end;
  __nv_bfloat16* o;
  float* lse;
  const CUtensorMap* tm_o;
  __nv_bfloat16* o_scratch;
  bool drop_here;
  int drop_item;
  const unsigned* ready;
  unsigned* gabort;
  __device__ __forceinline__ bool ready_wait(unsigned* err) const;
};

constexpr unsigned kSiteRowReady = 1;   // kErrFused sites (3: the workers' tile-id ring)
constexpr unsigned kSiteTilesDone = 2;

__device__ __forceinline__ bool BsaTile::ready_wait(unsigned* err) const {
  return wait_counter(ready, 1u, gabort, err, kErrFused, kSiteRowReady);
}

// ---- the end of a range: the two softmax groups' partial results merged ----
// Each group g holds (m_g, l_g) per row in the exchange area xr ([group][m,
// l][row]) and its O_g in TMEM; h_g: whether the group held a block of the
// range.  Symmetric in the two groups (every product and sum rounded on its
// own), so the result does not depend on which group held which of the
// range's blocks: a range that starts at an odd block of the row gives its
// blocks to the groups the other way round from a launch of that range
// alone, with the same result.
struct RangeWeights {
  float f0, f1, lse;  // O = f0 O_0 + f1 O_1; the range's LSE (natural log)
};
__device__ __forceinline__ RangeWeights range_weights(const float* xr, int row, bool h0,
                                                      bool h1) {
  const float m0 = xr[0 * 128 + row], l0 = xr[1 * 128 + row];
  const float m1 = xr[2 * 128 + row], l1 = xr[3 * 128 + row];
  // a group without a block of the range takes no part, not even in m
  const float m = h0 && h1 ? fmaxf(m0, m1) : (h0 ? m0 : m1);
  const float w0 = h0 ? fast_exp2(m0 - m) : 0.f;
  const float w1 = h1 ? fast_exp2(m1 - m) : 0.f;
  const float l = __fadd_rn(__fmul_rn(l0, w0), __fmul_rn(l1, w1));
  const bool any = h0 || h1;
  const float inv = any ? 1.f / l : 0.f;
  // an empty range: O = 0, LSE = -inf.  The LSE is rounded as it is stored
  // (explicit rounding: where the merge uses it at once, no later operation
  // may fuse with its product).
  return {__fmul_rn(w0, inv), __fmul_rn(w1, inv),
          any ? __fmul_rn(__fadd_rn(m, __log2f(l)), 0.69314718055994531f) : -INFINITY};
}

// 32 columns of the range's O for this thread's row (O_0 at taddr, O_1 D
// columns after it) as bf16, 8 per 16-byte vector.  h0 / h1 are uniform
// over the CTA, so the warp-collective TMEM loads stay convergent.
template <int D>
__device__ __forceinline__ void range_out32(uint32_t taddr, bool h0, bool h1,
                                            const RangeWeights& rw, uint4* pk4) {
  float t0[32];
  if (h0 && h1) {
    float t1[32];
    tmem_ld32(taddr, t0);
    tmem_ld32(taddr + D, t1);
#pragma unroll
    for (int e = 0; e < 32; ++e)
      t0[e] = __fadd_rn(__fmul_rn(t0[e], rw.f0), __fmul_rn(t1[e], rw.f1));
  } else if (h0 || h1) {
    tmem_ld32(taddr + (h1 ? D : 0), t0);
    const float f = h1 ? rw.f1 : rw.f0;
#pragma unroll
    for (int e = 0; e < 32; ++e) t0[e] = __fmul_rn(t0[e], f);
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) t0[e] = 0.f;
  }
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i0 = q4 * 8 + 2 * e;
      __nv_bfloat162 v2 = __floats2bfloat162_rn(t0[i0], t0[i0 + 1]);
      w4[e] = *reinterpret_cast<uint32_t*>(&v2);
    }
    pk4[q4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
}

// The end of the first of two ranges (blocks [0, n0) of the row), for one
// softmax warp: exchange (m, l) with the other group, write the range's O
// as bf16 to this row's o_scratch columns (read back by the same thread for
// the merge), and mark the first range's O_0 and O_1 read (range_done), so
// that the second range's first P V may overwrite them.  Out of line: it
// runs once per CTA, between the two ranges' loops.
struct FirstRange {
  int grp, row;
  uint32_t lane_base, tmem_o0;
  int n0;
  float m_run, l_run;
  float* xm;
  uint32_t o_done, xbar, range_done;
  volatile int* abort_flag;
  unsigned* err;
  __nv_bfloat16* scratch_row;  // o_scratch at this row
};
struct FirstResult {
  float lse;
  bool ok;
};
template <int D>
__device__ __noinline__ FirstResult finish_first_range(const FirstRange f, bool ok) {
  const bool h0 = f.n0 >= 1, h1 = f.n0 >= 2;  // group g holds blocks j = g (mod 2)
  const bool mine = f.grp ? h1 : h0;
  const int j_last = !mine ? -1 : (((f.n0 - 1) & 1) == f.grp ? f.n0 - 1 : f.n0 - 2);
  f.xm[(f.grp * 2 + 0) * 128 + f.row] = f.m_run;
  f.xm[(f.grp * 2 + 1) * 128 + f.row] = f.l_run;
  if (ok && j_last >= 0 &&
      !mbar_wait_warp(f.o_done, (j_last >> 1) & 1, f.abort_flag, f.err, kErrBsaTc,
                      kSiteODoneFinal))
    ok = false;
  mbar_arrive(f.xbar);
  if (!mbar_wait_warp(f.xbar, 0, f.abort_flag, f.err, kErrBsaTc, kSiteXchg)) ok = false;
  float lse = -INFINITY;
  if (ok) {
    tc_fence_after();
    const RangeWeights rw = range_weights(f.xm, f.row, h0, h1);
    lse = rw.lse;
#pragma unroll
    for (int cc = 0; cc < D / 64; ++cc) {
      const int col = f.grp * (D / 2) + cc * 32;
      uint4 pk4[4];
      range_out32<D>(f.tmem_o0 + f.lane_base + col, h0, h1, rw, pk4);
      uint4* dst = reinterpret_cast<uint4*>(f.scratch_row + col);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) dst[q4] = pk4[q4];
    }
  }
  tc_fence_before();
  mbar_arrive(f.range_done);
  return {lse, ok};
}

// kTwo: the CTA may attend to two ranges and merge them (compiled apart from
// the one-range body, whose code it would otherwise slow down).
template <int D, bool kFused, bool kTwo = false>
__device__ __forceinline__ void bsa_cta(const BsaArgs& a, const BsaTile& tile, uint8_t* smem) {
  using L = Layout<D>;
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  int* n_sm = reinterpret_cast<int*>(smem + L::kMisc + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 8);
  volatile int* row_bad = reinterpret_cast<volatile int*>(smem + L::kMisc + 12);
  int* n0_sm = reinterpret_cast<int*>(smem + L::kMisc + 16);

  // barrier addresses
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0 + 0;
  auto slot_full = [&](int s) { return bar0 + 8 * (1 + s); };
  auto slot_empty = [&](int s) { return bar0 + 8 * (1 + L::kSlots + s); };
  constexpr int kB2 = 1 + 2 * L::kSlots;
  auto s_full = [&](int g) { return bar0 + 8 * (kB2 + g); };    // S(j) ready, g = j % 2
  auto p_full = [&](int g) { return bar0 + 8 * (kB2 + 2 + g); };  // P(j) written
  auto o_done = [&](int g) { return bar0 + 8 * (kB2 + 4 + g); };  // P V(j) complete
  const uint32_t mma_final = bar0 + 8 * (kB2 + 6);
  const uint32_t xbar = bar0 + 8 * (kB2 + 7);          // a range's groups exchange (m, l)
  const uint32_t stage_full = bar0 + 8 * (kB2 + 8);    // O tile staged for the store
  const uint32_t range_done = bar0 + 8 * (kB2 + 9);    // first range's O read from TMEM

  const int b = tile.b, h = tile.h, qb = tile.qb, kb_begin = tile.kb_begin, kb_end = tile.kb_end;
  const int kb_split = tile.kb_split;
  const bool two = kTwo && kb_split < kb_end;  // two ranges, merged in this CTA
  const int nqb = a.nqb, Hq = a.Hq, q_len = a.q_len;
  const float scale_log2 = a.scale_log2;
  unsigned* err = a.err;
  __nv_bfloat16* __restrict__ o = tile.o;
  float* __restrict__ lse = tile.lse;
  const int nkb = a.Lk / kBlock;
  const int hk = h / (Hq / a.Hkv);
  const int diag = a.cur + qb;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* mrow = a.mask + (((long long)b * Hq + h) * nqb + qb) * nkb;
  const int kb_last = min(kb_end, diag + 1);
  const bool drop_here = tile.drop_here;
  int kb_first = kb_last;  // producer: key block of the K tile copied before the count

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(slot_full(s), 1);
      mbar_init(slot_empty(s), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(s_full(g), 1);
      mbar_init(p_full(g), 128);
      mbar_init(o_done(g), 1);
    }
    mbar_init(xbar, 256);
    mbar_init(stage_full, 256);
    mbar_init(range_done, 256);
    mbar_init(mma_final, 1);
    *abort_flag = 0;
    *n_sm = 0;
    *n0_sm = 0;
    *row_bad = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    // Q and the first selected K tile do not depend on the block count, so
    // their copies start now and their latency overlaps the count's
    tma_prefetch_map(a.tm_q);
    tma_prefetch_map(a.tm_k);
    tma_prefetch_map(a.tm_v);
    mbar_arrive_expect_tx(q_full, L::kTile);
    for (int r = 0; r < L::kRegions; ++r)
      tma_load_4d(sb + L::kQ + r * kRegion, a.tm_q, q_full, r * 64, h, qb * 128, b);
    // (fused step) the row's mask is written by another CTA: wait for its
    // ready flag before the first read of the row
    bool row_ok = true;
    if constexpr (kFused) row_ok = tile.ready_wait(a.err);
    if (!row_ok) *row_bad = 1;
    if (row_ok && !(drop_here && tile.drop_item == 0)) {
      int kb = kb_begin;
      while (kb < kb_last && !mask_first<kFused>(mrow + kb)) ++kb;
      if (kb < kb_last) {
        mbar_arrive_expect_tx(slot_full(0), L::kTile);
        for (int r = 0; r < L::kRegions; ++r)
          tma_load_4d(sb + L::kRing + r * kRegion, a.tm_k, slot_full(0), r * 64, hk, kb * 128, b);
        kb_first = kb;
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }

  // ---- count the selected key blocks of this row ----
  const uint8_t* mrow_c = mrow;  // the row where the count and the producer read it
  if constexpr (kFused) {
    __syncthreads();  // thread 0 has seen the ready flag
    uint8_t* ms = smem + L::kBytes;
    if (!*row_bad)
      for (int kb = tid; kb < kb_last; kb += kThreads) ms[kb] = __ldcg(mrow + kb);
    __syncthreads();
    mrow_c = ms;
  }
  int cnt = 0, cnt0 = 0;  // selected blocks: all, and of the first range
  if (!kFused || !*row_bad)
    for (int kb = kb_begin + tid; kb < kb_last; kb += kThreads) {
      const int sel = mrow_c[kb] ? 1 : 0;
      cnt += sel;
      cnt0 += kb < kb_split ? sel : 0;
    }
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  cnt0 = __reduce_add_sync(0xffffffffu, cnt0);
  __syncthreads();  // n_sm initialised
  if (lane == 0 && cnt) atomicAdd(n_sm, cnt);
  if (lane == 0 && cnt0) atomicAdd(n0_sm, cnt0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n = *n_sm;
  // blocks j < n0 (in the order of the row) belong to the first range; one
  // range: n0 = n
  const int n0 = two ? *n0_sm : n;
  // the diagonal block, when selected, is the last block of the row
  const bool diag_last = diag >= kb_begin && diag < kb_end && mrow_c[diag] != 0;
  const uint32_t tmem_s0 = tmem, tmem_o0 = tmem + 256;

  if (n == 0) {
    // no visible key: O = 0, LSE = -inf
    for (int e = tid; e < 128 * D / 8; e += kThreads) {
      const int r = e / (D / 8), c = e % (D / 8);
      reinterpret_cast<uint4*>(o + (((long long)b * q_len + qb * 128 + r) * Hq + h) * D)[c] =
          make_uint4(0, 0, 0, 0);
    }
    for (int r = tid; r < 128; r += kThreads)
      lse[((long long)b * Hq + h) * q_len + qb * 128 + r] = -INFINITY;
    if (tid == 0) drain_wait(q_full, 0);  // the early Q copy lands before the CTA exits
  } else if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      // Ring items in the order the tensor pipe consumes them,
      //   K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1},
      // item i in slot i % kSlots, so that the ring is a plain FIFO.  K_0
      // was copied before the count (unless the test hook drops item 0).
      const bool k0_copied = kb_first < kb_last;
      int issued = k0_copied ? 1 : 0;
      int kb = k0_copied ? kb_first : kb_begin - 1;
      int kb_even = k0_copied ? kb_first : 0, kb_odd = 0;  // key blocks of the two most recent K items
      bool ok = true;
      for (int i = issued; ok && i < 2 * n; ++i) {
        const bool is_k = i == 0 || ((i & 1) && (i + 1) / 2 < n);
        int blk;
        if (is_k) {
          blk = (i + 1) / 2;
          do {
            ++kb;
          } while (kb < kb_last && !mask_scan<kFused>(mrow_c + kb));
          if (kb >= kb_last) break;  // cannot happen: n counts these blocks
          if (blk & 1) kb_odd = kb; else kb_even = kb;
        } else {
          blk = i == 2 * n - 1 ? n - 1 : (i - 2) / 2;
        }
        if (drop_here && i == tile.drop_item) break;
        const int s = i % L::kSlots;
        if (i >= L::kSlots &&
            !mbar_wait(slot_empty(s), ((i / L::kSlots) - 1) & 1, abort_flag, err, kErrBsaTc,
                       kSiteKvEmpty)) {
          ok = false;
          break;
        }
        const uint32_t dst = sb + L::kRing + s * L::kTile;
        mbar_arrive_expect_tx(slot_full(s), L::kTile);
        const CUtensorMap* map = is_k ? a.tm_k : a.tm_v;
        for (int r = 0; r < L::kRegions; ++r)
          tma_load_4d(dst + r * kRegion, map, slot_full(s), r * 64, hk,
                      ((blk & 1) ? kb_odd : kb_even) * 128, b);
        issued = i + 1;
      }
      // copies still in flight must land before the CTA may exit
      drain_wait(q_full, 0);
      for (int s = 0; s < L::kSlots && s < issued; ++s)
        drain_wait(slot_full(s), ((issued - 1 - s) / L::kSlots) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    // The whole warp runs the loop, so that slot addresses and descriptors are
    // warp-uniform values; one elected lane issues the tcgen05 instructions.
    // (A single-lane issuer sharing its scheduler with ALU-bound softmax warps
    // cannot keep the tensor pipe fed.)  The tensor pipe accepts only a few
    // MMAs ahead, so the work between two batches is kept small: the order is
    //   S(0), S(1), [P V(0), S(2)], [P V(1), S(3)], ..., [P V(n-1)]
    // and each bracketed pair follows one group of waits (P(j), V_j, K_{j+2}).
    // With two ranges the sequence runs on across the boundary; the first
    // P V of the second range (which overwrites O_g) also waits until the
    // softmax warps have read the first range's O_0 and O_1.
    // Every lane keeps its own wait result and runs the same number of
    // iterations and __syncwarp()s; only the issuing lane's result decides
    // whether it issues, so a timed-out wait needs no warp vote.
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
    const bool leader = elect_one_sync();
    auto wait = [&](bool ok, uint32_t bar, uint32_t parity, unsigned site) -> bool {
      return ok && mbar_wait(bar, parity, abort_flag, err, kErrBsaTc, site);
    };
    // ring position of K_m and V_j (the producer's order)
    auto kpos = [&](int m) { return m == 0 ? 0 : 2 * m - 1; };
    auto vpos = [&](int j) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; };
    // The start-address field of a shared-memory descriptor is (address >> 4)
    // in its low bits; shared addresses are below 256 KB, so adding
    // (offset >> 4) to a descriptor moves it by `offset` bytes.
    const uint64_t dq = smem_desc_sw128(sb + L::kQ, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sb + L::kRing, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sb + L::kRing, kRegion, 1024);
    // S(m) = Q K_m^T into TMEM buffer m % 2 (K_m already waited for)
    auto issue_s = [&](int m) {
      const int s = kpos(m) % L::kSlots;
      const uint64_t dk = dk0 + (uint64_t)((s * L::kTile) >> 4);
      const uint32_t d_tmem = tmem_s0 + (m & 1) * 128;
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {  // 16 features per MMA
        const uint32_t off = ((k >> 2) * kRegion + (k & 3) * 32) >> 4;
        mma_bf16(d_tmem, dq + off, dk + off, idesc_qk, k > 0 ? 1u : 0u);
      }
      mma_commit(s_full(m & 1));
      mma_commit(slot_empty(s));
    };
    bool ok = wait(true, q_full, 0, kSiteQFull);
    for (int m = 0; m < 2 && m < n; ++m) {
      ok = wait(ok, slot_full(kpos(m) % L::kSlots), (kpos(m) / L::kSlots) & 1, kSiteKvFull);
      tc_fence_after();
      if (leader && ok) issue_s(m);
      __syncwarp();
    }
    // the steps j of blocks [rs, re); a range's first block of each group
    // (j - rs < 2) starts that group's O accumulator afresh
    auto issue_range = [&](const int rs, const int re) {
      for (int j = rs; j < re; ++j) {
        const int g = j & 1;
        const int iv = vpos(j), sv = iv % L::kSlots;
        const bool next_s = j + 2 < n;
        const int ik = kpos(j + 2), sk = ik % L::kSlots;
        // the three probes are issued back to back so that their latencies
        // overlap; the bounded waits run only if one of them found its phase
        // still open
        bool ready = false;
        if (ok) {
          const bool r0 = mbar_try_wait(p_full(g), (j >> 1) & 1);
          const bool r1 = mbar_try_wait(slot_full(sv), (iv / L::kSlots) & 1);
          const bool r2 = !next_s || mbar_try_wait(slot_full(sk), (ik / L::kSlots) & 1);
          ready = r0 & r1 & r2;
        }
        if (!ready) {
          ok = wait(ok, p_full(g), (j >> 1) & 1, kSitePFull);
          ok = wait(ok, slot_full(sv), (iv / L::kSlots) & 1, kSiteKvFull);
          if (next_s) ok = wait(ok, slot_full(sk), (ik / L::kSlots) & 1, kSiteKvFull);
        }
        const int jr = j - rs;
        tc_fence_after();
        if (leader && ok) {
          // O_g += P(j) V_j with P(j) read from TMEM buffer g (it overwrote S(j))
          const uint64_t dv = dv0 + (uint64_t)((sv * L::kTile) >> 4);
          const uint32_t p_tmem = tmem_s0 + g * 128;
          const uint32_t o_tmem = tmem_o0 + g * D;
#pragma unroll
          for (int k = 0; k < 8; ++k)  // 16 keys per MMA: 8 TMEM columns of bf16 pairs
            mma_bf16_tmem_a(o_tmem, p_tmem + k * 8, dv + (uint64_t)((k * 2048) >> 4), idesc_pv,
                            (jr >= 2 || k > 0) ? 1u : 0u);
          mma_commit(o_done(g));
          mma_commit(slot_empty(sv));
          // S(j+2) overwrites buffer g after P V(j) has read it: the tensor
          // pipe runs the MMAs in issue order
          if (next_s) issue_s(j + 2);
        }
        __syncwarp();
      }
    };
    if (two) {
      issue_range(0, n0);
      // the second range's first P V overwrites O_0 / O_1: only once the
      // softmax warps have read the first range's
      if (n0 > 0 && n0 < n) ok = wait(ok, range_done, 0, kSiteRangeDone);
      issue_range(n0, n);
    } else {
      issue_range(0, n);
    }
    // every MMA issued above completes before TMEM is released
    if (leader) mma_commit(mma_final);
    __syncwarp();
    drain_wait(mma_final, 0);
  } else {
    // ------------------------------ softmax -------------------------------
    const int quad = warp & 3;           // TMEM lane quadrant this warp may access
    const int grp = (warp - 2) >> 2;     // takes blocks j = grp, grp + 2, ...
    const int row = quad * 32 + lane;    // query row within the tile
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t sbuf = tmem_s0 + lane_base + grp * 128;
    const uint32_t obuf = tmem_o0 + lane_base + grp * D;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    float* xm = reinterpret_cast<float*>(smem + L::kXchg);  // [range][group][m, l][row]
    const long long orow = (((long long)b * q_len + qb * 128 + row) * Hq + h) * D;
    const long long lrow = ((long long)b * Hq + h) * q_len + qb * 128 + row;
    // (two ranges) this row's LSE over the first range, once it is finished
    float lse_first = -INFINITY;
    // This group's blocks j = j0, j0 + 2, ... below re (j0 = grp mod 2) of the
    // range that starts at block rs: with two ranges each group's sequence
    // runs on across the boundary.  The loop is compiled once per use (a
    // finish of the first range inside a single loop slowed it down), and so
    // is the issuer's.
    auto softmax_blocks = [&](const int j0, const int re, const int rs) {
      for (int j = j0; ok && j < re; j += 2) {
        const int jr = j - rs;  // the block's index within its range
        if (!mbar_wait_warp(s_full(grp), (j >> 1) & 1, abort_flag, err, kErrBsaTc, kSiteSFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // S(j) into registers, the diagonal block masked causally (key column c
        // is visible to row r iff c <= r)
        auto load_s = [&](float* x) {
          tmem_ld128(sbuf, x);
          if (diag_last && j == n - 1) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > row) x[c] = -INFINITY;
          }
        };
        // P = exp2(x * scale - m_run) as bf16 pairs, and the row sum.  The
        // exponent argument and the sum use the packed two-wide fp32 FMA/add:
        // the softmax warps share their schedulers with the MMA issuer and the
        // producer, and the launch runs under the power cap, so every
        // instruction saved counts.
        uint32_t pk[64];
        float2 ps[2];
        float alpha = 1.f;
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        auto exps = [&](const float* x) {
          ps[0] = make_float2(0.f, 0.f);
          ps[1] = make_float2(0.f, 0.f);
          const float2 nm2 = make_float2(-m_run, -m_run);
#pragma unroll
          for (int c = 0; c < 128; c += 2) {
            const float2 t = __ffma2_rn(make_float2(x[c], x[c + 1]), sc2, nm2);
            const float2 p = make_float2(fast_exp2(t.x), fast_exp2(t.y));
            ps[(c >> 1) & 1] = __fadd2_rn(ps[(c >> 1) & 1], p);
            __nv_bfloat162 b2 = __floats2bfloat162_rn(p.x, p.y);
            pk[c >> 1] = *reinterpret_cast<uint32_t*>(&b2);
          }
        };
        // After the group's first block the running max is not raised before
        // the exponentials: the block is exponentiated against the current
        // m_run, which is correct for any m_run (O and l carry the same scale)
        // as long as no P overflows.  A row sum within kMaxBlockSum bounds
        // every P of the row; beyond it (or inf/NaN) the warp takes the slow
        // path: the row max, the new m_run, the exponentials again and O_g
        // rescaled.  That drops the max pass from almost every block.
        bool slow = jr < 2;
        if (!slow) {
          float x[128];
          load_s(x);
          exps(x);
          const float sblk = (ps[0].x + ps[0].y) + (ps[1].x + ps[1].y);
          slow = __any_sync(0xffffffffu, !(sblk <= kMaxBlockSum));
        }
        if (slow) {
          float x[128];
          load_s(x);  // S(j) is still in TMEM: P has not been written over it
          // row max in eight independent chains of three-way max
          float mx[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = x[e];
#pragma unroll
          for (int c = 8; c < 128; c += 16)
#pragma unroll
            for (int e = 0; e < 8; ++e) mx[e] = fmax3(mx[e], x[c + e], x[c + 8 + e]);
          // (explicit rounding here and in the running sum below: the kernels
          // built from this body must round alike, whatever they fuse)
          const float mt = __fmul_rn(fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                           fmaxf(mx[6], mx[7])),
                                     scale_log2);
          if (mt > m_run) {
            alpha = fast_exp2(m_run - mt);  // 0 on the group's first block
            m_run = mt;
          }
          exps(x);
          // O_g is rescaled between P V(j-2) and P V(j).  P V(j-2) is
          // complete: the tensor pipe ran it before S(j), which we have read.
          if (jr >= 2) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              float t[32];
              tmem_ld32(obuf + cc * 32, t);
#pragma unroll
              for (int e = 0; e < 32; ++e) t[e] *= alpha;
              tmem_st32(obuf + cc * 32, t);
            }
          }
        }
        l_run = __fmaf_rn(l_run, alpha, (ps[0].x + ps[0].y) + (ps[1].x + ps[1].y));
        tmem_st64(sbuf, reinterpret_cast<const float*>(pk));  // P(j) over S(j)
        tc_fence_before();
        mbar_arrive(p_full(grp));
      }
    };
    if (two) {
      softmax_blocks(grp, n0, 0);
      // This group's first block of the second range (S of it is already
      // computed) goes first, with fresh running statistics, so that its P
      // is ready when the issuer resumes; then the end of the first range
      // (with the other group), then the rest of the second range.
      const float m_first = m_run, l_first = l_run;
      m_run = -INFINITY;
      l_run = 0.f;
      const int y = n0 + ((grp - n0) & 1);
      softmax_blocks(y, y + 1 < n ? y + 1 : n, n0);
      const FirstResult fr = finish_first_range<D>(
          FirstRange{grp, row, lane_base, tmem_o0, n0, m_first, l_first, xm, o_done(grp), xbar,
                     range_done, abort_flag, err, tile.o_scratch + orow},
          ok);
      lse_first = fr.lse;
      ok = fr.ok;
      softmax_blocks(y + 2, n, n0);
    } else {
      softmax_blocks(grp, n, 0);
    }
    // ---- end of the (last) range: the two groups' results merged per row ----
    {
      const int rs = two ? n0 : 0, re = n;
      const int nr = re - rs;
      // which groups hold a block of the range (uniform over the CTA, so the
      // warp-collective TMEM loads below stay convergent)
      const bool h0 = nr >= 2 || (nr == 1 && (rs & 1) == 0);
      const bool h1 = nr >= 2 || (nr == 1 && (rs & 1) == 1);
      const bool mine = grp ? h1 : h0;
      const int j_last = !mine ? -1 : (((re - 1) & 1) == grp ? re - 1 : re - 2);
      // (two ranges) the first range's O of this thread's columns, this
      // thread's own stores to o_scratch, loaded before the waits below so
      // that their latency is hidden
      uint4 first_o[D / 64][4];
      if (two) {
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          const uint4* scr =
              reinterpret_cast<const uint4*>(tile.o_scratch + orow + grp * (D / 2) + cc * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) first_o[cc][q4] = scr[q4];
        }
      }
      float* xr = xm + (two ? 2 * 2 * 128 : 0);
      xr[(grp * 2 + 0) * 128 + row] = m_run;
      xr[(grp * 2 + 1) * 128 + row] = l_run;
      if (ok && j_last >= 0 &&
          !mbar_wait_warp(o_done(grp), (j_last >> 1) & 1, abort_flag, err, kErrBsaTc,
                          kSiteODoneFinal))
        ok = false;
      mbar_arrive(xbar);
      if (!mbar_wait_warp(xbar, two ? 1 : 0, abort_flag, err, kErrBsaTc, kSiteXchg)) ok = false;
      if (ok) {
        tc_fence_after();
        const RangeWeights rw = range_weights(xr, row, h0, h1);
        // (second of two ranges) the two ranges' results as they would be
        // stored -- bf16 O, fp32 LSE, the first range's first -- merged as
        // bsx_merge_attn merges them
        MergeWeights mw{0.f, 0.f, -INFINITY};
        if (two) mw = merge_weights(lse_first, rw.lse);
        // This group writes output columns [grp * D/2, grp * D/2 + D/2) of
        // its row into the Q buffer (every MMA is complete), in the 128-byte
        // swizzled layout of the tensor map's box: feature f of row r sits in
        // region f / 64, 16-byte chunk ((f % 64) / 8) ^ (r % 8) of the row's
        // 128 bytes.  One TMA store then writes the tile.
        uint8_t* stage = smem + L::kQ;
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          const int col = grp * (D / 2) + cc * 32;
          uint4 pk4[4];
          range_out32<D>(tmem_o0 + lane_base + col, h0, h1, rw, pk4);
          if (two) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint4 u = first_o[cc][q4];
              const uint32_t a4[4] = {u.x, u.y, u.z, u.w};
              const uint32_t c4[4] = {pk4[q4].x, pk4[q4].y, pk4[q4].z, pk4[q4].w};
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 av =
                    __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a4[e]));
                const float2 cv =
                    __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&c4[e]));
                __nv_bfloat162 v2 = __floats2bfloat162_rn(merge_element(mw, av.x, cv.x),
                                                          merge_element(mw, av.y, cv.y));
                w4[e] = *reinterpret_cast<uint32_t*>(&v2);
              }
              pk4[q4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int f = col + q4 * 8;
            *reinterpret_cast<uint4*>(stage + (f >> 6) * kRegion + row * 128 +
                                      ((((f & 63) >> 3) ^ (row & 7)) << 4)) = pk4[q4];
          }
        }
        if (grp == 0) lse[lrow] = two ? mw.lse : rw.lse;
      }
    }
    // the staged tile is visible to the async proxy once every softmax
    // thread has arrived; one thread stores it and waits until the copy has
    // read shared memory (the CTA's shared memory must outlive the read).
    fence_proxy_async_smem();
    mbar_arrive(stage_full);
    if (tid == 64 && ok &&
        mbar_wait(stage_full, 0, abort_flag, err, kErrBsaTc, kSiteStage)) {
      for (int r = 0; r < L::kRegions; ++r)
        tma_store_4d(tile.tm_o, sb + L::kQ + r * kRegion, r * 64, h, qb * 128, b);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace bsa
}  // namespace bsx
