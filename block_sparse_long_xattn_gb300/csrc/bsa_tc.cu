// a5 on tcgen05 tensor cores: block-sparse causal attention with LSE (bf16).
//
// docs/xattention_algorithm_guide.md "BSA (Block Sparse Attention)": causal
// FlashAttention restricted to the selected 128x128 tiles of a per-head block
// mask (block size fixed at 128); xattn_bsa.py compute_chunked_prefill takes O
// and LSE from the history part and the current-chunk part and merges them.
//
// One CTA per (128-row q-tile, q-head, batch); 10 warps with fixed roles:
//   warp 0      TMA producer: Q once, then the K and V tiles of every selected
//               key block, found by scanning the mask row, into a ring of
//               tile-sized slots (K_0, V_0, K_1, V_1, ...).  A K slot is freed
//               as soon as its S MMA completes and a V slot after its P V MMA,
//               so loads run about two blocks ahead of the MMAs.
//   warp 1      tcgen05 issuer: S = Q K^T into one of two TMEM buffers, and
//               O += P V into a TMEM accumulator.
//   warps 2..9  softmax, two threads per query row (TMEM lane = row, each
//               thread 64 of the 128 key columns): read S,
//               mask the diagonal block causally, online max with lazy
//               rescaling of O (only when the running max grows by > 8 in
//               log2 units), P = exp2(x - m) as bf16 into shared memory in the
//               128-byte-swizzled K-major layout the MMA reads, row sums, and
//               at the end O / l and LSE to global memory.
// The S MMA of block j+1 runs while the softmax of block j runs; the P V MMA
// of block j runs while the softmax of block j+1 computes exponentials.
// Every wait is bounded (2 s of wall time); on expiry the CTA records the wait
// in the device error word, drains its in-flight copies and MMAs, frees TMEM
// and exits.
#include "launchers.h"
#include "tc_common.cuh"

namespace bsx {
namespace {

using namespace tc;

constexpr int kThreads = 320;   // producer, MMA issuer, 8 softmax warps
constexpr int kRegion = 128 * 128;  // bytes of one 128-row x 64-feature bf16 tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum Site : unsigned {
  kSiteKvEmpty = 1, kSiteQFull, kSiteKvFull, kSiteSFree, kSitePFull, kSiteSFull,
  kSiteODone, kSiteODoneFinal, kSiteXchg
};

template <int D>
struct Layout {
  static constexpr int kRegions = D / 64;
  static constexpr int kTile = kRegions * kRegion;        // Q, K or V tile bytes
  static constexpr int kSlots = D == 128 ? 5 : 8;         // K/V ring slots of kTile bytes
  static constexpr int kQ = 0;
  static constexpr int kP = kQ + kTile;                   // 128 x 128 bf16, two regions
  static constexpr int kRing = kP + 2 * kRegion;
  static constexpr int kBars = kRing + kSlots * kTile;    // mbarriers (8 B each)
  static constexpr int kNumBars = 32;
  static constexpr int kMisc = kBars + 8 * kNumBars;      // tmem slot, n, flags
  static constexpr int kXchg = kMisc + 64;                // [2 halves][128 rows] fp32
  static constexpr int kBytes = kXchg + 2 * 128 * 4;
  static constexpr uint32_t kTmemCols = 512;              // S0, S1, O (128 each; O uses D)
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) bsa_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const uint8_t* __restrict__ mask, int q_len,
    int Lk, int Hq, int Hkv, int cur, int kb_begin, int kb_end, float scale_log2,
    __nv_bfloat16* __restrict__ o, float* __restrict__ lse, unsigned* err) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  int* n_sm = reinterpret_cast<int*>(smem + L::kMisc + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 8);

  // barrier addresses
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0 + 0;
  auto slot_full = [&](int s) { return bar0 + 8 * (1 + s); };
  auto slot_empty = [&](int s) { return bar0 + 8 * (1 + L::kSlots + s); };
  constexpr int kB2 = 1 + 2 * L::kSlots;
  auto s_full = [&](int s) { return bar0 + 8 * (kB2 + s); };
  auto s_free = [&](int s) { return bar0 + 8 * (kB2 + 2 + s); };
  const uint32_t p_full = bar0 + 8 * (kB2 + 4);
  const uint32_t o_done = bar0 + 8 * (kB2 + 5);
  const uint32_t mma_final = bar0 + 8 * (kB2 + 6);
  auto xbar = [&](int q) { return bar0 + 8 * (kB2 + 7 + q); };  // softmax warp pairs

  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int nqb = gridDim.x;
  const int nkb = Lk / kBlock;
  const int hk = h / (Hq / Hkv);
  const int diag = cur + qb;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(slot_full(s), 1);
      mbar_init(slot_empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full(s), 1);
      mbar_init(s_free(s), 256);
    }
    for (int q = 0; q < 4; ++q) mbar_init(xbar(q), 64);
    mbar_init(p_full, 256);
    mbar_init(o_done, 1);
    mbar_init(mma_final, 1);
    *abort_flag = 0;
    *n_sm = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }

  // ---- count the selected key blocks of this row ----
  const uint8_t* mrow = mask + (((long long)b * Hq + h) * nqb + qb) * nkb;
  const int kb_last = min(kb_end, diag + 1);
  int cnt = 0;
  for (int kb = kb_begin + tid; kb < kb_last; kb += kThreads) cnt += mrow[kb] ? 1 : 0;
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  __syncthreads();  // n_sm initialised
  if (lane == 0 && cnt) atomicAdd(n_sm, cnt);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n = *n_sm;
  // the diagonal block, when selected, is the last block of the row
  const bool diag_last = diag >= kb_begin && diag < kb_end && mrow[diag] != 0;
  const uint32_t tmem_s0 = tmem, tmem_o = tmem + 256;

  if (n == 0) {
    // no visible key: O = 0, LSE = -inf
    for (int e = tid; e < 128 * D / 8; e += kThreads) {
      const int r = e / (D / 8), c = e % (D / 8);
      reinterpret_cast<uint4*>(o + (((long long)b * q_len + qb * 128 + r) * Hq + h) * D)[c] =
          make_uint4(0, 0, 0, 0);
    }
    for (int r = tid; r < 128; r += kThreads)
      lse[((long long)b * Hq + h) * q_len + qb * 128 + r] = -INFINITY;
  } else if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      mbar_arrive_expect_tx(q_full, L::kTile);
      for (int r = 0; r < L::kRegions; ++r)
        tma_load_4d(sb + L::kQ + r * kRegion, &tm_q, q_full, r * 64, h, qb * 128, b);
      // ring items in order K_0, V_0, K_1, V_1, ...; item i in slot i % kSlots
      int issued = 0;
      int kb = kb_begin - 1;
      bool ok = true;
      for (int j = 0; ok && j < n; ++j) {
        do {
          ++kb;
        } while (kb < kb_last && !__ldg(mrow + kb));
        if (kb >= kb_last) break;  // cannot happen: n counts these blocks
        for (int kind = 0; kind < 2; ++kind) {
          const int i = 2 * j + kind;
          const int s = i % L::kSlots;
          if (i >= L::kSlots &&
              !mbar_wait(slot_empty(s), ((i / L::kSlots) - 1) & 1, abort_flag, err, kErrBsaTc,
                         kSiteKvEmpty)) {
            ok = false;
            break;
          }
          const uint32_t dst = sb + L::kRing + s * L::kTile;
          mbar_arrive_expect_tx(slot_full(s), L::kTile);
          const CUtensorMap* map = kind == 0 ? &tm_k : &tm_v;
          for (int r = 0; r < L::kRegions; ++r)
            tma_load_4d(dst + r * kRegion, map, slot_full(s), r * 64, hk, kb * 128, b);
          issued = i + 1;
        }
      }
      // copies still in flight must land before the CTA may exit
      drain_wait(q_full, 0);
      for (int s = 0; s < L::kSlots && s < issued; ++s)
        drain_wait(slot_full(s), ((issued - 1 - s) / L::kSlots) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
      bool ok = mbar_wait(q_full, 0, abort_flag, err, kErrBsaTc, kSiteQFull);
      auto issue_pv = [&](int i) -> bool {
        const int item = 2 * i + 1;  // V_i
        const int s = item % L::kSlots;
        if (!mbar_wait(p_full, i & 1, abort_flag, err, kErrBsaTc, kSitePFull)) return false;
        if (!mbar_wait(slot_full(s), (item / L::kSlots) & 1, abort_flag, err, kErrBsaTc,
                       kSiteKvFull))
          return false;
        tc_fence_after();
        const uint32_t vbase = sb + L::kRing + s * L::kTile;
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // 16 keys per MMA
          const uint64_t a = smem_desc_sw128(sb + L::kP + (k >> 2) * kRegion + (k & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(vbase + k * 2048, kRegion, 1024);
          mma_bf16(tmem_o, a, bd, idesc_pv, (i > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(slot_empty(s));
        return true;
      };
      int j = 0;
      for (; ok && j < n; ++j) {
        const int item = 2 * j;  // K_j
        const int s = item % L::kSlots;
        const int buf = j & 1;
        if (!mbar_wait(slot_full(s), (item / L::kSlots) & 1, abort_flag, err, kErrBsaTc,
                       kSiteKvFull)) {
          ok = false;
          break;
        }
        if (j >= 2 &&
            !mbar_wait(s_free(buf), ((j >> 1) - 1) & 1, abort_flag, err, kErrBsaTc, kSiteSFree)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kbase = sb + L::kRing + s * L::kTile;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {  // 16 features per MMA
          const uint32_t off = (k >> 2) * kRegion + (k & 3) * 32;
          const uint64_t a = smem_desc_sw128(sb + L::kQ + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kbase + off, 16, 1024);
          mma_bf16(tmem_s0 + buf * 128, a, bd, idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(s_full(buf));
        mma_commit(slot_empty(s));
        if (j >= 1 && !issue_pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) issue_pv(n - 1);
      // every MMA issued above completes before TMEM is released
      mma_commit(mma_final);
      drain_wait(mma_final, 0);
    }
  } else {
    // ------------------------------ softmax -------------------------------
    // 8 warps: two per TMEM lane quadrant (a warp may only touch the lanes
    // 32 * (warp % 4) .. + 31), each owning 64 of the 128 columns of S, P
    // and O for the 32 query rows of that quadrant.  The two halves of a row
    // exchange their partial maxima (and at the end their row sums) through
    // shared memory, synchronised by a 64-thread mbarrier per quadrant.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quad * 32 + lane;    // query row within the tile
    const int c0 = half * 64;            // first column this thread owns
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float* xchg = reinterpret_cast<float*>(smem + L::kXchg);
    int xphase = 0;
    auto pair_sync = [&]() -> bool {
      mbar_arrive(xbar(quad));
      const bool r = mbar_wait(xbar(quad), xphase & 1, abort_flag, err, kErrBsaTc, kSiteXchg);
      ++xphase;
      return r;
    };
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int buf = j & 1;
      if (!mbar_wait(s_full(buf), (j >> 1) & 1, abort_flag, err, kErrBsaTc, kSiteSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[64];
      tmem_ld64(tmem_s0 + lane_base + buf * 128 + c0, x);
      tc_fence_before();
      mbar_arrive(s_free(buf));
      if (diag_last && j == n - 1) {
        // diagonal block: key column c is visible to row r iff c <= r
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c0 + c > row) x[c] = -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
      const float pm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      xchg[half * 128 + row] = pm;
      if (!pair_sync()) {
        ok = false;
        break;
      }
      const float mt = fmaxf(pm, xchg[(1 - half) * 128 + row]) * scale_log2;
      if (!pair_sync()) {  // the partner has read before the next write
        ok = false;
        break;
      }
      const bool need = mt > m_run + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = fast_exp2(m_run - mt);  // 0 on the first block
        m_run = mt;
      }
      // P = exp2(x * scale - m), packed to bf16 pairs while PV(j-1) still runs
      uint32_t pk[32];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      const float neg_m = -m_run;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float p0 = fast_exp2(fmaf(x[c], scale_log2, neg_m));
        const float p1 = fast_exp2(fmaf(x[c + 1], scale_log2, neg_m));
        ps[(c >> 1) & 3] += p0 + p1;
        __nv_bfloat162 t = __floats2bfloat162_rn(p0, p1);
        pk[c >> 1] = *reinterpret_cast<uint32_t*>(&t);
      }
      l_run = l_run * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      if (j > 0) {
        // PV(j-1) must be done before O is rescaled or P is overwritten
        if (!mbar_wait(o_done, (j - 1) & 1, abort_flag, err, kErrBsaTc, kSiteODone)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {  // this half's O columns
            float t[32];
            const uint32_t oc = tmem_o + lane_base + half * (D / 2) + cc * 32;
            tmem_ld32(oc, t);
#pragma unroll
            for (int e = 0; e < 32; ++e) t[e] *= alpha;
            tmem_st32(oc, t);
          }
        }
      }
      // store this half of P: region `half` (keys c0 .. c0+63), 128-byte
      // swizzled K-major rows of 16-byte chunks
      uint8_t* prow = smem + L::kP + half * kRegion + row * 128;
#pragma unroll
      for (int chunk = 0; chunk < 8; ++chunk)
        *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * chunk], pk[4 * chunk + 1], pk[4 * chunk + 2], pk[4 * chunk + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // row sum = both halves
    float l_tot = 0.f;
    if (ok) {
      xchg[half * 128 + row] = l_run;
      ok = pair_sync();
      if (ok) l_tot = l_run + xchg[(1 - half) * 128 + row];
    }
    if (ok && mbar_wait(o_done, (n - 1) & 1, abort_flag, err, kErrBsaTc, kSiteODoneFinal)) {
      tc_fence_after();
      const float inv = 1.f / l_tot;
      __nv_bfloat16* orow = o + (((long long)b * q_len + qb * 128 + row) * Hq + h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        float t[32];
        const int col = half * (D / 2) + cc * 32;
        tmem_ld32(tmem_o + lane_base + col, t);
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 pk4;
          __nv_bfloat162 t0 = __floats2bfloat162_rn(t[e + 0] * inv, t[e + 1] * inv);
          __nv_bfloat162 t1 = __floats2bfloat162_rn(t[e + 2] * inv, t[e + 3] * inv);
          __nv_bfloat162 t2 = __floats2bfloat162_rn(t[e + 4] * inv, t[e + 5] * inv);
          __nv_bfloat162 t3 = __floats2bfloat162_rn(t[e + 6] * inv, t[e + 7] * inv);
          pk4.x = *reinterpret_cast<uint32_t*>(&t0);
          pk4.y = *reinterpret_cast<uint32_t*>(&t1);
          pk4.z = *reinterpret_cast<uint32_t*>(&t2);
          pk4.w = *reinterpret_cast<uint32_t*>(&t3);
          reinterpret_cast<uint4*>(orow + col + e)[0] = pk4;
        }
      }
      if (half == 0)
        lse[((long long)b * Hq + h) * q_len + qb * 128 + row] =
            (m_run + __log2f(l_tot)) * 0.69314718055994531f;
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

template <int D>
cudaError_t launch_d(const Problem& p, const void* q, const void* k, const void* v,
                     const uint8_t* mask, int kb_begin, int kb_end, void* o, float* lse,
                     unsigned* err, cudaStream_t st) {
  using L = Layout<D>;
  CUtensorMap mq, mk, mv;
  const uint32_t box[4] = {64, 1, 128, 1};
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.Hq, (uint64_t)p.q_len, (uint64_t)p.B};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)p.Hq * D * 2,
                                 (uint64_t)p.q_len * p.Hq * D * 2};
    if (!encode_tmap_bf16(&mq, q, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.Hkv, (uint64_t)p.Lk, (uint64_t)p.B};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)p.Hkv * D * 2,
                                 (uint64_t)p.Lk * p.Hkv * D * 2};
    if (!encode_tmap_bf16(&mk, k, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&mv, v, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const size_t smem = L::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(bsa_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  dim3 grid(p.nqb, p.Hq, p.B);
  bsa_tc_kernel<D><<<grid, kThreads, smem, st>>>(
      mq, mk, mv, mask, p.q_len, p.Lk, p.Hq, p.Hkv, p.q_start_pos / kBlock, kb_begin, kb_end,
      scale_log2, static_cast<__nv_bfloat16*>(o), lse, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bsa_tc(const Problem& p, const void* q, const void* k, const void* v,
                          const uint8_t* mask, int kb_begin, int kb_end, void* o, float* lse,
                          unsigned* err, cudaStream_t st) {
  if (p.dtype != 1) return cudaErrorInvalidValue;
  if (p.d == 64) return launch_d<64>(p, q, k, v, mask, kb_begin, kb_end, o, lse, err, st);
  if (p.d == 128) return launch_d<128>(p, q, k, v, mask, kb_begin, kb_end, o, lse, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace bsx
