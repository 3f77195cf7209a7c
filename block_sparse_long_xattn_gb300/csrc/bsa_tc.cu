// a5 on tcgen05 tensor cores: block-sparse causal attention with LSE (bf16),
// one or two key-block ranges of the same queries in one launch.  The method
// and the CTA's structure are described in bsa_tc.cuh.
#include "bsa_tc.cuh"
#include "launchers.h"

namespace bsx {
namespace {

using namespace tc;
using namespace bsa;

// One launch computes up to two key-block ranges of the same queries, each
// into its own O and LSE (the history and the current chunk of a chunk step).
struct BsaPart {
  int kb_begin, kb_end;
  __nv_bfloat16* o;
  float* lse;
};
struct BsaParts {
  BsaPart p0, p1;
  int B, nqb;
  // failure-path test hook: CTA drop_cta's producer stops before ring item
  // drop_item (no copy, no arrival), so its consumers' bounded waits run out
  int drop_cta, drop_item;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) bsa_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o0,
    const __grid_constant__ CUtensorMap tm_o1, const uint8_t* __restrict__ mask, int q_len,
    int Lk, int Hq, int Hkv, int cur, float scale_log2, const BsaParts parts, unsigned* err) {
  // One linear grid, decoded here so that the dispatch order is explicit:
  // part 0 before part 1, then batch, then heads, query tiles fastest.  The
  // CTAs resident together then cover a few heads of one GQA group or two,
  // whose K/V stay in L2 for the whole wave (heads fastest would stream every
  // kv-head's K/V in every wave and re-read it from DRAM).  Query tiles run
  // last-first: with causal masking the late tiles see the most key blocks.
  const int nqb = parts.nqb;
  const int per_part = parts.B * nqb * Hq;
  const int part = (int)blockIdx.x / per_part;
  const int rem = (int)blockIdx.x - part * per_part;
  const int b = rem / (nqb * Hq);
  const int r2 = rem - b * (nqb * Hq);
  const int h = r2 / nqb;
  const int qb = nqb - 1 - (r2 - h * nqb);
  const int kb_begin = part ? parts.p1.kb_begin : parts.p0.kb_begin;
  const int kb_end = part ? parts.p1.kb_end : parts.p0.kb_end;
  __nv_bfloat16* __restrict__ o = part ? parts.p1.o : parts.p0.o;
  float* __restrict__ lse = part ? parts.p1.lse : parts.p0.lse;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const BsaArgs a{&tm_q, &tm_k, &tm_v, mask, q_len, Lk, Hq, Hkv, nqb, cur, scale_log2, err};
  const BsaTile tile{b,       h,      qb,  kb_begin, kb_end,  kb_end,
                     o,       lse,    part ? &tm_o1 : &tm_o0, nullptr,
                     (int)blockIdx.x == parts.drop_cta, parts.drop_item, nullptr, nullptr};
  bsa_cta<D, false>(a, tile, smem);
}

template <int D>
cudaError_t launch_d(const Problem& p, const void* q, const void* k, const void* v,
                     const uint8_t* mask, int nparts, const BsaRange* ranges, unsigned* err,
                     BsaDrop drop, cudaStream_t st) {
  using L = Layout<D>;
  CUtensorMap mq, mk, mv;
  const uint32_t box[4] = {64, 1, 128, 1};
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.Hq, (uint64_t)p.q_len, (uint64_t)p.B};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)p.Hq * D * 2,
                                 (uint64_t)p.q_len * p.Hq * D * 2};
    if (!encode_tmap_bf16(&mq, q, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  // O of each range, the same box as Q (stores of the staged tile)
  CUtensorMap mo[2];
  for (int i = 0; i < 2; ++i) {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.Hq, (uint64_t)p.q_len, (uint64_t)p.B};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)p.Hq * D * 2,
                                 (uint64_t)p.q_len * p.Hq * D * 2};
    if (!encode_tmap_bf16(&mo[i], ranges[i < nparts ? i : 0].o, 4, dims, strides, box))
      return cudaErrorInvalidValue;
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
  BsaParts parts;
  parts.B = p.B;
  parts.nqb = p.nqb;
  parts.drop_cta = drop.cta;
  parts.drop_item = drop.item;
  parts.p0 = {ranges[0].kb_begin, ranges[0].kb_end, static_cast<__nv_bfloat16*>(ranges[0].o),
              ranges[0].lse};
  parts.p1 = nparts > 1 ? BsaPart{ranges[1].kb_begin, ranges[1].kb_end,
                                  static_cast<__nv_bfloat16*>(ranges[1].o), ranges[1].lse}
                        : parts.p0;
  const dim3 grid(p.Hq * p.nqb * p.B * nparts);
  bsa_tc_kernel<D><<<grid, kThreads, smem, st>>>(mq, mk, mv, mo[0], mo[1], mask, p.q_len, p.Lk,
                                                 p.Hq, p.Hkv,
                                                 p.q_start_pos / kBlock, scale_log2, parts, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bsa_tc(const Problem& p, const void* q, const void* k, const void* v,
                          const uint8_t* mask, int nparts, const BsaRange* ranges,
                          unsigned* err, cudaStream_t st, BsaDrop drop) {
  if (p.dtype != 1 || nparts < 1 || nparts > 2) return cudaErrorInvalidValue;
  if (p.d == 64) return launch_d<64>(p, q, k, v, mask, nparts, ranges, err, drop, st);
  if (p.d == 128) return launch_d<128>(p, q, k, v, mask, nparts, ranges, err, drop, st);
  return cudaErrorInvalidValue;
}

}  // namespace bsx
