// a7: BSA-block mask -> CPU-block keep flags.
//
// nano-vllm task_plan.md "核心设计理解" sections 1 and 3: one 1024-token CPU
// block holds 8 BSA blocks and is kept if any of them is selected, OR over
// heads and q-blocks; xattn_bsa.py select_blocks Step 6 aggregates only the
// history blocks and then adds the first and last one.  One CTA per
// (b, history CPU block) ORs the Hq * nqb * (cpu_block_tokens/128) bytes.
// cpu_block_mask_kernel expands kept CPU blocks back into the BSA block mask
// of the pages' offload attention (xattn_bsa.py compute_chunked_prefill:
// history dense over the selected CPU blocks, current chunk dense causal).
#include "common.cuh"
#include "launchers.h"

namespace bsx {
namespace {

__global__ void __launch_bounds__(256) map_kernel(
    const uint8_t* __restrict__ mask, int Hq, int nqb, int nkb, int per,
    int n_cpu, int force_first_last, int words, uint8_t* __restrict__ keep) {
  const int c = blockIdx.x;
  const int b = blockIdx.y;
  const int pairs = Hq * nqb;
  const uint8_t* base = mask + (long long)b * pairs * nkb + (long long)c * per;
  unsigned long long any = 0;
  if (words) {
    // the CPU block's bytes of every (h, qb) row are 8-byte aligned words
    const int wpr = per >> 3;  // words per row
    for (int idx = threadIdx.x; idx < pairs * wpr; idx += blockDim.x) {
      const int hq = idx / wpr, w = idx - hq * wpr;
      any |= __ldg(reinterpret_cast<const unsigned long long*>(base + (long long)hq * nkb) + w);
    }
  } else {
    for (int idx = threadIdx.x; idx < pairs * per; idx += blockDim.x) {
      const int hq = idx / per, u = idx - hq * per;
      any |= base[(long long)hq * nkb + u];
    }
  }
  const int hit = __syncthreads_or(any != 0ull);
  if (threadIdx.x == 0) {
    const bool k = hit || (force_first_last && (c == 0 || c == n_cpu - 1));
    keep[(long long)b * n_cpu + c] = k ? 1 : 0;
  }
}

// Block mask of the pages' offload attention: key block kb of the history is
// visible to every head and q-block iff its CPU block is kept; the current
// chunk's blocks are visible causally (kb <= diagonal).
__global__ void __launch_bounds__(256) cpu_block_mask_kernel(
    const uint8_t* __restrict__ keep, int Hq, int nqb, int nkb, int cur, int per, int n_cpu,
    uint8_t* __restrict__ mask) {
  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int diag = cur + qb;
  uint8_t* row = mask + (((long long)b * Hq + h) * nqb + qb) * nkb;
  for (int kb = threadIdx.x; kb < nkb; kb += blockDim.x) {
    uint8_t m;
    if (kb < cur) m = keep[(long long)b * n_cpu + kb / per] ? 1 : 0;
    else m = kb <= diag ? 1 : 0;
    row[kb] = m;
  }
}

}  // namespace

cudaError_t launch_cpu_block_mask(const Problem& p, const uint8_t* keep, int cpu_block_tokens,
                                  uint8_t* mask, cudaStream_t st) {
  const int per = cpu_block_tokens / kBlock;
  const int n_cpu = p.q_start_pos / cpu_block_tokens;
  dim3 grid(p.nqb, p.Hq, p.B);
  cpu_block_mask_kernel<<<grid, 256, 0, st>>>(keep, p.Hq, p.nqb, p.nkb, p.q_start_pos / kBlock,
                                               per, n_cpu, mask);
  return cudaGetLastError();
}

cudaError_t launch_map(const Problem& p, const uint8_t* mask, int cpu_block_tokens,
                       int flags, uint8_t* keep, cudaStream_t st) {
  const int n_cpu = p.q_start_pos / cpu_block_tokens;
  if (n_cpu == 0 || p.B == 0) return cudaSuccess;
  const int per = cpu_block_tokens / kBlock;
  dim3 grid(n_cpu, p.B);
  // 8-byte loads when the mask, its rows and the CPU blocks are 8-byte aligned
  const int words = (reinterpret_cast<uintptr_t>(mask) % 8 == 0) && p.nkb % 8 == 0 && per % 8 == 0;
  map_kernel<<<grid, 256, 0, st>>>(mask, p.Hq, p.nqb, p.nkb, per, n_cpu,
                                    (flags & 1) ? 1 : 0, words, keep);
  return cudaGetLastError();
}

}  // namespace bsx
