// Host-side launchers of the kernels (one translation unit each).  The C ABI
// in abi.cu validates arguments and then calls these; they only enqueue work.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bsx {

struct Problem {
  int B, Hq, Hkv, d;
  int dtype;        // 0 = f32, 1 = bf16, 2 = e4m3 (the estimate only)
  int q_len, q_start_pos, Lk;
  int nqb, nkb;     // q_len/128, Lk/128
};

// a6: in-place LSE merge.
cudaError_t launch_merge(const Problem& p, void* o1, float* lse1, const void* o2,
                         const float* lse2, cudaStream_t st);

// a7: CPU-block keep flags.
cudaError_t launch_map(const Problem& p, const uint8_t* mask, int cpu_block_tokens,
                       int flags, uint8_t* keep, cudaStream_t st);

// Offload-mode block mask from CPU-block keep flags.
cudaError_t launch_cpu_block_mask(const Problem& p, const uint8_t* keep, int cpu_block_tokens,
                                  uint8_t* mask, cudaStream_t st);

// a1-a2 partial: per (b, h, key block, reshaped row) log-sum-exp of the scaled
// scores of that row over that block's reshaped columns (CUDA cores).
cudaError_t launch_estimate_simt(const Problem& p, const void* q, const void* k,
                                 int stride, float* lse_part, cudaStream_t st);

// a1-a2 partial, tensor-core version (bf16, tcgen05).
cudaError_t launch_estimate_tc(const Problem& p, const void* q, const void* k,
                               int stride, float* lse_part, unsigned* err,
                               cudaStream_t st);

// a2-a4: row normalisation, block sums and threshold selection.
cudaError_t launch_select(const Problem& p, int stride, float threshold,
                          const float* lse_part, uint8_t* mask, float* block_sums,
                          cudaStream_t st);

// bf16 -> e4m3 bytes (round to nearest even, saturate to +-448), n values.
cudaError_t launch_quantize_e4m3(const void* src, uint8_t* dst, long long n, cudaStream_t st);

// a5: block-sparse attention on CUDA cores (any dtype, d in {64, 128}).
cudaError_t launch_bsa_simt(const Problem& p, const void* q, const void* k,
                            const void* v, const uint8_t* mask, int kb_begin,
                            int kb_end, void* o, float* lse, cudaStream_t st);

// One key-block range of a5 and where its result goes.
struct BsaRange {
  int kb_begin, kb_end;
  void* o;
  float* lse;
};

// a5: block-sparse attention on tcgen05 tensor cores (bf16), for one or two
// key-block ranges of the same queries in a single launch (the ranges' CTAs
// run in order, range 0 first).
// Failure-path test hook of launch_bsa_tc: CTA `cta` (linear grid index) stops
// loading before ring item `item`; cta < 0 disables it.
struct BsaDrop {
  int cta = -1, item = -1;
};
cudaError_t launch_bsa_tc(const Problem& p, const void* q, const void* k,
                          const void* v, const uint8_t* mask, int nparts,
                          const BsaRange* ranges, unsigned* err, cudaStream_t st,
                          BsaDrop drop = BsaDrop());

// f1 and the chunk step as one launch (bf16, stride in {4, 8, 16}, at most
// 1024 key blocks): estimate, selection and attention over every key block
// into (o, lse); or, with o_curr, the pages' chunk step -- attention on the
// history into (o, lse) and on the current chunk into (o_curr, lse_curr),
// merged by LSE into (o, lse) -- and, with keep, the CPU-block flags of
// cpu_block_tokens-token blocks (no first/last forcing).  `ctl` is a control
// block of fused_ctl_bytes() bytes, zeroed on the stream before the launch
// (so is keep); lse_part the estimate partials (as launch_estimate_tc).
// Test hook: skip_row >= 0 never marks that selection row ready, so its
// attention CTAs' bounded waits run out.
struct FusedOut {
  uint8_t* mask;
  void* o;
  float* lse;
  void* o_curr;      // nullptr: one range
  float* lse_curr;
  uint8_t* keep;     // nullptr: no CPU-block flags
  int cpu_block_tokens;
};
bool fused_step_supported(const Problem& p, int stride);
size_t fused_ctl_words_bytes(const Problem& p, int stride);  // counters and flags
size_t fused_ctl_bytes(const Problem& p, int stride);        // + per-tile row statistics
cudaError_t launch_fused_step(const Problem& p, const void* q, const void* k, const void* v,
                              int stride, float threshold, float* lse_part, unsigned* ctl,
                              size_t ctl_bytes, const FusedOut& out, unsigned* err,
                              int skip_row, cudaStream_t st);

}  // namespace bsx
