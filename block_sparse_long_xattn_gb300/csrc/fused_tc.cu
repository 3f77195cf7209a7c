// f1 fused chunk step: host-side dispatch to the kernel instantiations
// (fused_d*_e*.cu, fused_two_d*_e*.cu) and the control block's size.  The kernel is described in
// fused_tc.cuh.
#include "fused_tc.cuh"

namespace bsx {

#define BSX_FUSED_DECL(NAME)                                                            \
  cudaError_t NAME(const Problem& p, const void* q, const void* k, const void* v, int stride, \
                   float threshold, float* lse_part, unsigned* ctl, size_t ctl_bytes,         \
                   const FusedOut& out, unsigned* err, int skip_row, cudaStream_t st);
BSX_FUSED_DECL(launch_fused_d64_e2)
BSX_FUSED_DECL(launch_fused_d64_e8)
BSX_FUSED_DECL(launch_fused_d128_e2)
BSX_FUSED_DECL(launch_fused_d128_e8)
BSX_FUSED_DECL(launch_fused_two_d64_e2)
BSX_FUSED_DECL(launch_fused_two_d64_e8)
BSX_FUSED_DECL(launch_fused_two_d128_e2)
BSX_FUSED_DECL(launch_fused_two_d128_e8)
#undef BSX_FUSED_DECL

size_t fused_ctl_words_bytes(const Problem& p, int stride) {
  const long long R = p.q_len / stride;
  const long long n_rt = (R + est::kM - 1) / est::kM;
  // the head, tiles_done and row_ready
  const long long words = fused::kCtlHead + (long long)p.B * p.Hq * (n_rt + (long long)p.nqb);
  return (size_t)((words * 4 + 255) / 256 * 256);
}

size_t fused_ctl_bytes(const Problem& p, int stride) {
  const long long R = p.q_len / stride;
  const long long n_ktm = (p.q_start_pos / stride + R - 1) / est::kN + 1;
  const long long tile_lse = (long long)p.B * p.Hq * n_ktm * R * 4;
  return fused_ctl_words_bytes(p, stride) + (size_t)((tile_lse + 255) / 256 * 256);
}

bool fused_step_supported(const Problem& p, int stride) {
  return p.dtype == 1 && (p.d == 64 || p.d == 128) &&
         (stride == 4 || stride == 8 || stride == 16) && p.nkb <= 8 * fused::kSelThreads;
}

cudaError_t launch_fused_step(const Problem& p, const void* q, const void* k, const void* v,
                              int stride, float threshold, float* lse_part, unsigned* ctl,
                              size_t ctl_bytes, const FusedOut& out, unsigned* err,
                              int skip_row, cudaStream_t st) {
  if (!fused_step_supported(p, stride)) return cudaErrorInvalidValue;
  const bool small = p.nkb <= 2 * fused::kSelThreads;  // rows of up to 256 key blocks
  const bool two = out.o_curr != nullptr;  // the chunk step's two ranges
  auto launch =
      two ? (p.d == 64 ? (small ? launch_fused_two_d64_e2 : launch_fused_two_d64_e8)
                       : (small ? launch_fused_two_d128_e2 : launch_fused_two_d128_e8))
          : (p.d == 64 ? (small ? launch_fused_d64_e2 : launch_fused_d64_e8)
                       : (small ? launch_fused_d128_e2 : launch_fused_d128_e8));
  return launch(p, q, k, v, stride, threshold, lse_part, ctl, ctl_bytes, out, err, skip_row, st);
}

}  // namespace bsx
