// f1 fused chunk step: the kernels for d = 64 and rows of up to 256 key
// blocks (one translation unit per pair, so that they compile in parallel).
#include "fused_tc.cuh"

namespace bsx {

cudaError_t launch_fused_d64_e2(const Problem& p, const void* q, const void* k,
                                  const void* v, int stride, float threshold, float* lse_part,
                                  unsigned* ctl, size_t ctl_bytes, const FusedOut& out,
                                  unsigned* err, int skip_row, cudaStream_t st) {
  using namespace fused;
  switch (stride) {
    case 4:
      return launch_sde<4, 64, 2>(p, q, k, v, threshold, lse_part, ctl, ctl_bytes, out, err,
                                    skip_row, st);
    case 8:
      return launch_sde<8, 64, 2>(p, q, k, v, threshold, lse_part, ctl, ctl_bytes, out, err,
                                    skip_row, st);
    case 16:
      return launch_sde<16, 64, 2>(p, q, k, v, threshold, lse_part, ctl, ctl_bytes, out,
                                     err, skip_row, st);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace bsx
