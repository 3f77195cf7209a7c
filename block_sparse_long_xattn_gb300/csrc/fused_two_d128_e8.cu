// f1 fused chunk step: the kernels for d = 128, rows of up to 1024 key blocks
// and the chunk step's two ranges (history and current chunk, merged in each attention CTA).
#include "fused_tc.cuh"

namespace bsx {

BSX_FUSED_LAUNCHER(launch_fused_two_d128_e8, 128, 8, true)

}  // namespace bsx
