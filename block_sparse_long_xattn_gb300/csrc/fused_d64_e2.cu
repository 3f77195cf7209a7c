// f1 fused chunk step: the kernels for d = 64, rows of up to 256 key blocks
// and one range over every key block.
#include "fused_tc.cuh"

namespace bsx {

BSX_FUSED_LAUNCHER(launch_fused_d64_e2, 64, 2, false)

}  // namespace bsx
