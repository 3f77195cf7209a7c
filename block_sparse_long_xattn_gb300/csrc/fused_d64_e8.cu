// f1 fused chunk step: the kernels for d = 64, rows of up to 1024 key blocks
// and one range over every key block.
#include "fused_tc.cuh"

namespace bsx {

BSX_FUSED_LAUNCHER(launch_fused_d64_e8, 64, 8, false)

}  // namespace bsx
