// f1 fused chunk step: the kernels for d = 128, rows of up to 1024 key blocks
// and one range over every key block.
#include "fused_tc.cuh"

namespace bsx {

BSX_FUSED_LAUNCHER(launch_fused_d128_e8, 128, 8, false)

}  // namespace bsx
