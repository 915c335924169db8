// CUDA-core split kernel instantiations for e4m3 inputs, tiles in grid order.
#include "fa_simt_launch.cuh"

namespace fa {

FA_SIMT_INSTANCE(kE4M3, false);

}  // namespace fa
