// CUDA-core split kernel instantiations for e4m3 inputs, tiles in longest sequence first.
#include "fa_simt_launch.cuh"

namespace fa {

FA_SIMT_INSTANCE(kE4M3, true);

}  // namespace fa
