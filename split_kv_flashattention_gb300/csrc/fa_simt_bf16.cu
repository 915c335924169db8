// CUDA-core split kernel instantiations for bf16 inputs, tiles in grid order.
#include "fa_simt_launch.cuh"

namespace fa {

FA_SIMT_INSTANCE(kBF16, false);

}  // namespace fa
