// CUDA-core split kernel instantiations for fp16 inputs, tiles in grid order.
#include "fa_simt_launch.cuh"

namespace fa {

FA_SIMT_INSTANCE(kFP16, false);

}  // namespace fa
