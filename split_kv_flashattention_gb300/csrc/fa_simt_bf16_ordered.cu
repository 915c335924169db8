// CUDA-core split kernel instantiations for bf16 inputs, tiles in longest sequence first.
#include "fa_simt_launch.cuh"

namespace fa {

FA_SIMT_INSTANCE(kBF16, true);

}  // namespace fa
