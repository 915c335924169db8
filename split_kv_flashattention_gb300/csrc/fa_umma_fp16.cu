// tcgen05 split kernel instantiations for fp16 inputs.
#include "fa_umma_launch.cuh"

namespace fa {

cudaError_t launch_umma_fp16(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                             const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                             cudaStream_t stream) {
  if (d_qk == 64 && d_v == 64) return launch_umma_one<kFP16, 64, 64, 5, 5>(p, tmQ, tmK, tmV, grid, stream);
  if (d_qk == 128 && d_v == 128) return launch_umma_one<kFP16, 128, 128, 3, 3>(p, tmQ, tmK, tmV, grid, stream);
  // head dim 256: Q 64 KB + one 64 KB K stage + one 64 KB V stage; TMEM S 2x128 + O 256
  if (d_qk == 256 && d_v == 256) return launch_umma_one<kFP16, 256, 256, 1, 1>(p, tmQ, tmK, tmV, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
