// CUDA-core split kernel instantiations for bf16 inputs.
#include "fa_simt_launch.cuh"

namespace fa {

cudaError_t launch_simt_bf16(int d_qk, int d_v, int rt, const FwdParams& p, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, dim3 grid, cudaStream_t stream) {
  if (d_qk == 64 && d_v == 64) return launch_simt_dims<kBF16, 64, 64, 4>(rt, p, tmK, tmV, grid, stream);
  if (d_qk == 128 && d_v == 128) return launch_simt_dims<kBF16, 128, 128, 4>(rt, p, tmK, tmV, grid, stream);
  if (d_qk == 256 && d_v == 256) return launch_simt_dims<kBF16, 256, 256, 2>(rt, p, tmK, tmV, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
