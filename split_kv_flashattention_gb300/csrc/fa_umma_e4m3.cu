// tcgen05 split kernel instantiations for e4m3 inputs.
#include "fa_umma_launch.cuh"

namespace fa {

cudaError_t launch_umma_e4m3(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                             const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                             cudaStream_t stream) {
  if (d_qk == 128 && d_v == 128) return launch_umma_one<kE4M3, 128, 128, 6, 6>(p, tmQ, tmK, tmV, grid, stream);
  if (d_qk == 192 && d_v == 128) return launch_umma_one<kE4M3, 192, 128, 4, 4>(p, tmQ, tmK, tmV, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
