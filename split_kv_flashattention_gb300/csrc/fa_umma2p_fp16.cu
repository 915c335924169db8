// Persistent two-tile tcgen05 kernel instantiations for fp16 inputs.
#include "fa_umma2p_launch.cuh"

namespace fa {

cudaError_t launch_umma2p_fp16(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                               const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                               cudaStream_t stream) {
  if (d_qk == 64 && d_v == 64) return launch_umma2p_mask<kFP16, 64, 64, 5, 4>(p, tmQ, tmK, tmV, grid, stream);
  if (d_qk == 128 && d_v == 128) return launch_umma2p_mask<kFP16, 128, 128, 2, 2>(p, tmQ, tmK, tmV, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
