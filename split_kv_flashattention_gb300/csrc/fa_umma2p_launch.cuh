// Launch helper for the persistent two-tile tcgen05 kernel.
#pragma once

#include "fa_launch.h"
#include "fa_umma2p.cuh"

namespace fa {

template <int DT, int DQK, int DV, int KS, int VS, bool MASKED>
cudaError_t launch_umma2p_one(const FwdParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                              const CUtensorMap& tmV, dim3 grid, cudaStream_t stream) {
  using C = Umma2Cfg<DT, DQK, DV, KS, VS>;
  using CP = Umma2pCfg<DT, DQK, DV, KS, VS>;
  auto kern = umma2p_splitkv_kernel<DT, DQK, DV, KS, VS, MASKED>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), CP::SMEM);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, C::NTHREADS, CP::SMEM, stream, p, tmQ, tmK, tmV);
}

// The masked instantiation for calls with a causal or window mask.
template <int DT, int DQK, int DV, int KS, int VS>
cudaError_t launch_umma2p_mask(const FwdParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                               const CUtensorMap& tmV, dim3 grid, cudaStream_t stream) {
  if (p.causal || p.window_left >= 0)
    return launch_umma2p_one<DT, DQK, DV, KS, VS, true>(p, tmQ, tmK, tmV, grid, stream);
  return launch_umma2p_one<DT, DQK, DV, KS, VS, false>(p, tmQ, tmK, tmV, grid, stream);
}

}  // namespace fa
