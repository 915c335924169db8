// Launch helper for the two-tile tcgen05 split kernel.
#pragma once

#include "fa_launch.h"
#include "fa_umma2.cuh"

namespace fa {

template <int DT, int DQK, int DV, int KS, int VS>
cudaError_t launch_umma2_one(const FwdParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, dim3 grid, cudaStream_t stream) {
  using C = Umma2Cfg<DT, DQK, DV, KS, VS>;
  auto kern = umma2_splitkv_kernel<DT, DQK, DV, KS, VS>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, C::NTHREADS, C::SMEM, stream, p, tmQ, tmK, tmV);
}

}  // namespace fa
