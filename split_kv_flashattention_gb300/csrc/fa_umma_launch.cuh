// Launch helper for the tcgen05 split kernel.  Included by one translation
// unit per input dtype so the instantiations compile in parallel.
#pragma once

#include "fa_launch.h"
#include "fa_umma.cuh"

namespace fa {

template <int DT, int DQK, int DV, int KS, int VS>
cudaError_t launch_umma_one(const FwdParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, dim3 grid, cudaStream_t stream) {
  using C = UmmaCfg<DT, DQK, DV, KS, VS>;
  auto kern = umma_splitkv_kernel<DT, DQK, DV, KS, VS>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, C::NTHREADS, C::SMEM, stream, p, tmQ, tmK, tmV);
}

}  // namespace fa
