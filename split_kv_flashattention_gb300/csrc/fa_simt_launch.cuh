// Launch helper for the CUDA-core split kernel: picks the instantiation for
// (dtype, d_qk, d_v, rows per tile).  Included by one translation unit per
// input dtype so the instantiations compile in parallel.
#pragma once

#include "fa_launch.h"
#include "fa_simt.cuh"

namespace fa {

// Stage ring: about 96 KB (two CTAs per SM) but at least two stages per
// consumer warp, and a multiple of the consumer warps.
template <int DT, int DQK, int DV, int NW>
struct SimtStages {
  static constexpr int ES = Elem<DT>::size;
  static constexpr int STAGE = (((DQK * ES + 127) / 128) + ((DV * ES + 127) / 128)) * 4096;
  static constexpr int BUDGET = (96 * 1024) > 2 * NW * STAGE ? (96 * 1024) : 2 * NW * STAGE;
  static constexpr int NS_RAW = BUDGET / STAGE > 16 ? 16 : BUDGET / STAGE;
  static constexpr int NS = NS_RAW - NS_RAW % NW;
};

// Consumer warps: 4, or 2 when one 32-key stage is 32 KB (head dim 256) so
// that two stages per warp still fit.
template <int DT, int DQK, int DV>
struct SimtWarps {
  static constexpr int STAGE = SimtStages<DT, DQK, DV, 4>::STAGE;
  static constexpr int NW = STAGE >= 32 * 1024 ? 2 : 4;
};

template <int DT, int DQK, int DV, int RT, bool ORDERED>
cudaError_t launch_simt_one(const FwdParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            dim3 grid, cudaStream_t stream) {
  constexpr int NW = SimtWarps<DT, DQK, DV>::NW;
  constexpr int NS = SimtStages<DT, DQK, DV, NW>::NS;
  using C = SimtCfg<DT, DQK, DV, RT, NW, NS>;
  auto kern = simt_splitkv_kernel<DT, DQK, DV, RT, NW, NS, ORDERED>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, C::NTHREADS, C::SMEM, stream, p, tmK, tmV);
}

template <int DT, int DQK, int DV, int RTMAX, bool ORDERED>
cudaError_t launch_simt_dims(int rt, const FwdParams& p, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, dim3 grid, cudaStream_t stream) {
  if (rt == 1) return launch_simt_one<DT, DQK, DV, 1, ORDERED>(p, tmK, tmV, grid, stream);
  if (rt == 2) return launch_simt_one<DT, DQK, DV, 2, ORDERED>(p, tmK, tmV, grid, stream);
  if constexpr (RTMAX >= 4) {
    if (rt == 4) return launch_simt_one<DT, DQK, DV, 4, ORDERED>(p, tmK, tmV, grid, stream);
  }
  return cudaErrorInvalidValue;
}

// Head dims per input type; rows per tile up to 4 (2 at the widest heads).
template <int DT, bool ORDERED>
cudaError_t launch_simt_t(int d_qk, int d_v, int rt, const FwdParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, dim3 grid, cudaStream_t stream) {
  if constexpr (DT == kE4M3) {
    if (d_qk == 128 && d_v == 128)
      return launch_simt_dims<DT, 128, 128, 4, ORDERED>(rt, p, tmK, tmV, grid, stream);
    if (d_qk == 192 && d_v == 128)
      return launch_simt_dims<DT, 192, 128, 2, ORDERED>(rt, p, tmK, tmV, grid, stream);
  } else {
    if (d_qk == 64 && d_v == 64)
      return launch_simt_dims<DT, 64, 64, 4, ORDERED>(rt, p, tmK, tmV, grid, stream);
    if (d_qk == 128 && d_v == 128)
      return launch_simt_dims<DT, 128, 128, 4, ORDERED>(rt, p, tmK, tmV, grid, stream);
    if (d_qk == 256 && d_v == 256)
      return launch_simt_dims<DT, 256, 256, 2, ORDERED>(rt, p, tmK, tmV, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
