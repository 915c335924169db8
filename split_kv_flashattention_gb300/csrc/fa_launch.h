// Internal launch interface between the C ABI (fa_api.cu) and the kernel
// translation units.  Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

// Rows per CTA the CUDA-core kernel can hold in registers for this dtype and
// head dim (0 = unsupported).  Supported row tiles are 1, 2 and 4 up to it.
int simt_max_rows(int dtype, int d_qk, int d_v);

// Launch the CUDA-core split kernel.  grid = (row tiles, batch*h_kv, ns).
// `ordered` dispatches the tiles longest sequence first.
cudaError_t launch_simt(int dtype, int d_qk, int d_v, int rows_per_tile, bool ordered,
                        const FwdParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        dim3 grid, cudaStream_t stream);
// One instantiation per (input type, order), each in its own translation unit.
template <int DT, bool ORDERED>
cudaError_t launch_simt_t(int d_qk, int d_v, int rt, const FwdParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, dim3 grid, cudaStream_t stream);
#define FA_SIMT_INSTANCE(DT, ORD)                                                                \
  template cudaError_t launch_simt_t<DT, ORD>(int, int, int, const FwdParams&, const CUtensorMap&, \
                                              const CUtensorMap&, dim3, cudaStream_t)
#define FA_SIMT_EXTERN(DT, ORD) extern FA_SIMT_INSTANCE(DT, ORD)
FA_SIMT_EXTERN(kBF16, false);
FA_SIMT_EXTERN(kBF16, true);
FA_SIMT_EXTERN(kFP16, false);
FA_SIMT_EXTERN(kFP16, true);
FA_SIMT_EXTERN(kE4M3, false);
FA_SIMT_EXTERN(kE4M3, true);

// Launch the tcgen05 split kernel.  grid = (query tiles, batch*h_kv, ns).
cudaError_t launch_umma(int dtype, int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                        const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                        cudaStream_t stream);
cudaError_t launch_umma_bf16(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                             const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                             cudaStream_t stream);
cudaError_t launch_umma_fp16(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                             const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                             cudaStream_t stream);
cudaError_t launch_umma_e4m3(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                             const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                             cudaStream_t stream);

// Launch the two-tile (256-row) tcgen05 split kernel (16-bit inputs).
// grid = (query tile pairs, batch*h_kv, ns).
cudaError_t launch_umma2_bf16(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                              const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                              cudaStream_t stream);
cudaError_t launch_umma2_fp16(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                              const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                              cudaStream_t stream);

// Launch the persistent two-tile kernel (one split, packed K/V, at most 128
// sequences and kMaxUnits (sequence, query pair) units).  grid = (CTAs, 1, 1).
cudaError_t launch_umma2p_bf16(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                               const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                               cudaStream_t stream);
cudaError_t launch_umma2p_fp16(int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                               const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                               cudaStream_t stream);

// Launch the split combine (one warp per output row).
cudaError_t launch_combine(const FwdParams& p, cudaStream_t stream);

// Test hook kernel for split ranges.
cudaError_t launch_split_ranges(const int* cu_q, const int* cu_k, int batch, int max_seqlen_q,
                                int causal, int window_left, int ns, int tile_q, int* out,
                                cudaStream_t stream);

// Sets the dynamic shared-memory limit of a kernel (once per kernel and
// device; thread-safe).
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

// Launches a partial kernel with programmatic stream serialisation: its CTAs
// may be scheduled while the previous kernel in the stream drains, and the
// kernel waits for that kernel (griddepcontrol.wait) before its first global
// memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, int threads, int smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace fa
