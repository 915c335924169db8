// fa_fwd_splitkv_noalloc: the split-KV forward for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain scratch memory: code that runs inside
// a framework or runtime that owns every device allocation (a custom
// allocator or memory pool the caller cannot reach from its call site), a
// plugin with no allocator handle, or a latency-critical path that must not
// call cudaMalloc because it synchronises the device.  They still own their
// inputs and outputs, but not the fp32 split workspace.  This entry point
// takes that workspace from a fixed array in device global memory that the
// library itself defines, so no call allocates anything.
//
// The array lives in this file as a static __device__ object of
// FA_NOALLOC_SCRATCH_BYTES.  In host code its name is only a host-side
// stand-in, not a device address (a kernel given it would fault or, where
// the GPU can reach host memory, silently use the wrong memory), so the
// device address is looked up with cudaGetSymbolAddress once per device, on
// the first call made with that device current, and cached.
#include <mutex>

#include "../../include/fa_splitkv.h"
#include "fa_common.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kScratchFloats = FA_NOALLOC_SCRATCH_BYTES / sizeof(float);

// Shared by every call on a device.  Holds whatever the last call left.
// The split kernels write every partial they later read, and the one word
// that must start at zero (the persistent prefill kernel's tile counter in
// the first bytes) is zeroed in stream order by each call before its launch.
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device).  Returns FA_OK or FA_ERR_CUDA.
int scratch_address(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v,
                                      const int* cu_seqlens_q, const int* cu_seqlens_k,
                                      int batch, int total_q, int total_k, int max_seqlen_q,
                                      int h_q, int h_kv, int d_qk, int d_v, float scale,
                                      int causal, int window_left, int num_splits, void* out,
                                      float* lse, int in_dtype, int out_dtype,
                                      const float* descale_q, const float* descale_k,
                                      const float* descale_v, int flags, void* stream) {
  if (batch < 0 || max_seqlen_q < 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || d_v <= 0 ||
      num_splits < 0 || num_splits > 128)
    return FA_ERR_INVALID_ARG;
  // Workspace the call needs; bigger problems than the fixed array are
  // refused here, before anything is launched.
  size_t need = 0;
  if (batch > 0 && max_seqlen_q > 0) {
    need = fa_fwd_splitkv_workspace_size(batch, max_seqlen_q, h_q, h_kv, d_v, num_splits);
    int ns = 0;
    if (fa_plan(batch, max_seqlen_q, h_q, h_kv, num_splits, 0, &ns, nullptr) != FA_OK)
      return FA_ERR_CUDA;
    if (ns > 1 && need == 0) return FA_ERR_INVALID_ARG;
  }
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  float* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  return fa_fwd_splitkv_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                           max_seqlen_q, h_q, h_kv, d_qk, d_v, scale, causal, window_left,
                           num_splits, out, lse, scratch, (size_t)FA_NOALLOC_SCRATCH_BYTES,
                           in_dtype, out_dtype, descale_q, descale_k, descale_v, flags, stream);
}
