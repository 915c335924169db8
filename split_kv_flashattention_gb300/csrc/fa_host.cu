// fa_fwd_splitkv_host: the split-KV forward on host buffers.
//
// The inputs are copied from host memory into a caller-owned device buffer,
// the forward pass runs on those copies, and O and LSE are copied back to
// host memory: every step is stream-ordered on the caller's stream (one
// cudaMemcpyAsync per buffer), and nothing is allocated.  The device buffer
// is carved into 256-byte aligned regions in a fixed order: Q, K, V,
// cu_seqlens_q, cu_seqlens_k, the three descales (e4m3 inputs), O, LSE and
// the split workspace.
#include <stdint.h>

#include "../../include/fa_splitkv.h"
#include "fa_common.cuh"

namespace {

struct HostLayout {
  size_t q, k, v, cq, ck, dsc, out, lse, ws, ws_bytes, total;
  size_t q_bytes, k_bytes, v_bytes, cu_bytes, out_bytes, lse_bytes;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int elem_size(int dtype) {
  if (dtype == FA_E4M3) return 1;
  if (dtype == FA_BF16 || dtype == FA_FP16) return 2;
  return 0;
}

// The regions of the device buffer; false for sizes or dtypes no call takes.
bool host_layout(int batch, int total_q, int total_k, int max_seqlen_q, int h_q, int h_kv,
                 int d_qk, int d_v, int in_dtype, int out_dtype, int num_splits, HostLayout* L) {
  const int es = elem_size(in_dtype), oes = elem_size(out_dtype);
  if (es == 0 || oes == 0 || batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 ||
      h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || d_qk <= 0 || d_v <= 0 || num_splits < 0 ||
      num_splits > 128)
    return false;
  L->q_bytes = (size_t)total_q * h_q * d_qk * es;
  L->k_bytes = (size_t)total_k * h_kv * d_qk * es;
  L->v_bytes = (size_t)total_k * h_kv * d_v * es;
  L->cu_bytes = (size_t)(batch + 1) * sizeof(int);
  L->out_bytes = (size_t)total_q * h_q * d_v * oes;
  L->lse_bytes = (size_t)h_q * total_q * sizeof(float);
  L->ws_bytes = 0;
  if (batch > 0 && max_seqlen_q > 0) {
    L->ws_bytes = fa_fwd_splitkv_workspace_size(batch, max_seqlen_q, h_q, h_kv, d_v, num_splits);
    if (L->ws_bytes == 0) return false;
  }
  size_t o = 0;
  L->q = o;
  o = align256(o + L->q_bytes);
  L->k = o;
  o = align256(o + L->k_bytes);
  L->v = o;
  o = align256(o + L->v_bytes);
  L->cq = o;
  o = align256(o + L->cu_bytes);
  L->ck = o;
  o = align256(o + L->cu_bytes);
  L->dsc = o;
  o = align256(o + 3 * sizeof(float));
  L->out = o;
  o = align256(o + L->out_bytes);
  L->lse = o;
  o = align256(o + L->lse_bytes);
  L->ws = o;
  o = align256(o + L->ws_bytes);
  L->total = o;
  return true;
}

int h2d(char* base, size_t off, const void* src, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return FA_OK;
  if (src == nullptr) return FA_ERR_INVALID_ARG;
  return cudaMemcpyAsync(base + off, src, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // namespace

extern "C" size_t fa_fwd_splitkv_host_buffer_size(int batch, int total_q, int total_k,
                                                  int max_seqlen_q, int h_q, int h_kv, int d_qk,
                                                  int d_v, int in_dtype, int out_dtype,
                                                  int num_splits) {
  HostLayout L;
  if (!host_layout(batch, total_q, total_k, max_seqlen_q, h_q, h_kv, d_qk, d_v, in_dtype,
                   out_dtype, num_splits, &L))
    return 0;
  return L.total;
}

extern "C" int fa_fwd_splitkv_host(const void* q, const void* k, const void* v,
                                   const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                                   int total_q, int total_k, int max_seqlen_q, int h_q, int h_kv,
                                   int d_qk, int d_v, float scale, int causal, int window_left,
                                   int num_splits, void* out, float* lse, void* device_buffer,
                                   size_t device_buffer_bytes, int in_dtype, int out_dtype,
                                   const float* descale_q, const float* descale_k,
                                   const float* descale_v, int flags, void* stream) {
  HostLayout L;
  if (!host_layout(batch, total_q, total_k, max_seqlen_q, h_q, h_kv, d_qk, d_v, in_dtype,
                   out_dtype, num_splits, &L))
    return FA_ERR_INVALID_ARG;
  if (device_buffer == nullptr || (reinterpret_cast<uintptr_t>(device_buffer) & 255u) != 0)
    return FA_ERR_INVALID_ARG;
  if (device_buffer_bytes < L.total) return FA_ERR_WORKSPACE;
  if ((L.out_bytes > 0 && out == nullptr) || cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)
    return FA_ERR_INVALID_ARG;
  const bool fp8 = in_dtype == FA_E4M3;
  if (fp8 && (descale_q == nullptr || descale_k == nullptr || descale_v == nullptr))
    return FA_ERR_INVALID_ARG;
  char* base = static_cast<char*>(device_buffer);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int st;
  if ((st = h2d(base, L.q, q, L.q_bytes, s)) != FA_OK) return st;
  if ((st = h2d(base, L.k, k, L.k_bytes, s)) != FA_OK) return st;
  if ((st = h2d(base, L.v, v, L.v_bytes, s)) != FA_OK) return st;
  if ((st = h2d(base, L.cq, cu_seqlens_q, L.cu_bytes, s)) != FA_OK) return st;
  if ((st = h2d(base, L.ck, cu_seqlens_k, L.cu_bytes, s)) != FA_OK) return st;
  float* dsc = reinterpret_cast<float*>(base + L.dsc);
  if (fp8) {
    if ((st = h2d(base, L.dsc, descale_q, sizeof(float), s)) != FA_OK) return st;
    if ((st = h2d(base, L.dsc + sizeof(float), descale_k, sizeof(float), s)) != FA_OK) return st;
    if ((st = h2d(base, L.dsc + 2 * sizeof(float), descale_v, sizeof(float), s)) != FA_OK)
      return st;
  }
  st = fa_fwd_splitkv_ex(base + L.q, base + L.k, base + L.v,
                         reinterpret_cast<const int*>(base + L.cq),
                         reinterpret_cast<const int*>(base + L.ck), batch, total_q, total_k,
                         max_seqlen_q, h_q, h_kv, d_qk, d_v, scale, causal, window_left,
                         num_splits, base + L.out,
                         lse != nullptr ? reinterpret_cast<float*>(base + L.lse) : nullptr,
                         L.ws_bytes > 0 ? base + L.ws : nullptr, L.ws_bytes, in_dtype, out_dtype,
                         fp8 ? dsc : nullptr, fp8 ? dsc + 1 : nullptr, fp8 ? dsc + 2 : nullptr,
                         flags, stream);
  if (st != FA_OK) return st;
  if (L.out_bytes > 0 &&
      cudaMemcpyAsync(out, base + L.out, L.out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FA_ERR_CUDA;
  if (lse != nullptr && L.lse_bytes > 0 &&
      cudaMemcpyAsync(lse, base + L.lse, L.lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}
