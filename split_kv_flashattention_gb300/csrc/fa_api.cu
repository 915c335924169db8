// Host side of the C ABI declared in include/fa_splitkv.h: argument
// validation, the split planner, TMA descriptor encoding and kernel dispatch.
// Nothing here allocates device memory or synchronises a stream.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/fa_splitkv.h"
#include "fa_combine.cuh"
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

// Sticky device error word (one per device that loads the library).
__device__ int g_device_error;

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_sms[kMaxDevices] = {0};
int* g_err_ptr[kMaxDevices] = {nullptr};
std::map<std::pair<const void*, int>, int> g_smem_attr;

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Order of the persistent prefill kernel's tile walk (both longest first).
// Sequence-major: sequences by key count, each one's query pairs from the
// last down, every KV head of a (sequence, pair) together; a sequence's key
// prefix is then read by consecutive tiles while it is in L2.  m-major (a
// masked call's option): every sequence's last pair first, level by level,
// which revisits each (sequence, KV head) once per level; its KV heads can
// be walked in groups whose K/V fits kHeadGroupBytes of L2.
constexpr int kMaskedMmajor = 0;
constexpr long long kHeadGroupBytes = 32ll << 20;
void persistent_order(int h_kv, int total_k, int kv_row_elems, int es, bool masked,
                      int* mmajor, int* head_group) {
  *mmajor = masked && kMaskedMmajor;
  *head_group = h_kv;
  if (!*mmajor) return;
  const long long per_head = (long long)total_k * kv_row_elems * es;
  int best = 1;
  for (int g = 1; g <= h_kv; ++g)
    if (h_kv % g == 0 && (long long)g * per_head <= kHeadGroupBytes) best = g;
  *head_group = best;
}

// The partial kernel the calling thread's last forward call launched
// (fa_kernel_id), for fa_debug_last_kernel.
thread_local int t_last_kernel = FA_KID_NONE;

int current_device(int* dev) {
  return cudaGetDevice(dev) == cudaSuccess && *dev >= 0 && *dev < kMaxDevices ? FA_OK : FA_ERR_CUDA;
}

int device_sms(int* sms) {
  int dev;
  if (current_device(&dev) != FA_OK) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return FA_ERR_CUDA;
    g_sms[dev] = n;
  }
  *sms = g_sms[dev];
  return FA_OK;
}

int device_error_ptr(int** out) {
  int dev;
  if (current_device(&dev) != FA_OK) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return FA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_err_ptr[dev];
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// 3-D map over a packed [rows, heads, dim] buffer with a 128-byte-wide,
// 128B-swizzled box of box_heads heads x box_rows rows.  Rows past `rows`
// and columns past `dim` read as zero.
int make_tmap_3d(CUtensorMap* m, const void* base, int dtype, int dim, int heads, int rows,
                 int box_rows, int box_heads = 1) {
  auto enc = encoder();
  if (enc == nullptr) return FA_ERR_CUDA;
  const int es = dtype == kE4M3 ? 1 : 2;
  CUtensorMapDataType t = dtype == kE4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                          : dtype == kFP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t gstride[2] = {(cuuint64_t)dim * es, (cuuint64_t)dim * es * heads};
  cuuint32_t box[3] = {(cuuint32_t)(128 / es), (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  CUresult r = enc(m, t, 3, const_cast<void*>(base), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int plan_impl(int batch, int max_seqlen_q, int h_q, int h_kv, int num_splits, int num_sms,
              int* ns_out, int* units_out) {
  const int group = h_q / h_kv;
  const long long m_blocks = ((long long)max_seqlen_q * group + 127) / 128;
  const long long units = (long long)batch * h_kv * m_blocks;
  if (units_out) *units_out = (int)(units > 0x7fffffff ? 0x7fffffff : units);
  int ns;
  if (num_splits > 0) {
    ns = num_splits < kMaxSplits ? num_splits : kMaxSplits;
  } else if (units <= 0 || units >= 2LL * num_sms) {
    ns = 1;
  } else {
    ns = 0;
    long long best_num = 0, best_den = 1;
    int best_ns = 1;
    for (int s = 1; s <= kMaxSplits; ++s) {
      const long long work = units * s;
      const long long waves = (work + num_sms - 1) / num_sms;
      const long long den = waves * num_sms;
      if (10 * work >= 9 * den) {
        ns = s;
        break;
      }
      if (work * best_den > best_num * den) {
        best_ns = s;
        best_num = work;
        best_den = den;
      }
    }
    if (ns == 0) ns = best_ns;
  }
  *ns_out = ns;
  return FA_OK;
}

bool dims_supported(int in_dtype, int d_qk, int d_v) {
  if (in_dtype == kE4M3) return (d_qk == 128 || d_qk == 192) && d_v == 128;
  return (d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128) || (d_qk == 256 && d_v == 256);
}

}  // namespace

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(kernel, dev);
  auto it = g_smem_attr.find(key);
  if (it != g_smem_attr.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_smem_attr[key] = bytes;
  return e;
}

int simt_max_rows(int dtype, int d_qk, int d_v) {
  if (!dims_supported(dtype, d_qk, d_v)) return 0;
  if ((dtype == kE4M3 && d_qk == 192) || d_qk == 256) return 2;
  return 4;
}

// The most rows per KV head AUTO gives the CUDA-core kernel.  Measured on
// varlen and long decode: from 3 rows on (d = 128, 16-bit and e4m3) the
// one-tile tensor-core kernel streams K/V faster (GQA-4 batch: 6.87 against
// 6.21 TB/s), with 1 or 2 rows the CUDA-core kernel does; with d = 64 it
// stays ahead up to its 4-row limit.
int simt_auto_rows(int dtype, int d_qk, int d_v) {
  const int m = simt_max_rows(dtype, d_qk, d_v);
  return d_qk == 64 ? m : (m < 2 ? m : 2);
}

cudaError_t launch_simt(int dtype, int d_qk, int d_v, int rt, bool ordered, const FwdParams& p,
                        const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                        cudaStream_t stream) {
  switch (dtype) {
    case kBF16:
      return ordered ? launch_simt_t<kBF16, true>(d_qk, d_v, rt, p, tmK, tmV, grid, stream)
                     : launch_simt_t<kBF16, false>(d_qk, d_v, rt, p, tmK, tmV, grid, stream);
    case kFP16:
      return ordered ? launch_simt_t<kFP16, true>(d_qk, d_v, rt, p, tmK, tmV, grid, stream)
                     : launch_simt_t<kFP16, false>(d_qk, d_v, rt, p, tmK, tmV, grid, stream);
    case kE4M3:
      return ordered ? launch_simt_t<kE4M3, true>(d_qk, d_v, rt, p, tmK, tmV, grid, stream)
                     : launch_simt_t<kE4M3, false>(d_qk, d_v, rt, p, tmK, tmV, grid, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_umma(int dtype, int d_qk, int d_v, const FwdParams& p, const CUtensorMap& tmQ,
                        const CUtensorMap& tmK, const CUtensorMap& tmV, dim3 grid,
                        cudaStream_t stream) {
  switch (dtype) {
    case kBF16: return launch_umma_bf16(d_qk, d_v, p, tmQ, tmK, tmV, grid, stream);
    case kFP16: return launch_umma_fp16(d_qk, d_v, p, tmQ, tmK, tmV, grid, stream);
    case kE4M3: return launch_umma_e4m3(d_qk, d_v, p, tmQ, tmK, tmV, grid, stream);
  }
  return cudaErrorInvalidValue;
}

// The combine is launched with programmatic stream serialisation so its
// launch overlaps the tail of the partial kernel; it waits for the partial
// grid's writes with griddepcontrol.wait.
cudaError_t launch_combine(const FwdParams& p, cudaStream_t stream) {
  const long long warps = (long long)p.slots * p.h_q;
  const unsigned blocks = (unsigned)((warps + 3) / 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (p.d_v) {
    case 64: return cudaLaunchKernelEx(&cfg, combine_kernel<64>, p);
    case 128: return cudaLaunchKernelEx(&cfg, combine_kernel<128>, p);
    case 256: return cudaLaunchKernelEx(&cfg, combine_kernel<256>, p);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_split_ranges(const int* cu_q, const int* cu_k, int batch, int max_seqlen_q,
                                int causal, int window_left, int ns, int tile_q, int* out,
                                cudaStream_t stream) {
  const int m_blocks = (max_seqlen_q + tile_q - 1) / tile_q;
  const long long total = (long long)m_blocks * batch * ns;
  if (total == 0) return cudaSuccess;
  split_ranges_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(
      cu_q, cu_k, batch, max_seqlen_q, causal, window_left, ns, tile_q, m_blocks, out);
  return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    case FA_ERR_DEVICE_ARG: return "FA_ERR_DEVICE_ARG";
    case FA_ERR_DEVICE_BOUNDS: return "FA_ERR_DEVICE_BOUNDS";
  }
  return "FA_UNKNOWN_STATUS";
}

int fa_plan(int batch, int max_seqlen_q, int h_q, int h_kv, int num_splits, int num_sms,
            int* num_splits_out, int* units_out) {
  if (num_splits_out == nullptr || batch < 0 || max_seqlen_q < 0 || h_q <= 0 || h_kv <= 0 ||
      h_q % h_kv != 0 || num_splits < 0)
    return FA_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    int st = device_sms(&num_sms);
    if (st != FA_OK) return st;
  }
  return plan_impl(batch, max_seqlen_q, h_q, h_kv, num_splits, num_sms, num_splits_out, units_out);
}

size_t fa_fwd_splitkv_workspace_size(int batch, int max_seqlen_q, int h_q, int h_kv, int d_v,
                                     int num_splits) {
  if (batch < 0 || max_seqlen_q < 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || d_v <= 0 ||
      num_splits < 0 || num_splits > kMaxSplits)
    return 0;
  int ns = num_splits;
  if (ns == 0) {
    int sms;
    if (device_sms(&sms) != FA_OK) return 0;
    plan_impl(batch, max_seqlen_q, h_q, h_kv, 0, sms, &ns, nullptr);
  }
  if (ns <= 1) return kSchedBytes;  // the persistent kernel's ticket counter
  const size_t slots = (size_t)batch * max_seqlen_q * h_q;
  return 4 * (size_t)ns * slots * (size_t)(d_v + 1);
}

int fa_get_device_error(int clear) {
  int* ptr = nullptr;
  int st = device_error_ptr(&ptr);
  if (st != FA_OK) return st;
  int v = 0;
  if (cudaMemcpy(&v, ptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (clear && v != 0) {
    int z = 0;
    if (cudaMemcpy(ptr, &z, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  }
  return v;
}

int fa_debug_last_kernel(void) { return t_last_kernel; }

int fa_debug_wait_timeout(unsigned int timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return FA_ERR_INVALID_ARG;
  int* err = nullptr;
  const int st = device_error_ptr(&err);
  if (st != FA_OK) return st;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      err, (unsigned long long)timeout_ms * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_debug_split_ranges(const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                          int max_seqlen_q, int causal, int window_left, int num_splits,
                          int tile_queries, int* ranges_out, void* stream) {
  if (batch < 0 || max_seqlen_q < 0 || num_splits < 1 || num_splits > kMaxSplits ||
      tile_queries < 1)
    return FA_ERR_INVALID_ARG;
  if (batch == 0 || max_seqlen_q == 0) return FA_OK;
  if (!cu_seqlens_q || !cu_seqlens_k || !ranges_out) return FA_ERR_INVALID_ARG;
  cudaError_t e = launch_split_ranges(cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, causal,
                                      window_left, num_splits, tile_queries, ranges_out,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Shared body of fa_fwd_splitkv_ex (contiguous K/V addressed by cu_seqlens_k)
// and fa_fwd_splitkv_paged (page pools addressed by block_table/seqlens_k,
// page_size > 0).
int fwd_impl(const void* q, const void* k, const void* v, const int* cu_seqlens_q,
             const int* cu_seqlens_k, int batch, int total_q, int total_k, int max_seqlen_q,
             int h_q, int h_kv, int d_qk, int d_v, float scale, int causal, int window_left,
             int num_splits, void* out, float* lse, void* workspace, size_t workspace_bytes,
             int in_dtype, int out_dtype, const float* descale_q, const float* descale_k,
             const float* descale_v, int flags, void* stream, const int* block_table,
             const int* seqlens_k, int max_pages, int page_size) {
  const bool paged = page_size > 0;
  t_last_kernel = FA_KID_NONE;
  // ---- argument validation (synchronous, before any launch)
  if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0) return FA_ERR_INVALID_ARG;
  if (h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || h_q / h_kv > 128) return FA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  if (in_dtype != kBF16 && in_dtype != kFP16 && in_dtype != kE4M3) return FA_ERR_INVALID_ARG;
  if (out_dtype != kBF16 && out_dtype != kFP16 && out_dtype != kE4M3) return FA_ERR_INVALID_ARG;
  // 16-bit inputs write their own type or e4m3; e4m3 inputs write any of the three
  if (in_dtype != kE4M3 && out_dtype != in_dtype && out_dtype != kE4M3) return FA_ERR_UNSUPPORTED;
  if (!dims_supported(in_dtype, d_qk, d_v)) return FA_ERR_UNSUPPORTED;
  if (isnan(scale) || isinf(scale)) return FA_ERR_INVALID_ARG;
  const int kernel_sel = flags & FA_KERNEL_MASK;
  if (kernel_sel == FA_KERNEL_UMMA2 && (in_dtype == kE4M3 || d_qk > 128)) return FA_ERR_UNSUPPORTED;
  if (flags & ~(FA_KERNEL_MASK | FA_RUN_PARTIAL_ONLY | FA_RUN_COMBINE_ONLY)) return FA_ERR_INVALID_ARG;
  const bool run_partial = !(flags & FA_RUN_COMBINE_ONLY);
  const bool run_combine = !(flags & FA_RUN_PARTIAL_ONLY);
  if (!run_partial && !run_combine) return FA_ERR_INVALID_ARG;
  if (batch == 0 || max_seqlen_q == 0 || total_q == 0) return FA_OK;  // nothing to compute
  if (!q || !k || !v || !cu_seqlens_q || !out) return FA_ERR_INVALID_ARG;
  if (!paged && !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  if (paged && (!block_table || !seqlens_k || max_pages <= 0)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
  const int es = in_dtype == kE4M3 ? 1 : 2;
  if (((long long)h_q * d_qk * es) % 16 || ((long long)h_kv * d_qk * es) % 16 ||
      ((long long)h_kv * d_v * es) % 16)
    return FA_ERR_INVALID_ARG;
  if (in_dtype == kE4M3 && (!descale_q || !descale_k || !descale_v)) return FA_ERR_INVALID_ARG;

  // ---- plan (the device is queried only for an automatic split count)
  int sms = 1;
  int st = FA_OK;
  if (num_splits == 0) {
    st = device_sms(&sms);
    if (st != FA_OK) return st;
  }
  int ns = 1;
  plan_impl(batch, max_seqlen_q, h_q, h_kv, num_splits, sms, &ns, nullptr);
  const long long slots = (long long)batch * max_seqlen_q;
  if (slots > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  const size_t need = ns > 1 ? 4 * (size_t)ns * slots * h_q * (size_t)(d_v + 1) : 0;
  if (need > 0) {
    if (workspace == nullptr || !aligned16(workspace)) return FA_ERR_WORKSPACE;
    if (workspace_bytes != (size_t)-1 && workspace_bytes < need) return FA_ERR_WORKSPACE;
  }
  int* err = nullptr;
  st = device_error_ptr(&err);
  if (st != FA_OK) return st;

  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.q = q;
  p.k = k;
  p.v = v;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.out = out;
  p.lse = lse;
  p.ws_o = ns > 1 ? static_cast<float*>(workspace) : nullptr;
  p.ws_l = ns > 1 ? static_cast<float*>(workspace) + (size_t)ns * slots * h_q * d_v : nullptr;
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  p.descale_v = descale_v;
  p.err = err;
  p.batch = batch;
  p.total_q = total_q;
  p.total_k = total_k;
  p.max_seqlen_q = max_seqlen_q;
  p.h_q = h_q;
  p.h_kv = h_kv;
  p.group = h_q / h_kv;
  p.d_qk = d_qk;
  p.d_v = d_v;
  p.num_splits = ns;
  p.causal = causal ? 1 : 0;
  p.window_left = window_left < 0 ? -1 : window_left;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)d_qk);
  p.out_dtype = out_dtype;
  p.slots = (int)slots;
  p.block_table = paged ? block_table : nullptr;
  p.seqlens_k = paged ? seqlens_k : nullptr;
  p.max_pages = paged ? max_pages : 0;
  p.page_size = paged ? page_size : 0;
  p.page_shift = 0;
  while (paged && (1 << p.page_shift) < page_size) ++p.page_shift;
  // SM count (already queried for an automatic split count; a failed query
  // only disables the kernels' look-ahead prefetch)
  p.num_sms = sms;
  if (num_splits != 0 && device_sms(&p.num_sms) != FA_OK) p.num_sms = 0;

  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // ---- kernel choice: few rows per KV head (decode) stream on the CUDA
  // cores; more rows form a dense contraction for the tensor cores.
  const int rows = max_seqlen_q * p.group;
  const int rt_max = simt_max_rows(in_dtype, d_qk, d_v);
  const bool auto_tc = kernel_sel == FA_KERNEL_AUTO && rows > simt_auto_rows(in_dtype, d_qk, d_v);
  // More than one 128-row tile per KV head with 16-bit inputs: two tiles per
  // CTA share each K/V block and overlap their softmax with the other tile's
  // MMAs.  Otherwise one tile per CTA.
  const bool use_umma2 =
      kernel_sel == FA_KERNEL_UMMA2 || (auto_tc && rows > 128 && in_dtype != kE4M3 && d_qk <= 128);
  const bool use_umma = !use_umma2 && (kernel_sel == FA_KERNEL_UMMA || auto_tc);
  if ((unsigned)(batch * h_kv) > 65535u) return FA_ERR_UNSUPPORTED;
  if (run_partial) {
    CUtensorMap tmK, tmV;
    int box_keys = (use_umma || use_umma2) ? kBlockN : 32;
    if (paged && page_size < box_keys) box_keys = page_size;  // one load per page piece
    st = make_tmap_3d(&tmK, k, in_dtype, d_qk, h_kv, total_k, box_keys);
    if (st != FA_OK) return st;
    st = make_tmap_3d(&tmV, v, in_dtype, d_v, h_kv, total_k, box_keys);
    if (st != FA_OK) return st;
    cudaError_t e;
    int launched = FA_KID_NONE;
    if (use_umma2) {
      const int qpt = 128 / p.group;
      p.tile_rows = 2 * qpt * p.group;
      CUtensorMap tmQ;
      st = make_tmap_3d(&tmQ, q, in_dtype, d_qk, h_q, total_q, qpt, p.group);
      if (st != FA_OK) return st;
      // One split over packed K/V, chosen automatically: the persistent form
      // walks a tile list held in shared memory, so the batch and its query
      // pairs must fit that list; it claims tiles from a ticket counter kept
      // in the first bytes of the workspace (zeroed here, in stream order);
      // and it writes O rows with 32-byte stores, so out must be 32-byte
      // aligned (rows are then too: h_q * d_v * element size is a multiple
      // of 32).  Otherwise the non-persistent grid runs.
      const long long pairs = ceil_div(max_seqlen_q, 2 * qpt);
      const bool has_sched = workspace != nullptr && aligned16(workspace) &&
                             (workspace_bytes == (size_t)-1 || workspace_bytes >= kSchedBytes);
      const bool out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
      const bool persistent = kernel_sel == FA_KERNEL_AUTO && ns == 1 && !paged && has_sched &&
                              out32 && batch <= 128 && pairs <= kMaxUnitPairs &&
                              (long long)batch * pairs <= kMaxUnits;
      if (persistent) {
        int sms = 0;
        st = device_sms(&sms);
        if (st != FA_OK) return st;
        const long long tiles = (long long)batch * pairs * h_kv;
        dim3 grid((unsigned)(tiles < sms ? tiles : sms), 1, 1);
        p.sched = static_cast<int*>(workspace);
        persistent_order(h_kv, total_k, d_qk + d_v, es, p.causal || p.window_left >= 0,
                         &p.unit_mmajor, &p.kv_head_group);
        if (cudaMemsetAsync(p.sched, 0, sizeof(int), s) != cudaSuccess) return FA_ERR_CUDA;
        e = in_dtype == kFP16 ? launch_umma2p_fp16(d_qk, d_v, p, tmQ, tmK, tmV, grid, s)
                              : launch_umma2p_bf16(d_qk, d_v, p, tmQ, tmK, tmV, grid, s);
        launched = FA_KID_UMMA2_PERSISTENT;
      } else {
        dim3 grid((unsigned)ceil_div(max_seqlen_q, 2 * qpt), (unsigned)(batch * h_kv), (unsigned)ns);
        e = in_dtype == kFP16 ? launch_umma2_fp16(d_qk, d_v, p, tmQ, tmK, tmV, grid, s)
                              : launch_umma2_bf16(d_qk, d_v, p, tmQ, tmK, tmV, grid, s);
        launched = FA_KID_UMMA2;
      }
    } else if (use_umma) {
      const int qpt = 128 / p.group;
      p.tile_rows = qpt * p.group;
      CUtensorMap tmQ;
      st = make_tmap_3d(&tmQ, q, in_dtype, d_qk, h_q, total_q, qpt, p.group);
      if (st != FA_OK) return st;
      dim3 grid((unsigned)ceil_div(max_seqlen_q, qpt), (unsigned)(batch * h_kv), (unsigned)ns);
      e = launch_umma(in_dtype, d_qk, d_v, p, tmQ, tmK, tmV, grid, s);
      launched = FA_KID_UMMA;
    } else {
      int rt = 1;
      while (rt < rows && rt < rt_max) rt *= 2;
      p.tile_rows = rt;
      dim3 grid((unsigned)ceil_div(rows, rt), (unsigned)(batch * h_kv), (unsigned)ns);
      // Longest sequence first pays off once there are several sequences of
      // different lengths to balance; one sequence keeps the grid order.
      const bool ordered = batch > 1 && batch <= kMaxRankedSeqs;
      e = launch_simt(in_dtype, d_qk, d_v, rt, ordered, p, tmK, tmV, grid, s);
      launched = FA_KID_SIMT;
    }
    if (e != cudaSuccess) return FA_ERR_CUDA;
    t_last_kernel = launched;
  }
  if (run_combine && ns > 1) {
    cudaError_t e;
    e = launch_combine(p, s);
    if (e != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd_splitkv_ex(const void* q, const void* k, const void* v, const int* cu_seqlens_q,
                      const int* cu_seqlens_k, int batch, int total_q, int total_k,
                      int max_seqlen_q, int h_q, int h_kv, int d_qk, int d_v, float scale,
                      int causal, int window_left, int num_splits, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, int in_dtype, int out_dtype,
                      const float* descale_q, const float* descale_k, const float* descale_v,
                      int flags, void* stream) {
  return fwd_impl(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, max_seqlen_q,
                  h_q, h_kv, d_qk, d_v, scale, causal, window_left, num_splits, out, lse,
                  workspace, workspace_bytes, in_dtype, out_dtype, descale_q, descale_k,
                  descale_v, flags, stream, nullptr, nullptr, 0, 0);
}

int fa_fwd_splitkv_paged(const void* q, const void* k_cache, const void* v_cache,
                         const int* cu_seqlens_q, const int* seqlens_k, const int* block_table,
                         int batch, int total_q, int num_pages, int page_size,
                         int max_pages_per_seq, int max_seqlen_q, int h_q, int h_kv, int d_qk,
                         int d_v, float scale, int causal, int window_left, int num_splits,
                         void* out, float* lse, void* workspace, size_t workspace_bytes,
                         int in_dtype, int out_dtype, const float* descale_q,
                         const float* descale_k, const float* descale_v, int flags,
                         void* stream) {
  if (page_size < kMinPage || (page_size & (page_size - 1)) != 0 || page_size > (1 << 20))
    return FA_ERR_INVALID_ARG;
  if (num_pages < 0 || max_pages_per_seq < 0 || (long long)num_pages * page_size > 0x7fffffffLL)
    return FA_ERR_INVALID_ARG;
  if (batch > 0 && max_seqlen_q > 0 && total_q > 0 && (num_pages == 0 || max_pages_per_seq == 0))
    return FA_ERR_INVALID_ARG;
  return fwd_impl(q, k_cache, v_cache, cu_seqlens_q, nullptr, batch, total_q,
                  num_pages * page_size, max_seqlen_q, h_q, h_kv, d_qk, d_v, scale, causal,
                  window_left, num_splits, out, lse, workspace, workspace_bytes, in_dtype,
                  out_dtype, descale_q, descale_k, descale_v, flags, stream, block_table,
                  seqlens_k, max_pages_per_seq, page_size);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, const int* cu_seqlens_q,
                   const int* cu_seqlens_k, int batch, int total_q, int total_k,
                   int max_seqlen_q, int h_q, int h_kv, int d_qk, int d_v, float scale,
                   int causal, int window_left, int num_splits, void* out, float* lse,
                   void* workspace, void* stream) {
  return fa_fwd_splitkv_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                           max_seqlen_q, h_q, h_kv, d_qk, d_v, scale, causal, window_left,
                           num_splits, out, lse, workspace, (size_t)-1, FA_BF16, FA_BF16,
                           nullptr, nullptr, nullptr, FA_KERNEL_AUTO, stream);
}

}  // extern "C"
