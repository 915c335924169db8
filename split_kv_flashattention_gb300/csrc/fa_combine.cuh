// LSE-weighted combine of split partials (flash-decoding's second kernel).
//
// aiter PR "[FlyDSL] Enable FP8 FMHA split-K for short cached-prefix
// queries": the timed unit is "attention and split combine", with a per-call
// fp32 workspace.  For every output row (token t, head h) one warp reads the
// ns partial LSEs (lanes take splits s, s+32, ...) together with the partial
// O rows (one round of loads for up to 16 splits), forms
//     M = max_s lse_s,  w_s = exp(lse_s - M),  LSE = M + ln(sum_s w_s)
// and accumulates O = sum_s (w_s / sum w) * O_s with 128-bit loads, lane l
// owning columns [l*d_v/32, (l+1)*d_v/32).  The row is written with 128-bit
// stores: lanes convert their columns to the output type and the first lane
// of each group that makes 16 bytes gathers the group's words by shuffles
// (d_v = 128, 16-bit: 16 lanes store 8 values each).  Rows whose splits are
// all empty (M = -inf) get O = 0 and LSE = -inf.
#pragma once

#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_convert.cuh"
#include "fa_ptx.cuh"

namespace fa {

template <int DV>
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ FwdParams p) {
  constexpr int DPL = DV / 32;
  constexpr int CH = DPL >= 8 ? 8 : 16;  // partial O rows loaded per round
  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const bool in_grid = gw < (long long)p.slots * p.h_q;
  const int slot = in_grid ? (int)(gw / p.h_q) : 0;
  const int h = in_grid ? (int)(gw - (long long)slot * p.h_q) : 0;
  const int b = slot / p.max_seqlen_q;
  const int i = slot - b * p.max_seqlen_q;
  // The sequence offsets do not come from the partial kernel: read them
  // before waiting for it (programmatic dependent launch).
  SeqInfo sq;
  const bool valid = in_grid && load_seq(p, b, sq) && i < sq.lq;  // bad offsets: reported by the partial kernel
  pdl_wait();
  // The next kernel in the stream may start its prologue now (its own
  // griddepcontrol.wait still waits for this grid to finish).
  pdl_launch_dependents();
  if (!valid) return;
  // A recorded timeout means the partials are incomplete: write nothing (the
  // word is read with the partials, in the same round of loads).
  const bool timed_out = timed_out_before(p.err);
  const int t = sq.q0 + i;
  const int ns = p.num_splits;
  const size_t split_stride = (size_t)p.slots * p.h_q;
  const size_t row0 = (size_t)slot * p.h_q + h;
  const float* obase = p.ws_o + row0 * DV + lane * DPL;
  const size_t ostride = split_stride * DV;

  // One round of loads: every partial LSE (lane l holds splits l, l+32, ...)
  // and the first CH partial O rows.  Splits past a sequence's key range were
  // written as O = 0, LSE = -inf, so every split below ns is readable.
  auto load_o = [&](int s, float* v) {
    const float* src = obase + (size_t)s * ostride;
    if (!ws_o_ok(p, (size_t)(src - p.ws_o), DPL)) src = p.ws_o;
    if constexpr (DPL % 4 == 0) {
#pragma unroll
      for (int e = 0; e < DPL; e += 4) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(src + e));
        v[e] = q.x;
        v[e + 1] = q.y;
        v[e + 2] = q.z;
        v[e + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < DPL; e += 2) {
        const float2 q = __ldg(reinterpret_cast<const float2*>(src + e));
        v[e] = q.x;
        v[e + 1] = q.y;
      }
    }
  };
  float ov[CH][DPL];
#pragma unroll
  for (int c = 0; c < CH; ++c)
    if (c < ns) load_o(c, ov[c]);
  float lv[kMaxSplits / 32];
#pragma unroll
  for (int u = 0; u < kMaxSplits / 32; ++u) {
    const int s = u * 32 + lane;
    lv[u] = s < ns && ws_l_ok(p, s * split_stride + row0) ? __ldg(p.ws_l + s * split_stride + row0)
                                                          : -CUDART_INF_F;
  }

  constexpr float kLog2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.69314718055994531f;
  float M = -CUDART_INF_F;
#pragma unroll
  for (int u = 0; u < kMaxSplits / 32; ++u) M = fmaxf(M, lv[u]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  float lse_out = -CUDART_INF_F;
  if (M != -CUDART_INF_F) {
    float w[kMaxSplits / 32];
    float L = 0.f;
#pragma unroll
    for (int u = 0; u < kMaxSplits / 32; ++u) {
      w[u] = fast_exp2((lv[u] - M) * kLog2e);  // empty split: exp2(-inf) = 0
      L += w[u];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float inv = 1.f / L;
    lse_out = M + __log2f(L) * kLn2;
#pragma unroll
    for (int u = 0; u < kMaxSplits / 32; ++u) w[u] *= inv;
    for (int s0 = 0; s0 < ns; s0 += CH) {
      if (s0 > 0) {
#pragma unroll
        for (int c = 0; c < CH; ++c)
          if (s0 + c < ns) load_o(s0 + c, ov[c]);
      }
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int s = s0 + c;
        if (s < ns) {
          const int u = s >> 5;
          const float wu = u == 0 ? w[0] : u == 1 ? w[1] : u == 2 ? w[2] : w[3];
          const float ws = __shfl_sync(0xffffffffu, wu, s & 31);
          if (ws != 0.f) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[e] = fmaf(ws, ov[c][e], acc[e]);
          }
        }
      }
    }
  }

  if (__any_sync(0xffffffffu, timed_out)) return;
  if (o_ok(p, ((size_t)t * p.h_q + h) * DV, DV))  // warp-uniform
    store_combined_row<DPL>(p.out, ((size_t)t * p.h_q + h) * DV, acc, lane, p.out_dtype);
  if (p.lse != nullptr && lane == 0 && lse_ok(p, h, t)) p.lse[(size_t)h * p.total_q + t] = lse_out;
}

// Test hook: one thread waits, through the kernels' own bounded wait, on an
// mbarrier phase that no thread ever completes.  The wait gives up after
// timeout_ns, records FA_ERR_DEVICE_TIMEOUT in the device error word and the
// kernel returns: the path a broken pipeline takes, without breaking one.
__global__ void wait_timeout_kernel(int* err, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, err, &abort_flag, timeout_ns);
}

// Test hook: the per-split key ranges the kernels compute, for a tile of
// `tile_q` queries.  One thread per (m_block, b, split).
__global__ void split_ranges_kernel(const int* cu_q, const int* cu_k, int batch, int max_seqlen_q,
                                    int causal, int window_left, int ns, int tile_q, int m_blocks,
                                    int* out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)m_blocks * batch * ns;
  if (idx >= total) return;
  const int s = (int)(idx % ns);
  const int b = (int)((idx / ns) % batch);
  const int m = (int)(idx / ((long long)ns * batch));
  const int lq = cu_q[b + 1] - cu_q[b];
  const int lk = cu_k[b + 1] - cu_k[b];
  int k0 = 0, k1 = 0;
  const int i_lo = m * tile_q;
  if (i_lo < lq) {
    const int i_hi = min(lq - 1, i_lo + tile_q - 1);
    tile_split_range(i_lo, i_hi, lq, lk, causal, window_left, ns, s, k0, k1);
  }
  out[2 * idx] = k0;
  out[2 * idx + 1] = k1;
}

}  // namespace fa
