// Element conversions between the storage types (bf16, fp16, e4m3) and fp32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "fa_common.cuh"

namespace fa {

template <int DT>
struct Elem;
template <>
struct Elem<kBF16> {
  static constexpr int size = 2;
};
template <>
struct Elem<kFP16> {
  static constexpr int size = 2;
};
template <>
struct Elem<kE4M3> {
  static constexpr int size = 1;
};

// One 32-bit word of packed elements -> floats (2 for 16-bit, 4 for e4m3).
template <int DT>
__device__ __forceinline__ void word_to_float(uint32_t w, float* f);

template <>
__device__ __forceinline__ void word_to_float<kBF16>(uint32_t w, float* f) {
  f[0] = __uint_as_float(w << 16);
  f[1] = __uint_as_float(w & 0xffff0000u);
}

template <>
__device__ __forceinline__ void word_to_float<kFP16>(uint32_t w, float* f) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  float2 v = __half22float2(h);
  f[0] = v.x;
  f[1] = v.y;
}

template <>
__device__ __forceinline__ void word_to_float<kE4M3>(uint32_t w, float* f) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu),
                                               __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16),
                                               __NV_E4M3);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

template <int DT>
struct PerWord {
  static constexpr int n = 4 / Elem<DT>::size;
};

// NW words -> NW * PerWord floats.
template <int DT, int NWORDS>
__device__ __forceinline__ void words_to_float(const uint32_t* w, float* f) {
#pragma unroll
  for (int i = 0; i < NWORDS; ++i) word_to_float<DT>(w[i], f + i * PerWord<DT>::n);
}

// ----------------------------------------------------------- packed fp32x2
// Two fp32 values in one 64-bit register pair; sm_100-class SMs execute
// fma/mul on such pairs as one instruction (twice the FP32 rate per issue).
using f32x2 = unsigned long long;

__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ float2 f2_split(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

// a * b + c on both halves
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max of three fp32 values in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// One 32-bit word of packed elements -> pairs (1 pair for 16-bit, 2 for e4m3).
template <int DT>
__device__ __forceinline__ void word_to_f2(uint32_t w, f32x2* f) {
  float t[4];
  word_to_float<DT>(w, t);
  f[0] = f2_make(t[0], t[1]);
  if constexpr (DT == kE4M3) f[1] = f2_make(t[2], t[3]);
}

// Two floats -> one packed 16-bit pair for the output type (round to nearest).
__device__ __forceinline__ uint32_t pack2(float a, float b, int out_dtype) {
  if (out_dtype == kFP16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// N consecutive output elements (already normalised, times `scale`) at
// element index `elem` of O: 16-bit types as 2N bytes (round to nearest), e4m3
// as N bytes (round to nearest even, saturating to +-448).  N is 2, 4, 8 or
// 32; the address is aligned to the store width (2N or N bytes).  WIDE (N = 32
// only): 32-byte stores, the address 32-byte aligned.
__device__ __forceinline__ void st_global_32B(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
template <int N, bool WIDE = false>
__device__ __forceinline__ void store_o(void* out, size_t elem, const float* f, float scale,
                                        int out_dtype) {
  static_assert(!WIDE || N == 32, "wide stores take 32 values");
  static_assert(N == 2 || N == 4 || N == 8 || N == 32, "store width");
  if (out_dtype == kE4M3) {
    uint8_t* dst = static_cast<uint8_t*>(out) + elem;
    uint32_t w[(N + 3) / 4];
#pragma unroll
    for (int i = 0; i < (N + 3) / 4; ++i) w[i] = 0u;
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const uint32_t two = (uint32_t)__nv_cvt_float2_to_fp8x2(
          make_float2(f[i] * scale, f[i + 1] * scale), __NV_SATFINITE, __NV_E4M3);
      w[i / 4] |= two << (8 * (i % 4));
    }
    if constexpr (N == 2) {
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w[0];
    } else if constexpr (N == 4) {
      *reinterpret_cast<uint32_t*>(dst) = w[0];
    } else if constexpr (N == 8) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else if constexpr (WIDE) {
      st_global_32B(dst, w);
    } else {
#pragma unroll
      for (int i = 0; i < N / 16; ++i)
        reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  } else {
    uint8_t* dst = static_cast<uint8_t*>(out) + elem * 2;
    uint32_t w[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) w[i] = pack2(f[2 * i] * scale, f[2 * i + 1] * scale, out_dtype);
    if constexpr (N == 2) {
      *reinterpret_cast<uint32_t*>(dst) = w[0];
    } else if constexpr (N == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else if constexpr (WIDE) {
      st_global_32B(dst, w);
      st_global_32B(dst + 32, w + 8);
    } else {
#pragma unroll
      for (int i = 0; i < N / 8; ++i)
        reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
}

// Output row of one warp (lane l holds columns [l*DPL, (l+1)*DPL)) written
// with 16-byte stores.  W packed 32-bit words per lane; the first lane of
// every group of 4/W lanes collects the group's 16 bytes.  The row starts
// on a 16-byte boundary (O is 16-byte aligned, rows are d_v elements).
template <int W>
__device__ __forceinline__ void store_row_16B(uint8_t* row, int lane, const uint32_t* w) {
  constexpr int G = 4 / W;
  uint32_t v[4];
#pragma unroll
  for (int i = 0; i < W; ++i) v[i] = w[i];
#pragma unroll
  for (int g = 1; g < G; ++g)
#pragma unroll
    for (int i = 0; i < W; ++i) v[g * W + i] = __shfl_down_sync(0xffffffffu, w[i], g);
  if ((lane & (G - 1)) == 0)
    *reinterpret_cast<uint4*>(row + lane * W * 4) = make_uint4(v[0], v[1], v[2], v[3]);
}

template <int DPL>
__device__ __forceinline__ void store_combined_row(void* out, size_t row_elem, const float* f,
                                                   int lane, int out_dtype) {
  if (out_dtype == kE4M3) {
    if constexpr (DPL % 4 == 0) {
      uint32_t w[DPL / 4];
#pragma unroll
      for (int i = 0; i < DPL / 4; ++i) {
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(f[4 * i], f[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(f[4 * i + 2], f[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
        w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      store_row_16B<DPL / 4>(static_cast<uint8_t*>(out) + row_elem, lane, w);
    } else {
      store_o<DPL>(out, row_elem + lane * DPL, f, 1.f, out_dtype);
    }
  } else {
    uint32_t w[DPL / 2];
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) w[i] = pack2(f[2 * i], f[2 * i + 1], out_dtype);
    store_row_16B<DPL / 2>(static_cast<uint8_t*>(out) + row_elem * 2, lane, w);
  }
}

}  // namespace fa
