// CUDA-core split-KV partial kernel for few query rows per KV head (decode,
// GQA decode).  Such a tile is a matrix-vector product per key: it is bound
// by the HBM stream of K and V, not by arithmetic, so it stays on the FP32
// pipes and spends its effort on keeping bytes in flight.
//
// One CTA = one (row tile, sequence * KV head, split), dispatched longest
// sequence first for varlen batches (longest_first_tile).  A producer warp
// streams 32-key chunks of K and V for its KV head through an NS-stage ring
// of 128B-swizzled shared-memory panels with TMA (cp.async.bulk.tensor), one
// mbarrier pair per stage.  NW consumer warps take chunks round-robin; each
// keeps its own online-softmax state (running max m, sum l, accumulator) in
// the exp2 domain, and the warps' states are merged at the end exactly like
// splits are merged by the combine kernel.  Lane layout for QK^T: four lanes
// per key (8 keys per step), each lane owning a fixed quarter of the head dim
// (chosen so the swizzled 16-byte reads of 8 lanes hit 8 distinct bank
// groups); the query rows stay in registers.  For PV each lane owns d_v/32
// output columns.
//
// flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference":
// split KV at one query row is where one split leaves the GPU idle
// ("Benchmarks" sweep).  The exp2 online softmax follows the same page's test
// log (exp2 in the softmax).
#pragma once

#include <cuda.h>
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_convert.cuh"
#include "fa_ptx.cuh"

namespace fa {

template <int DT, int DQK, int DV, int RT, int NW, int NS>
struct SimtCfg {
  static constexpr int ES = Elem<DT>::size;
  static constexpr int KC = 32;                         // keys per chunk
  static constexpr int PANEL_ELEMS = 128 / ES;          // elements per 128-byte row
  static constexpr int NPK = (DQK * ES + 127) / 128;    // K panels per chunk
  static constexpr int NPV = (DV * ES + 127) / 128;     // V panels per chunk
  static constexpr int PANEL = KC * 128;                // bytes per panel
  static constexpr int STAGE = (NPK + NPV) * PANEL;
  static constexpr int CPL = 2 * NPK;                   // 16-byte K chunks per lane per key
  static constexpr int EPC = 16 / ES;                   // elements per 16-byte chunk
  static constexpr int QR = CPL * EPC;                  // query values per lane per row
  static constexpr int DPL = DV / 32;                   // output columns per lane
  static constexpr int BPL = DV * ES / 32;              // V bytes per lane per key
  static constexpr int NTHREADS = (NW + 1) * 32;
  static constexpr int OFF_BAR = NS * STAGE;
  static constexpr int OFF_PS = OFF_BAR + 2 * NS * 8;
  static constexpr int OFF_MRG = OFF_PS + NW * RT * KC * 4;
  static constexpr int MRG_STRIDE = DV + 2;
  static constexpr int OFF_FLAG = OFF_MRG + NW * RT * MRG_STRIDE * 4;
  static constexpr int OFF_RANK = OFF_FLAG + 16;        // dispatch-order scratch
  static constexpr int SMEM = OFF_RANK + (kMaxRankedSeqs + 4) * 4 + 1024;  // + alignment slack
  static_assert(DV % 32 == 0, "d_v must be a multiple of 32");
  static_assert(BPL == 2 || BPL == 4 || BPL == 8 || BPL == 16, "unsupported V lane width");
  static_assert(RT <= NW, "one epilogue warp per row");
  // Chunk c uses stage c % NS and warp c % NW.  With NS a multiple of NW the
  // previous user of a stage (chunk c - NS) is the same warp, which has
  // already consumed it, so a parity wait can never match a phase two behind
  // (a different warp could still be waiting on that older load).
  static_assert(NS % NW == 0 && NS >= 2 * NW, "stages must be a multiple of the consumer warps");
  static_assert(NPV <= 4 && NPK <= 4, "head dim too large for this kernel");
};

template <int NBYTES>
__device__ __forceinline__ void lds_words(const uint8_t* p, uint32_t* w) {
  if constexpr (NBYTES == 16) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (NBYTES == 8) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  } else if constexpr (NBYTES == 4) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else {
    w[0] = *reinterpret_cast<const uint16_t*>(p);
  }
}

template <int DT, int DQK, int DV, int RT, int NW, int NS, bool ORDERED>
__global__ void __launch_bounds__((NW + 1) * 32)
    simt_splitkv_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV) {
  using C = SimtCfg<DT, DQK, DV, RT, NW, NS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_u32 + pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {  // descriptors fetched while the prologue runs
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  pdl_wait();  // the previous kernel in the stream is complete from here on
  int* rank_scratch = reinterpret_cast<int*>(smem + C::OFF_RANK);
  // The order is a compile-time choice: the kernel's decode loop is sensitive
  // to the code around it, and the grid-order variant keeps single-sequence
  // launches on the leanest code.
  const TileIdx tile = ORDERED ? longest_first_tile(p, rank_scratch, rank_scratch + kMaxRankedSeqs)
                               : grid_order_tile(p);
  const int m_blk = tile.m_blk;
  const int b = tile.b;
  const int kh = tile.kh;
  const int split = tile.split;

  // The sequence offsets are loaded before the error-word check so that both
  // reads share one memory latency.
  SeqInfo sq;
  const bool seq_ok = load_seq(p, b, sq);
  if (__syncthreads_or(timed_out_before(p.err))) return;
  if (!seq_ok) {
    if (threadIdx.x == 0) record_error(p.err, kErrDeviceArg);
    return;
  }
  const int rows = sq.lq * p.group;
  const int r0 = m_blk * RT;
  if (r0 >= rows) return;  // tile past this sequence's rows: nothing to write
  const int nrows = min(RT, rows - r0);
  const int i_lo = r0 / p.group;
  const int i_hi = (r0 + nrows - 1) / p.group;
  int k0, k1;
  tile_split_range(i_lo, i_hi, sq.lq, sq.lk, p.causal, p.window_left, p.num_splits, split, k0,
                   k1);
  const int key0 = load_base(p, k0, C::KC);  // first key of chunk 0
  const int nchunks = k1 > k0 ? (k1 - key0 + C::KC - 1) / C::KC : 0;

  const uint32_t bar_full = sbase + C::OFF_BAR;
  const uint32_t bar_empty = bar_full + NS * 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  float* mrg = reinterpret_cast<float*>(smem + C::OFF_MRG);
  int issued = 0;  // producer: chunks whose loads were issued

  if (warp == NW) {
    // ---------------------------------------------------------- producer
    if (lane == 0 && nchunks > 0) {
      const uint64_t pol = gridDim.x == 1 ? l2_policy_evict_first() : l2_policy_evict_last();
      PageCursor pages;
      for (int c = 0; c < nchunks; ++c) {
        const int st = c % NS;
        const int row = kv_row_walk(p, sq, b, key0 + c * C::KC, C::KC, pages);
        if (c >= NS && !mbar_wait(bar_empty + 8 * st, ((c / NS) - 1) & 1, p.err, abort_flag)) break;
        const uint32_t dst = sbase + st * C::STAGE;
        const uint32_t fb = bar_full + 8 * st;
        mbar_arrive_expect_tx(fb, C::STAGE);
#pragma unroll
        for (int pk = 0; pk < C::NPK; ++pk)
          tma_load_3d(dst + pk * C::PANEL, &tmK, fb, pk * C::PANEL_ELEMS, kh, row, pol);
#pragma unroll
        for (int pv = 0; pv < C::NPV; ++pv)
          tma_load_3d(dst + (C::NPK + pv) * C::PANEL, &tmV, fb, pv * C::PANEL_ELEMS, kh, row, pol);
        issued = c + 1;
      }
    }
  } else {
    // ---------------------------------------------------------- consumers
    const int kk = lane >> 2;   // key within an 8-key step (= swizzle row phase)
    const int sub = lane & 3;   // quarter of the head dim
    float qscale = p.scale * 1.4426950408889634f;
    if (DT == kE4M3) qscale *= __ldg(p.descale_q) * __ldg(p.descale_k);

    f32x2 qf[RT][C::QR / 2];  // query values of this lane's columns, in pairs
    int lo_r[RT], hi_r[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      lo_r[r] = 0;
      hi_r[r] = 0;
#pragma unroll
      for (int e = 0; e < C::QR / 2; ++e) qf[r][e] = 0ull;
      if (r < nrows) {
        const int R = r0 + r;
        const int i = R / p.group;
        const int h = kh * p.group + (R - i * p.group);
        const uint8_t* qrow = static_cast<const uint8_t*>(p.q) +
                              ((size_t)(sq.q0 + i) * p.h_q + h) * (size_t)DQK * C::ES;
#pragma unroll
        for (int t = 0; t < C::CPL; ++t) {
          const int pk = t >> 1, half = t & 1;
          const int pc = sub + 4 * ((half + kk) & 1);
          const int lc = pc ^ kk;
          const int dim0 = pk * C::PANEL_ELEMS + lc * C::EPC;
          if (dim0 < DQK) {
            uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow + (size_t)dim0 * C::ES));
            uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            float f[C::EPC];
            words_to_float<DT, 4>(w, f);
#pragma unroll
            for (int e = 0; e < C::EPC; e += 2)
              qf[r][(t * C::EPC + e) / 2] = f2_make(f[e] * qscale, f[e + 1] * qscale);
          }
        }
        int lo, hi;
        row_key_range(i, sq.lq, sq.lk, p.causal, p.window_left, lo, hi);
        lo_r[r] = max(lo, k0);
        hi_r[r] = min(hi, k1);
      }
    }

    float m_run[RT], l_run[RT];
    f32x2 acc[RT][C::DPL / 2];  // this lane's output columns, in pairs
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      m_run[r] = -CUDART_INF_F;
      l_run[r] = 0.f;
#pragma unroll
      for (int e = 0; e < C::DPL / 2; ++e) acc[r][e] = 0ull;
    }
    float* ps = reinterpret_cast<float*>(smem + C::OFF_PS) + warp * RT * C::KC;

    // V columns owned by this lane: logical bytes [lane*BPL, lane*BPL+BPL).
    const int vlb = lane * C::BPL;
    const int v_panel = vlb >> 7;
    const int v_lc = (vlb & 127) >> 4;
    const int v_off = vlb & 15;

    for (int c = warp; c < nchunks; c += NW) {
      const int st = c % NS;
      const bool ok = mbar_wait(bar_full + 8 * st, (c / NS) & 1, p.err, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;  // leave together: shuffles below need all lanes
      const uint8_t* kbase = smem + st * C::STAGE;
      const uint8_t* vbase = kbase + C::NPK * C::PANEL;
      const int key_base = key0 + c * C::KC;

      float sc[RT][4];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int krow = it * 8 + kk;
        f32x2 d2[RT];
#pragma unroll
        for (int r = 0; r < RT; ++r) d2[r] = 0ull;
#pragma unroll
        for (int t = 0; t < C::CPL; ++t) {
          const int pk = t >> 1, half = t & 1;
          const int pc = sub + 4 * ((half + kk) & 1);
          uint32_t w[4];
          lds_words<16>(kbase + pk * C::PANEL + krow * 128 + pc * 16, w);
          f32x2 kv[C::EPC / 2];
#pragma unroll
          for (int u = 0; u < 4; ++u) word_to_f2<DT>(w[u], kv + u * (C::EPC / 8));
#pragma unroll
          for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int e = 0; e < C::EPC / 2; ++e)
              d2[r] = f2_fma(qf[r][(t * C::EPC) / 2 + e], kv[e], d2[r]);
        }
        const int j = key_base + krow;
        float d[RT];
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          const float2 dd = f2_split(d2[r]);
          d[r] = dd.x + dd.y;
          d[r] += __shfl_xor_sync(0xffffffffu, d[r], 1);
          d[r] += __shfl_xor_sync(0xffffffffu, d[r], 2);
          sc[r][it] = (j >= lo_r[r] && j < hi_r[r]) ? d[r] : -CUDART_INF_F;
        }
      }

#pragma unroll
      for (int r = 0; r < RT; ++r) {
        float mx = fmaxf(fmaxf(sc[r][0], sc[r][1]), fmaxf(sc[r][2], sc[r][3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run[r], mx);
        float alpha = 1.f;
        float pv[4] = {0.f, 0.f, 0.f, 0.f};
        if (m_new != -CUDART_INF_F) {
          alpha = fast_exp2(m_run[r] - m_new);
#pragma unroll
          for (int it = 0; it < 4; ++it) pv[it] = fast_exp2(sc[r][it] - m_new);
        }
        m_run[r] = m_new;
        l_run[r] = l_run[r] * alpha + (sub == 0 ? (pv[0] + pv[1]) + (pv[2] + pv[3]) : 0.f);
        const f32x2 a2 = f2_make(alpha, alpha);
#pragma unroll
        for (int e = 0; e < C::DPL / 2; ++e) acc[r][e] = f2_mul(acc[r][e], a2);
        if (sub == 0) {
#pragma unroll
          for (int it = 0; it < 4; ++it) ps[r * C::KC + it * 8 + kk] = pv[it];
        }
      }
      __syncwarp();

#pragma unroll 2
      for (int key = 0; key < C::KC; key += 4) {
        float4 pr[RT];
#pragma unroll
        for (int r = 0; r < RT; ++r) pr[r] = *reinterpret_cast<const float4*>(ps + r * C::KC + key);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int vrow = key + u;
          uint32_t w[(C::BPL + 3) / 4];
          lds_words<C::BPL>(vbase + v_panel * C::PANEL + vrow * 128 + ((v_lc ^ (vrow & 7)) << 4) + v_off,
                            w);
          f32x2 vv[C::DPL / 2];
          if constexpr (C::BPL >= 4) {
#pragma unroll
            for (int u2 = 0; u2 < C::BPL / 4; ++u2) word_to_f2<DT>(w[u2], vv + u2 * (C::DPL / 2) / (C::BPL / 4));
          } else {
            // 2 bytes = two e4m3 values
            __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[0]), __NV_E4M3);
            float2 fv = __half22float2(*reinterpret_cast<__half2*>(&h2));
            vv[0] = f2_make(fv.x, fv.y);
          }
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const float pw = u == 0 ? pr[r].x : u == 1 ? pr[r].y : u == 2 ? pr[r].z : pr[r].w;
            const f32x2 pw2 = f2_make(pw, pw);
#pragma unroll
            for (int e = 0; e < C::DPL / 2; ++e) acc[r][e] = f2_fma(pw2, vv[e], acc[r][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }

    // Publish this warp's state for the CTA-level merge.
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      float l = l_run[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      float* dst = mrg + (warp * RT + r) * C::MRG_STRIDE;
      if (lane == 0) {
        dst[0] = m_run[r];
        dst[1] = l;
      }
#pragma unroll
      for (int e = 0; e < C::DPL / 2; ++e) {
        const float2 a = f2_split(acc[r][e]);
        dst[2 + lane * C::DPL + 2 * e] = a.x;
        dst[2 + lane * C::DPL + 2 * e + 1] = a.y;
      }
    }
  }
  __syncthreads();
  pdl_launch_dependents();

  // ------------------------------------------------------------ epilogue
  if (warp < nrows) {
    const int r = warp;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg[(w * RT + r) * C::MRG_STRIDE]);
    float L = 0.f;
    float o[C::DPL];
#pragma unroll
    for (int e = 0; e < C::DPL; ++e) o[e] = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float* src = mrg + (w * RT + r) * C::MRG_STRIDE;
        const float f = fast_exp2(src[0] - M);
        L += src[1] * f;
#pragma unroll
        for (int e = 0; e < C::DPL; ++e) o[e] = fmaf(src[2 + lane * C::DPL + e], f, o[e]);
      }
    }
    float lse_v = -CUDART_INF_F;
    if (M != -CUDART_INF_F && L > 0.f) {
      float inv = 1.f / L;
      if (DT == kE4M3) inv *= __ldg(p.descale_v);
#pragma unroll
      for (int e = 0; e < C::DPL; ++e) o[e] *= inv;
      lse_v = (M + __log2f(L)) * 0.69314718055994531f;
    } else {
#pragma unroll
      for (int e = 0; e < C::DPL; ++e) o[e] = 0.f;
    }
    const int R = r0 + r;
    const int i = R / p.group;
    const int h = kh * p.group + (R - i * p.group);
    const int t = sq.q0 + i;
    if (p.num_splits == 1) {
      const size_t oe = ((size_t)t * p.h_q + h) * DV + lane * C::DPL;
      if (o_ok(p, oe, C::DPL)) store_o<C::DPL>(p.out, oe, o, 1.f, p.out_dtype);
      if (p.lse != nullptr && lane == 0 && lse_ok(p, h, t)) p.lse[(size_t)h * p.total_q + t] = lse_v;
    } else {
      const size_t slot = (size_t)b * p.max_seqlen_q + i;
      const size_t row = ((size_t)split * p.slots + slot) * p.h_q + h;
      if (ws_o_ok(p, row * DV + lane * C::DPL, C::DPL)) {
        float* wo = p.ws_o + row * DV + lane * C::DPL;
#pragma unroll
        for (int e = 0; e < C::DPL; e += 2)
          *reinterpret_cast<float2*>(wo + e) = make_float2(o[e], o[e + 1]);
      }
      if (lane == 0 && ws_l_ok(p, row)) p.ws_l[row] = lse_v;
    }
  }

  // If a wait gave up, let the loads already issued land before the CTA exits.
  if (warp == NW && lane == 0 && *abort_flag) {
    for (int st = 0; st < NS && st < issued; ++st) {
      const int c_last = st + ((issued - 1 - st) / NS) * NS;
      mbar_wait(bar_full + 8 * st, (c_last / NS) & 1, nullptr, nullptr);
    }
  }
}

}  // namespace fa
