// Tensor-core split-KV partial kernel (tcgen05 + TMEM + TMA) for tiles with
// many query rows per KV head: short cached-prefix queries, GQA groups of
// eight or more, varlen prefill.
//
// flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference":
// the Blackwell MMA has M = 128 and a CTA holding one 128-row query tile
// (q_stage = 1) is what short-query split-KV needs; the GQA query rows of a
// KV head are packed into that tile (row r = query r / group, head r % group)
// so few queries still fill it.
//
// One CTA = one (128-row tile, sequence * KV head, split); 6 warps:
//   warp 0      TMA producer: Q tile once, then K and V tiles of 128 keys
//               through separate rings (KS deep for K, VS for V).  A K stage
//               is released as soon as its S MMA completes, so K runs ahead
//               of V: loads for block j+2 are in flight while block j's
//               softmax and PV run, which hides the L2/HBM latency;
//   warp 1      allocates 512 TMEM columns; lane 0 issues the MMAs:
//               S_j = Q K_j^T into one of two TMEM S buffers (ping-pong, so
//               S_{j+1} overlaps the softmax of S_j), then O += P_j V_j into
//               the TMEM O accumulator;
//   warps 2-5   one thread per query row (TMEM lane): load the S row, apply
//               the residual / bottom-right causal / window mask, online
//               softmax in the exp2 domain, rescale the O row in TMEM when
//               the running max moves, write P (bf16 / fp16 / e4m3) into
//               TMEM over the S columns it came from, and finally normalise O
//               and store it (or the fp32 split partial) with row-predicated
//               vector stores (cutlass "Adds variable sequence lengths to the
//               Hopper CuTe DSL FMHA example", "Implementation": rows past a
//               sequence are computed but never stored).
//
// Operand layouts (all 128B-swizzled, 1024-byte aligned, 128-byte rows):
//   Q  [128 rows][d_qk]  K-major A of S      K [128 keys][d_qk]  K-major B of S
//   P  [128 rows][128 keys] in TMEM, A of PV  V [128 keys][d_v]  MN-major B of PV
// each split into 128-byte-wide panels of 128 rows (16 KB).
#pragma once

#include <cuda.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_convert.cuh"
#include "fa_ptx.cuh"

namespace fa {

template <int DT, int DQK, int DV, int KS, int VS>
struct UmmaCfg {
  static constexpr int ES = Elem<DT>::size;
  static constexpr int PANEL_ELEMS = 128 / ES;
  static constexpr int PANEL = 128 * 128;                  // 128 rows x 128 bytes
  static constexpr int NPQ = (DQK * ES + 127) / 128;       // panels of Q / K
  static constexpr int NPV = (DV * ES + 127) / 128;        // panels of V
  // P stays in TMEM (over the S columns it came from) as the PV MMA's A
  // operand: 16-bit P two per column, e4m3 P four per column.
  static constexpr int UMMA_K = 32 / ES;                   // K elements per MMA
  static constexpr int KSTEPS_PER_PANEL = PANEL_ELEMS / UMMA_K;
  static constexpr int S_KSTEPS = (DQK + UMMA_K - 1) / UMMA_K;
  static constexpr int PV_KSTEPS = 128 / UMMA_K;
  static constexpr int TMEM_COLS = 512;
  static constexpr int TM_S0 = 0, TM_S1 = 128, TM_O = 256;
  static constexpr int OFF_Q = 0;
  static constexpr int K_STAGE = NPQ * PANEL;
  static constexpr int V_STAGE = NPV * PANEL;
  static constexpr int OFF_K = OFF_Q + NPQ * PANEL;
  static constexpr int OFF_V = OFF_K + KS * K_STAGE;
  static constexpr int OFF_BAR = OFF_V + VS * V_STAGE;
  // barriers: q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2],
  // p_ready, o_ready, drain
  static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 2 + 3;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_FLAG = OFF_TMEM_SLOT + 16;
  static constexpr int SMEM = OFF_FLAG + 16 + 1024;
  static constexpr int NTHREADS = 192;
  static constexpr uint32_t IDESC_S =
      mma_idesc(DT == kBF16 ? 1u : 0u, 128, 128, 0, 0);    // Q K^T: both K-major
  static constexpr uint32_t IDESC_PV =
      mma_idesc(DT == kBF16 ? 1u : 0u, 128, DV, 0, 1);     // P V: V is MN-major
  static_assert(DV <= 256 && DV % 16 == 0, "d_v");
  static_assert(TM_O + DV <= TMEM_COLS, "TMEM columns");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <int DT>
__device__ __forceinline__ void mma_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
  if constexpr (DT == kE4M3)
    tc_mma_f8(d, a, b, idesc, acc);
  else
    tc_mma_f16(d, a, b, idesc, acc);
}

// Lazy rescale threshold (log2 units): the running max used for the
// exponentials is only raised when a row's true max exceeds it by more
// than this, so O in TMEM is rarely rescaled.  With it a probability is at
// most 2^kThreshold; e4m3 P is scaled by kP8Scale = 2^(8 - 4) so that it
// stays within e4m3's range (448) while small values keep their leading bits.
template <int DT>
struct Lazy {
  static constexpr float kThreshold = DT == kE4M3 ? 4.f : 8.f;
};
constexpr float kP8Scale = 16.f;

template <int DT, int DQK, int DV, int KS, int VS>
__global__ void __launch_bounds__(192, 1)
    umma_splitkv_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV) {
  using C = UmmaCfg<DT, DQK, DV, KS, VS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_u32 + pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heaviest tiles first: with causal masks later query tiles see more keys.
  const TileIdx tile = query_tile_order(p);  // heaviest (latest) tiles first
  const int m_blk = tile.m_blk;
  const int b = tile.b;
  const int kh = tile.kh;
  const int split = tile.split;
  const int group = p.group;
  const int qpt = 128 / group;  // queries per tile

  if (threadIdx.x == 0) {  // descriptors fetched while the prologue runs
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  pdl_wait();  // the previous kernel in the stream is complete from here on
  // The sequence offsets are loaded before the error-word check so that both
  // reads share one memory latency.
  SeqInfo sq;
  const bool seq_ok = load_seq(p, b, sq);
  if (__syncthreads_or(timed_out_before(p.err))) return;
  if (!seq_ok) {
    if (threadIdx.x == 0) record_error(p.err, kErrDeviceArg);
    return;
  }
  const int q_start = m_blk * qpt;
  if (q_start >= sq.lq) return;  // tile past this sequence's queries
  const int nq = min(qpt, sq.lq - q_start);
  const int nrows = nq * group;
  int k0, k1;
  tile_split_range(q_start, q_start + nq - 1, sq.lq, sq.lk, p.causal, p.window_left, p.num_splits,
                   split, k0, k1);
  const int kb0 = load_base(p, k0, kBlockN);  // first key of block 0
  const int nblk = k1 > k0 ? (k1 - kb0 + kBlockN - 1) / kBlockN : 0;
  // TMA boxes per 128-key block: several when K/V pages are smaller than 128
  const int box_rows = (p.page_size > 0 && p.page_size < kBlockN) ? p.page_size : kBlockN;
  const int nsub = kBlockN / box_rows;

  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t q_full = bar0;
  const uint32_t k_full = bar0 + 8;                  // [KS]
  const uint32_t k_empty = k_full + 8 * KS;          // [KS]
  const uint32_t v_full = k_empty + 8 * KS;          // [VS]
  const uint32_t v_empty = v_full + 8 * VS;          // [VS]
  const uint32_t s_full = v_empty + 8 * VS;          // [2]
  const uint32_t p_ready = s_full + 16;
  const uint32_t o_ready = p_ready + 8;
  const uint32_t drain = o_ready + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(k_full + 8 * s, 1);
      mbar_init(k_empty + 8 * s, 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(v_full + 8 * s, 1);
      mbar_init(v_empty + 8 * s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_full + 8, 1);
    mbar_init(p_ready, 128);
    mbar_init(o_ready, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + C::OFF_TMEM_SLOT, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued_k = 0, issued_v = 0;  // producer: K / V blocks issued

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0 && nblk > 0) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = gridDim.x == 1 ? l2_policy_evict_first() : l2_policy_evict_last();
      mbar_arrive_expect_tx(q_full, C::NPQ * qpt * group * 128);
#pragma unroll
      for (int pq = 0; pq < C::NPQ; ++pq)
        tma_load_3d(sbase + C::OFF_Q + pq * C::PANEL, &tmQ, q_full, pq * C::PANEL_ELEMS,
                    kh * group, q_row_ok(p, sq.q0 + q_start) ? sq.q0 + q_start : 0, pol_q);
      // K(0), K(1), V(0), K(2), V(1), ...: K one block ahead of V.
      PageCursor pages_k, pages_v;
      for (int j = 0; j <= nblk; ++j) {
        if (j < nblk) {
          const int st = j % KS;
          int rows[kMaxSub];  // rows resolved before the wait, off the refill's critical path
#pragma unroll
          for (int sb = 0; sb < kMaxSub; ++sb)
            if (sb < nsub)
              rows[sb] = kv_row_walk(p, sq, b, kb0 + j * kBlockN + sb * box_rows, box_rows,
                                     pages_k);
          if (j >= KS && !mbar_wait(k_empty + 8 * st, ((j / KS) - 1) & 1, p.err, abort_flag)) break;
          const uint32_t dst = sbase + C::OFF_K + st * C::K_STAGE;
          mbar_arrive_expect_tx(k_full + 8 * st, C::K_STAGE);
#pragma unroll
          for (int sb = 0; sb < kMaxSub; ++sb)
            if (sb < nsub)
#pragma unroll
              for (int pk = 0; pk < C::NPQ; ++pk)
                tma_load_3d(dst + pk * C::PANEL + sb * box_rows * 128, &tmK, k_full + 8 * st,
                            pk * C::PANEL_ELEMS, kh, rows[sb], pol_kv);
          issued_k = j + 1;
        }
        if (j >= 1) {
          const int jv = j - 1;
          const int st = jv % VS;
          int rows[kMaxSub];  // rows resolved before the wait, off the refill's critical path
#pragma unroll
          for (int sb = 0; sb < kMaxSub; ++sb)
            if (sb < nsub)
              rows[sb] = kv_row_walk(p, sq, b, kb0 + jv * kBlockN + sb * box_rows, box_rows,
                                     pages_v);
          if (jv >= VS && !mbar_wait(v_empty + 8 * st, ((jv / VS) - 1) & 1, p.err, abort_flag)) break;
          const uint32_t dst = sbase + C::OFF_V + st * C::V_STAGE;
          mbar_arrive_expect_tx(v_full + 8 * st, C::V_STAGE);
#pragma unroll
          for (int sb = 0; sb < kMaxSub; ++sb)
            if (sb < nsub)
#pragma unroll
              for (int pv = 0; pv < C::NPV; ++pv)
                tma_load_3d(dst + pv * C::PANEL + sb * box_rows * 128, &tmV, v_full + 8 * st,
                            pv * C::PANEL_ELEMS, kh, rows[sb], pol_kv);
          issued_v = jv + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0 && nblk > 0) {
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag);
      const uint32_t q_addr = sbase + C::OFF_Q;
      auto issue_s = [&](int j) {
        const int st = j % KS;
        const uint32_t k_addr = sbase + C::OFF_K + st * C::K_STAGE;
        const uint32_t d = tmem + ((j & 1) ? C::TM_S1 : C::TM_S0);
#pragma unroll
        for (int ks = 0; ks < C::S_KSTEPS; ++ks) {
          const uint32_t off = (ks / C::KSTEPS_PER_PANEL) * C::PANEL + (ks % C::KSTEPS_PER_PANEL) * 32;
          mma_issue<DT>(d, smem_desc_sw128(q_addr + off, 16, 1024),
                        smem_desc_sw128(k_addr + off, 16, 1024), C::IDESC_S, ks > 0 ? 1u : 0u);
        }
        tc_commit(s_full + 8 * (j & 1));
        tc_commit(k_empty + 8 * st);
      };
      if (ok) ok = mbar_wait(k_full, 0, p.err, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < nblk; ++j) {
        const int st = j % VS;
        if (j + 1 < nblk) {
          const int st1 = (j + 1) % KS;
          ok = mbar_wait(k_full + 8 * st1, ((j + 1) / KS) & 1, p.err, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        ok = mbar_wait(p_ready, j & 1, p.err, abort_flag) &&
             mbar_wait(v_full + 8 * st, (j / VS) & 1, p.err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t v_addr = sbase + C::OFF_V + st * C::V_STAGE;
#pragma unroll
        for (int ks = 0; ks < C::PV_KSTEPS; ++ks) {
          const uint32_t b_off = ks * C::UMMA_K * 128;
          const uint64_t v_desc = smem_desc_sw128(v_addr + b_off, C::PANEL, 1024);
          const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
          const uint32_t a_t = tmem + ((j & 1) ? C::TM_S1 : C::TM_S0) + ks * 8;
          if constexpr (DT == kE4M3)
            tc_mma_f8_ts(tmem + C::TM_O, a_t, v_desc, C::IDESC_PV, acc);
          else
            tc_mma_f16_ts(tmem + C::TM_O, a_t, v_desc, C::IDESC_PV, acc);
        }
        tc_commit(o_ready);
        tc_commit(v_empty + 8 * st);
      }
      // Let every issued MMA finish before TMEM can be released.
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr, nullptr);
    }
  } else {
    // ----------------------------------------------------- softmax warps
    const int quarter = warp & 3;          // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;     // tile row = TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const bool row_ok = r < nrows;
    const bool warp_active = quarter * 32 < nrows;
    const int i = q_start + r / group;
    const int h = kh * group + (r - (r / group) * group);
    // Rows outside the tile (past the sequence's queries, or beyond the
    // group's heads) are never stored: they take an unbounded key range so
    // that they never ask for masking, keeping every warp on one path.
    int lo = -(1 << 30), hi = 1 << 30;
    if (row_ok) {
      row_key_range(i, sq.lq, sq.lk, p.causal, p.window_left, lo, hi);
      lo = max(lo, k0);
      hi = min(hi, k1);
    }
    float sl2 = p.scale * 1.4426950408889634f;
    if (DT == kE4M3) sl2 *= __ldg(p.descale_q) * __ldg(p.descale_k);
    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;

    for (int j = 0; j < nblk; ++j) {
      float s[128];
      float m_new = m_run;
      float alpha = 1.f, rsum = 0.f;
      if (warp_active) {
        ok = mbar_wait(s_full + 8 * (j & 1), (j >> 1) & 1, p.err, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        const uint32_t s_addr = tmem + lane_base + ((j & 1) ? C::TM_S1 : C::TM_S0);
        const int kb = kb0 + j * kBlockN;
        tmem_ld128(s_addr, reinterpret_cast<uint32_t*>(s));
        // Max of the raw scores (the scale is positive): eight independent
        // chains; keys outside [lo, hi) only exist in boundary blocks.
        float mx[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mx[t] = -CUDART_INF_F;
        // Masking is decided for the whole warp (a lane-divergent branch
        // here would split the warp for the rest of the block).
        if (__any_sync(0xffffffffu, !(kb >= lo && kb + kBlockN <= hi))) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int key = kb + c;
            s[c] = (key >= lo && key < hi) ? s[c] : -CUDART_INF_F;
          }
        }
        // three-input max: 8 chains over 16 values each
#pragma unroll
        for (int c = 0; c < 128; c += 16)
#pragma unroll
          for (int t = 0; t < 8; ++t) mx[t] = fmax3(mx[t], s[c + t], s[c + 8 + t]);
        const float bmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
        // Lazy rescale: keep the max in use unless the block's max exceeds
        // it by more than the threshold (probabilities then stay <= 2^thr).
        m_new = (bmax > m_run + Lazy<DT>::kThreshold) ? bmax : m_run;
        const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
        // alpha rescales what was accumulated so far; a row that has seen no
        // key yet holds O = 0 and l = 0, so it needs no rescale.
        alpha = m_run == m_new ? 1.f : fast_exp2(m_run - m_use);
        // e4m3 P is produced pre-scaled by kP8Scale = 2^4 (offset in the
        // exponent); the row sum is scaled back exactly.
        const float e_off = DT == kE4M3 ? m_use - 4.f : m_use;
        // exponent arguments and row sums on packed fp32 pairs
        const f32x2 sl2x2 = f2_make(sl2, sl2);
        const f32x2 noff = f2_make(-e_off, -e_off);
        f32x2 sm[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) sm[t] = 0ull;
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          const float2 x = f2_split(f2_fma(f2_make(s[c], s[c + 1]), sl2x2, noff));
          const float e0 = fast_exp2(x.x), e1 = fast_exp2(x.y);  // masked: exp2(-inf) = 0
          s[c] = e0;
          s[c + 1] = e1;
          sm[(c >> 1) & 3] = f2_add(sm[(c >> 1) & 3], f2_make(e0, e1));
        }
        const float2 r01 = f2_split(f2_add(f2_add(sm[0], sm[1]), f2_add(sm[2], sm[3])));
        rsum = r01.x + r01.y;
        if (DT == kE4M3) rsum *= 1.f / kP8Scale;
      }
      // PV of the previous block must be done before O is rescaled and the
      // P buffer is overwritten (the exponentials above overlap it).
      if (j > 0) {
        ok = mbar_wait(o_ready, (j - 1) & 1, p.err, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
      }
      if (warp_active) {
        const bool rescale = j > 0 && m_run != -CUDART_INF_F && alpha != 1.f;
        if (__any_sync(0xffffffffu, rescale)) {
          const uint32_t o_addr = tmem + lane_base + C::TM_O;
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(o_addr + 32 * c, o);
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
            tmem_st32(o_addr + 32 * c, o);
          }
          tmem_st_wait();
        }
        l_run = l_run * alpha + rsum;
        m_run = m_new;
        // P over the first 64 columns of this block's S buffer (already read):
        // column c holds keys 2c (low half) and 2c+1.
        const uint32_t p_addr_t = tmem + lane_base + ((j & 1) ? C::TM_S1 : C::TM_S0);
        if constexpr (DT == kE4M3) {
          // e4m3: probabilities were produced pre-scaled by kP8Scale
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(s[4 * c], s[4 * c + 1]), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(s[4 * c + 2], s[4 * c + 3]), __NV_SATFINITE, __NV_E4M3);
            pk[c] = (uint32_t)lo | ((uint32_t)hi << 16);
          }
          tmem_st32(p_addr_t, pk);
        } else {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = pack2(s[64 * h2 + 2 * c], s[64 * h2 + 2 * c + 1], DT);
            tmem_st32(p_addr_t + 32 * h2, pk);
          }
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(p_ready);
    }

    // ------------------------------------------------------------ epilogue
    pdl_launch_dependents();
    if (ok && nblk > 0) {
      ok = mbar_wait(o_ready, (nblk - 1) & 1, p.err, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (warp_active && ok) {
      float inv = 0.f, lse_v = -CUDART_INF_F;
      if (row_ok && l_run > 0.f && m_run != -CUDART_INF_F) {
        inv = 1.f / l_run;
        if (DT == kE4M3) inv *= __ldg(p.descale_v) * (1.f / kP8Scale);
        lse_v = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      }
      const int t = sq.q0 + i;
      const uint32_t o_addr = tmem + lane_base + C::TM_O;
      const bool ws_wide = (reinterpret_cast<uintptr_t>(p.ws_o) & 31u) == 0;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        if (nblk > 0) {
          tmem_ld32(o_addr + 32 * c, o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (!row_ok) continue;
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(o[e]) * inv;
        if (p.num_splits == 1) {
          const size_t oe = ((size_t)t * p.h_q + h) * DV + c * 32;
          if (o_ok(p, oe, 32)) store_o<32>(p.out, oe, f, 1.f, p.out_dtype);
        } else {
          const size_t slot = (size_t)b * p.max_seqlen_q + i;
          const size_t we = (((size_t)split * p.slots + slot) * p.h_q + h) * DV + c * 32;
          if (ws_o_ok(p, we, 32)) {
            // whole 32-byte sectors when the workspace allows it (each
            // thread writes its own row, so a store touches 32 rows)
            if (ws_wide) {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                st_global_32B(p.ws_o + we + 8 * e, reinterpret_cast<const uint32_t*>(f + 8 * e));
            } else {
              float4* dst = reinterpret_cast<float4*>(p.ws_o + we);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
            }
          }
        }
      }
      if (row_ok) {
        if (p.num_splits == 1) {
          if (p.lse != nullptr && lse_ok(p, h, t)) p.lse[(size_t)h * p.total_q + t] = lse_v;
        } else {
          const size_t slot = (size_t)b * p.max_seqlen_q + i;
          const size_t wl = ((size_t)split * p.slots + slot) * p.h_q + h;
          if (ws_l_ok(p, wl)) p.ws_l[wl] = lse_v;
        }
      }
    }
  }

  // ------------------------------------------------------------- teardown
  if (warp == 0 && lane == 0 && *abort_flag) {
    // let issued loads land before the CTA's shared memory is released
    for (int st = 0; st < KS && st < issued_k; ++st) {
      const int j_last = st + ((issued_k - 1 - st) / KS) * KS;
      mbar_wait(k_full + 8 * st, (j_last / KS) & 1, nullptr, nullptr);
    }
    for (int st = 0; st < VS && st < issued_v; ++st) {
      const int j_last = st + ((issued_v - 1 - st) / VS) * VS;
      mbar_wait(v_full + 8 * st, (j_last / VS) & 1, nullptr, nullptr);
    }
    if (nblk > 0) mbar_wait(q_full, 0, nullptr, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fa
