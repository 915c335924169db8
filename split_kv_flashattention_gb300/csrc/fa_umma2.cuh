// Tensor-core split kernel with two 128-row query tiles per CTA (256 rows),
// for prefill-sized tiles.
//
// flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference",
// description: a CTA tile of 256 query rows is two parallel M = 128 tensor
// core pipelines; the review asks whether softmax and MMA overlap.  Here
// they do: the two tiles (A, B) share every K/V block, and the MMA warp
// alternates between them so that while one tile's softmax runs, the tensor
// core works on the other tile:
//
//   S_A(0) S_B(0) | PV_A(0) S_A(1) PV_B(0) S_B(1) | PV_A(1) S_A(2) ...
//
// Warps (384 threads, three warpgroups): 0 TMA producer; 1 TMEM allocator +
// MMA issuer; 2-3 idle; 4-7 softmax of tile A; 8-11 softmax of tile B (one
// thread per row = TMEM lane; warp w reads TMEM lanes 32*(w%4) ..
// 32*(w%4)+31).  setmaxnreg moves registers from the first warpgroup to the
// softmax warpgroups, which keep a whole 128-column S row in registers.  TMEM (512 columns): S_A, S_B (128 each), O_A, O_B
// (d_v each).  P is written back over the S columns it came from as packed
// 16-bit pairs and the PV MMA reads its A operand from TMEM, so shared memory
// only holds the two Q tiles and the K/V ring.  Issue order on the MMA warp
// guarantees PV_A(j) reads P_A(j) before S_A(j+1) overwrites those columns,
// and the commit that signals S_A(j+1) also covers PV_A(j), so the softmax
// of block j+1 sees O_A final for block j and can rescale it.
#pragma once

#include <cuda.h>
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_convert.cuh"
#include "fa_ptx.cuh"

namespace fa {

// Non-blocking test of an mbarrier phase (no suspension).  A test or wait
// on a phase that has completed still takes about 70 cycles; several tests
// issued back to back overlap those latencies, where the same number of
// waits in a row would add them up on the MMA thread's path.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The shared-memory descriptor of fa_ptx.cuh (smem_desc_sw128) in two words.  For fixed offsets only the low word
// (start address and leading byte offset) depends on the address, so an
// issue loop keeps the high word in one register and steps the low word:
// desc(saddr + off) = desc(saddr) + off / 16 while saddr + off < 256 KB.
__host__ __device__ constexpr uint32_t smem_desc_sw128_hi(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint32_t smem_desc_sw128_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint64_t smem_desc_join(uint32_t lo, uint32_t hi) {
  return ((uint64_t)hi << 32) | lo;
}


// Whether the two softmax warpgroups strictly alternate (measured slower on
// GB300 than letting both run: each tile's softmax then has only one warp
// per SM sub-partition to hide latency with).
constexpr bool kPingPong = false;

template <int DT, int DQK, int DV, int KS, int VS>
struct Umma2Cfg {
  static_assert(DT != kE4M3, "two-tile kernel is for 16-bit inputs");
  static constexpr int ES = 2;
  static constexpr int PANEL_ELEMS = 64;
  static constexpr int PANEL = 128 * 128;
  static constexpr int NPQ = (DQK * ES + 127) / 128;
  static constexpr int NPV = (DV * ES + 127) / 128;
  static constexpr int UMMA_K = 16;
  static constexpr int KSTEPS_PER_PANEL = 4;
  static constexpr int S_KSTEPS = DQK / UMMA_K;
  static constexpr int PV_KSTEPS = 128 / UMMA_K;
  static constexpr int TMEM_COLS = 512;
  // TMEM columns of tile t's S/P and O
  __device__ static constexpr int tm_s(int t) { return 128 * t; }
  __device__ static constexpr int tm_o(int t) { return 256 + DV * t; }
  static constexpr int OFF_Q = 0;  // tile A panels, then tile B panels
  static constexpr int K_STAGE = NPQ * PANEL;
  static constexpr int V_STAGE = NPV * PANEL;
  static constexpr int OFF_K = OFF_Q + 2 * NPQ * PANEL;
  static constexpr int OFF_V = OFF_K + KS * K_STAGE;
  static constexpr int OFF_BAR = OFF_V + VS * V_STAGE;
  // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2], p_ready[2],
  // o_done[2], drain, turn[2]
  static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 2 + 2 + 2 + 1 + 2;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_FLAG = OFF_TMEM_SLOT + 16;
  static constexpr int SMEM = OFF_FLAG + 16 + 1024;
  static constexpr int NTHREADS = 384;
  // Register split (launch: 384 x 168 = 64512): the TMA/MMA warpgroup gives
  // registers to the two softmax warpgroups, 128*56 + 256*224 = 64512.
  static constexpr int REGS_CTRL = 56;
  static constexpr int REGS_SOFTMAX = 224;
  static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX <= 384 * 168, "register split");
  static constexpr uint32_t IDESC_S = mma_idesc(DT == kBF16 ? 1u : 0u, 128, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = mma_idesc(DT == kBF16 ? 1u : 0u, 128, DV, 0, 1);
  static_assert(256 + 2 * DV <= TMEM_COLS, "TMEM columns");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <int DT, int DQK, int DV, int KS, int VS>
__global__ void __launch_bounds__(384, 1)
    umma2_splitkv_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV) {
  using C = Umma2Cfg<DT, DQK, DV, KS, VS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_u32 + pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const TileIdx tile = query_tile_order(p);  // heaviest (latest) tiles first
  const int m_blk = tile.m_blk;
  const int b = tile.b;
  const int kh = tile.kh;
  const int split = tile.split;
  const int group = p.group;
  const int qpt = 128 / group;

  pdl_wait();  // the previous kernel in the stream is complete from here on
  if (__syncthreads_or(timed_out_before(p.err))) return;
  SeqInfo sq;
  if (!load_seq(p, b, sq)) {
    if (threadIdx.x == 0) record_error(p.err, kErrDeviceArg);
    return;
  }
  const int q_start = m_blk * 2 * qpt;
  if (q_start >= sq.lq) return;
  const int nq_a = min(qpt, sq.lq - q_start);
  const int nq_b = max(0, min(qpt, sq.lq - q_start - qpt));
  const bool has_b = nq_b > 0;
  int k0, k1;
  tile_split_range(q_start, q_start + nq_a + nq_b - 1, sq.lq, sq.lk, p.causal, p.window_left,
                   p.num_splits, split, k0, k1);
  const int kb0 = load_base(p, k0, kBlockN);  // first key of block 0
  const int nblk = k1 > k0 ? (k1 - kb0 + kBlockN - 1) / kBlockN : 0;
  // TMA boxes per 128-key block: several when K/V pages are smaller than 128
  const int box_rows = (p.page_size > 0 && p.page_size < kBlockN) ? p.page_size : kBlockN;
  const int nsub = kBlockN / box_rows;

  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t q_full = bar0;
  const uint32_t k_full = bar0 + 8;               // [KS]
  const uint32_t k_empty = k_full + 8 * KS;        // [KS]
  const uint32_t v_full = k_empty + 8 * KS;        // [VS]
  const uint32_t v_empty = v_full + 8 * VS;        // [VS]
  const uint32_t s_full = v_empty + 8 * VS;        // [2]
  const uint32_t p_ready = s_full + 16;           // [2]
  const uint32_t o_done = p_ready + 16;           // [2]
  const uint32_t drain = o_done + 16;
  const uint32_t turn = drain + 8;                // [2]: softmax ping-pong
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
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full + 8 * t, 1);
      mbar_init(p_ready + 8 * t, 128);
      mbar_init(o_done + 8 * t, 1);
    }
    mbar_init(drain, 1);
    mbar_init(turn, 128);
    mbar_init(turn + 8, 128);
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
  // The two register budgets never meet again: each side runs its own
  // teardown (CTA barrier, then the TMEM release on the MMA warp).
  if (warp < 4) {
    regs_dec<C::REGS_CTRL>();
  int issued_k = 0, issued_v = 0;

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0 && nblk > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      const int ntiles = has_b ? 2 : 1;
      mbar_arrive_expect_tx(q_full, ntiles * C::NPQ * qpt * group * 128);
      for (int t = 0; t < ntiles; ++t)
#pragma unroll
        for (int pq = 0; pq < C::NPQ; ++pq)
          tma_load_3d(sbase + C::OFF_Q + (t * C::NPQ + pq) * C::PANEL, &tmQ, q_full,
                      pq * C::PANEL_ELEMS, kh * group,
                      q_row_ok(p, sq.q0 + q_start + t * qpt) ? sq.q0 + q_start + t * qpt : 0,
                      pol_q);
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
      // The CTA this SM most likely runs next (CTAs are dispatched in linear
      // block order, one per SM): its Q and first K/V block into L2, so its
      // prologue does not wait on DRAM for them.
      if (p.num_sms > 0 && p.page_size <= 0) {
        const long long lin =
            blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
        const long long nxt = lin + p.num_sms;
        if (nxt < (long long)gridDim.x * gridDim.y * gridDim.z) {
          const int x2 = (int)(nxt % gridDim.x);
          const long long r2 = nxt / gridDim.x;
          const TileIdx t2 = query_tile_order_at(p, x2, (int)(r2 % gridDim.y), (int)(r2 / gridDim.y));
          SeqInfo s2;
          const int qs2 = t2.m_blk * 2 * qpt;
          if (load_seq(p, t2.b, s2) && qs2 < s2.lq) {
            const int nq2 = min(2 * qpt, s2.lq - qs2);
            for (int t = 0; t * qpt < nq2; ++t)
#pragma unroll
              for (int pq = 0; pq < C::NPQ; ++pq)
                tma_prefetch_l2_3d(&tmQ, pq * C::PANEL_ELEMS, t2.kh * group, s2.q0 + qs2 + t * qpt);
            int a0, a1;
            tile_split_range(qs2, qs2 + nq2 - 1, s2.lq, s2.lk, p.causal, p.window_left,
                             p.num_splits, t2.split, a0, a1);
            if (a1 > a0) {
#pragma unroll
              for (int pk = 0; pk < C::NPQ; ++pk)
                tma_prefetch_l2_3d(&tmK, pk * C::PANEL_ELEMS, t2.kh, s2.k0 + a0);
#pragma unroll
              for (int pv = 0; pv < C::NPV; ++pv)
                tma_prefetch_l2_3d(&tmV, pv * C::PANEL_ELEMS, t2.kh, s2.k0 + a0);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0 && nblk > 0) {
      const int ntiles = has_b ? 2 : 1;
      // Descriptors: the high word is a constant, a k-step adds to the low
      // word (fewer instructions per MMA for the one issuing thread).
      constexpr uint32_t kHi = smem_desc_sw128_hi(1024);
      auto issue_s = [&](int t, int j) {
        const uint32_t qd = smem_desc_sw128_lo(sbase + C::OFF_Q + t * C::NPQ * C::PANEL, 16);
        const uint32_t kd = smem_desc_sw128_lo(sbase + C::OFF_K + (j % KS) * C::K_STAGE, 16);
#pragma unroll
        for (int ks = 0; ks < C::S_KSTEPS; ++ks) {
          const uint32_t off =
              ((ks / C::KSTEPS_PER_PANEL) * C::PANEL + (ks % C::KSTEPS_PER_PANEL) * 32) >> 4;
          tc_mma_f16(tmem + C::tm_s(t), smem_desc_join(qd + off, kHi), smem_desc_join(kd + off, kHi),
                     C::IDESC_S, ks > 0 ? 1u : 0u);
        }
        tc_commit(s_full + 8 * t);
      };
      auto issue_pv = [&](int t, int j) {
        const uint32_t vd = smem_desc_sw128_lo(sbase + C::OFF_V + (j % VS) * C::V_STAGE, C::PANEL);
#pragma unroll
        for (int ks = 0; ks < C::PV_KSTEPS; ++ks)
          tc_mma_f16_ts(tmem + C::tm_o(t), tmem + C::tm_s(t) + ks * 8,
                        smem_desc_join(vd + ((ks * C::UMMA_K * 128) >> 4), kHi), C::IDESC_PV,
                        (j > 0 || ks > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag) && mbar_wait(k_full, 0, p.err, abort_flag);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < ntiles; ++t) issue_s(t, 0);
        tc_commit(k_empty);  // K(0) is free once both S(0) are done
      }
      for (int j = 0; ok && j < nblk; ++j) {
        for (int t = 0; t < ntiles; ++t) {
          // slot A's P, V(j) and K(j+1) tested together first (their
          // latencies overlap); waited for one by one only when one is not
          // complete
          bool ready = false;
          if (t == 0)
            ready = mbar_test_wait(p_ready, j & 1) &
                    mbar_test_wait(v_full + 8 * (j % VS), (j / VS) & 1) &
                    (j + 1 >= nblk ||
                     mbar_test_wait(k_full + 8 * ((j + 1) % KS), ((j + 1) / KS) & 1));
          if (!ready) {
            ok = mbar_wait(p_ready + 8 * t, j & 1, p.err, abort_flag);
            if (ok && t == 0)
              ok = mbar_wait(v_full + 8 * (j % VS), (j / VS) & 1, p.err, abort_flag);
            if (ok && t == 0 && j + 1 < nblk)
              ok = mbar_wait(k_full + 8 * ((j + 1) % KS), ((j + 1) / KS) & 1, p.err, abort_flag);
          }
          if (!ok) break;
          tc_fence_after();
          issue_pv(t, j);
          if (j + 1 < nblk)
            issue_s(t, j + 1);
          else
            tc_commit(o_done + 8 * t);
        }
        if (!ok) break;
        tc_commit(v_empty + 8 * (j % VS));
        if (j + 1 < nblk) tc_commit(k_empty + 8 * ((j + 1) % KS));
      }
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr, nullptr);
    }
  }
  // ----------------------------------------------------- teardown (TMA/MMA side)
  if (warp == 0 && lane == 0 && *abort_flag) {
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
  } else {
    regs_inc<C::REGS_SOFTMAX>();
    // ----------------------------------------------------- softmax warps
    const int t = (warp - 4) >> 2;        // tile 0 (A): warps 4-7, tile 1 (B): warps 8-11
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int nq = t == 0 ? nq_a : nq_b;
    const int nrows = nq * group;
    const bool tile_on = nq > 0;
    const bool warp_active = quarter * 32 < nrows;
    const bool row_ok = r < nrows;
    const int i = q_start + t * qpt + r / group;
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
    const float sl2 = p.scale * 1.4426950408889634f;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    const uint32_t s_addr = tmem + lane_base + C::tm_s(t);
    const uint32_t o_addr = tmem + lane_base + C::tm_o(t);
    bool ok = true;

    for (int j = 0; tile_on && j < nblk; ++j) {
      if (kPingPong && has_b && (t == 1 || j > 0)) {
        ok = mbar_wait(turn + 8 * t, (t == 1 ? j : j - 1) & 1, p.err, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      ok = mbar_wait(s_full + 8 * t, j & 1, p.err, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      if (warp_active) {
        const int kb = kb0 + j * kBlockN;
        float s[128];
        tmem_ld128(s_addr, reinterpret_cast<uint32_t*>(s));
        // Masking is decided for the whole warp (a lane-divergent branch
        // here would split the warp for the rest of the block).
        if (__any_sync(0xffffffffu, !(kb >= lo && kb + kBlockN <= hi))) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int key = kb + c;
            s[c] = (key >= lo && key < hi) ? s[c] : -CUDART_INF_F;
          }
        }
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 128; c += 16)
#pragma unroll
          for (int u = 0; u < 8; ++u) mx[u] = fmax3(mx[u], s[c + u], s[c + 8 + u]);
        const float bmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
        const float m_new = (bmax > m_run + 8.f) ? bmax : m_run;  // lazy rescale, 2^8
        const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
        const float alpha = m_run == m_new ? 1.f : fast_exp2(m_run - m_use);
        const bool rescale = j > 0 && m_run != -CUDART_INF_F && alpha != 1.f;
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds block j-1's result: the S(j) commit covered PV(j-1).
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(o_addr + 32 * c, o);
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            tmem_st32(o_addr + 32 * c, o);
          }
        }
        const f32x2 sl2x2 = f2_make(sl2, sl2);
        const f32x2 noff = f2_make(-m_use, -m_use);
        f32x2 sm[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) sm[u] = 0ull;
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          const float2 x = f2_split(f2_fma(f2_make(s[c], s[c + 1]), sl2x2, noff));
          const float e0 = fast_exp2(x.x), e1 = fast_exp2(x.y);
          s[c] = e0;
          s[c + 1] = e1;
          sm[(c >> 1) & 3] = f2_add(sm[(c >> 1) & 3], f2_make(e0, e1));
        }
        // P over the first 64 columns of this tile's S buffer (already read)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = pack2(s[64 * h2 + 2 * c], s[64 * h2 + 2 * c + 1], DT);
          tmem_st32(s_addr + 32 * h2, pk);
        }
        tmem_st_wait();
        const float2 r01 = f2_split(f2_add(f2_add(sm[0], sm[1]), f2_add(sm[2], sm[3])));
        l_run = l_run * alpha + (r01.x + r01.y);
        m_run = m_new;
      }
      tc_fence_before();
      mbar_arrive(p_ready + 8 * t);
      if (kPingPong && has_b) mbar_arrive(turn + 8 * (1 - t));
    }

    // ------------------------------------------------------------ epilogue
    pdl_launch_dependents();
    if (tile_on && ok && nblk > 0) {
      ok = mbar_wait(o_done + 8 * t, 0, p.err, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (tile_on && warp_active && ok) {
      float inv = 0.f, lse_v = -CUDART_INF_F;
      if (row_ok && l_run > 0.f && m_run != -CUDART_INF_F) {
        inv = 1.f / l_run;
        lse_v = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      }
      const int tok = sq.q0 + i;
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
          const size_t oe = ((size_t)tok * p.h_q + h) * DV + c * 32;
          if (o_ok(p, oe, 32)) store_o<32>(p.out, oe, f, 1.f, p.out_dtype);
        } else {
          const size_t slot = (size_t)b * p.max_seqlen_q + i;
          const size_t we = (((size_t)split * p.slots + slot) * p.h_q + h) * DV + c * 32;
          if (ws_o_ok(p, we, 32)) {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + we);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
          }
        }
      }
      if (row_ok) {
        if (p.num_splits == 1) {
          if (p.lse != nullptr && lse_ok(p, h, tok)) p.lse[(size_t)h * p.total_q + tok] = lse_v;
        } else {
          const size_t slot = (size_t)b * p.max_seqlen_q + i;
          const size_t wl = ((size_t)split * p.slots + slot) * p.h_q + h;
          if (ws_l_ok(p, wl)) p.ws_l[wl] = lse_v;
        }
      }
    }

    // teardown (softmax side): the TMEM release waits for these warps
    tc_fence_before();
    __syncthreads();
  }
}

}  // namespace fa
