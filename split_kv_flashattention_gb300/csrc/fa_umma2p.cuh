// Persistent form of the two-tile tensor-core kernel, for one-split prefill.
//
// The non-persistent kernel pays, per 256-row query tile pair, a prologue
// (offsets, barriers, TMEM allocation, then the latency of Q and the first K
// block) and an epilogue (O out of TMEM) during which the tensor core idles;
// across a varlen prefill that was about a seventh of each CTA's life.  Here
// one CTA per SM walks a list of tiles: the next tile's Q and K/V are loaded
// while the current tile's last blocks and epilogue run, and the TMEM
// allocation, barriers and descriptors are set up once.
//
// cutlass "Adds variable sequence lengths to the Hopper CuTe DSL FMHA
// example", section "Performance (GH200)": a persistent kernel that assigns
// the max-length grid round-robin balances skewed lengths poorly, and a
// length-aware schedule is the named follow-up.  This one first compacts the
// tiles that exist (sequence, 256-row query pair) into a list ordered
// longest first -- by key count without a mask, by query-pair index (the
// causal work) with one.  Each CTA starts on the tile of its own index and
// claims every later one from a ticket counter in global memory once the
// current tile's loads are all issued: the list goes out greedily, longest
// first, to whichever CTA is free, and no CTA holds a tile it will not start
// for a while.  The producer hands each decoded tile to the MMA and softmax
// roles through a small ring in shared memory (full/empty barriers; b < 0
// ends the walk).
//
// Per tile everything is as in the two-tile kernel (fa_umma2.cuh): two
// 128-row query tiles A and B share each K/V block, the MMA warp alternates
// PV_A(j) S_A(j+1) PV_B(j) S_B(j+1), and the softmax warpgroups run the same
// block body.  Across tiles the K/V rings, the S buffers and every barrier
// keep running phase counts; two barriers are added: q_empty (the MMA warp's
// commit after a tile's last S MMAs, so the producer may load the next Q) and
// o_free[t] (the softmax warps' arrival once they have read a tile's O out of
// TMEM, so the next tile's first PV may overwrite it).  At a tile's last
// block the MMA warp issues the next tile's S(0) into each slot right behind
// that slot's last PV, so the softmax warps find it ready when their
// epilogue ends.
#pragma once

#include <cuda.h>
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_convert.cuh"
#include "fa_ptx.cuh"
#include "fa_umma2.cuh"

namespace fa {

template <int DT, int DQK, int DV, int KS, int VS>
struct Umma2pCfg {
  using B = Umma2Cfg<DT, DQK, DV, KS, VS>;
  // Shared layout of the two-tile kernel, then: q_empty, o_free[2], the
  // tile ring's full/empty barriers and slots, the unit count and the unit
  // list (b | m << 7, uint16).
  static constexpr int OFF_BAR2 = B::OFF_FLAG + 16;
  static constexpr int OFF_TRING_BAR = OFF_BAR2 + 24;               // full[R], empty[R]
  static constexpr int OFF_TRING = OFF_TRING_BAR + 16 * kTileRing;  // decoded tiles [R]
  static constexpr int TRING_SLOT = 64;
  static constexpr int OFF_NUNITS = OFF_TRING + TRING_SLOT * kTileRing;
  static constexpr int OFF_UNITS = OFF_NUNITS + 8;
  static constexpr int SMEM = OFF_UNITS + 2 * kMaxUnits + 1024;
  // Register split (launch: 384 x 168): the producer and MMA roles carry the
  // tile walk (72 per thread), the softmax warpgroups keep a whole S row
  // (216): 128*72 + 256*216 = 64512.
  static constexpr int REGS_CTRL = 72;
  static constexpr int REGS_SOFTMAX = 216;
  static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX <= 384 * 168, "register split");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  // Scratch for building the list (the K ring, before any load).
  static constexpr int OFF_SCRATCH = B::OFF_K;
  static_assert(KS * B::K_STAGE >= 4 * 129 * 4, "list scratch");
};

// The tile a claim from the ticket counter stands for, or -1 once the list is
// exhausted.  Tiles 0..G-1 are every CTA's first (its own index, no claim);
// ticket t of the counter is tile G + t, so tiles go out in list order to
// whichever CTA asks first.
__device__ __forceinline__ int ticket_tile(int ticket, int n_tiles) {
  const int r = (int)gridDim.x + ticket;
  return r < n_tiles ? r : -1;
}

// Everything about one tile that every role needs, computed the same way by
// each of them.
struct PTile {
  int b, kh, m_blk;  // b < 0: the end of the walk
  SeqInfo sq;
  int q_start, nq_a, nq_b;
  int k0, k1, kb0, nblk;
};
static_assert(sizeof(PTile) <= 64, "tile ring slot");

// Tile r of the walk: KV heads in groups of p.kv_head_group; within a group
// the unit list in order, the group's heads innermost.  One group (all
// heads) without a mask; under a mask the host sizes a group so that its K/V
// stays in L2 while the m-major list revisits each sequence's key prefix.
__device__ __forceinline__ void decode_ptile(const FwdParams& p, const uint16_t* units, int r,
                                             int n_units, int qpt, PTile& t) {
  const int hg = p.kv_head_group;
  const int per_group = n_units * hg;
  const int g = r / per_group;
  const int rem = r - g * per_group;
  const int u = units[rem / hg];
  t.kh = g * hg + (rem - (rem / hg) * hg);
  t.b = u & 127;
  t.m_blk = u >> 7;
  load_seq(p, t.b, t.sq);  // validated when the list was built
  t.q_start = t.m_blk * 2 * qpt;
  t.nq_a = min(qpt, t.sq.lq - t.q_start);
  t.nq_b = max(0, min(qpt, t.sq.lq - t.q_start - qpt));
  tile_split_range(t.q_start, t.q_start + t.nq_a + t.nq_b - 1, t.sq.lq, t.sq.lk, p.causal,
                   p.window_left, 1, 0, t.k0, t.k1);
  t.kb0 = t.k0;
  t.nblk = t.k1 > t.k0 ? (t.k1 - t.kb0 + kBlockN - 1) / kBlockN : 0;
}

// MASKED: instantiated for calls with a causal or window mask.
template <int DT, int DQK, int DV, int KS, int VS, bool MASKED>
__global__ void __launch_bounds__(384, 1)
    umma2p_splitkv_kernel(const __grid_constant__ FwdParams p,
                          const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV) {
  using C = Umma2Cfg<DT, DQK, DV, KS, VS>;
  using CP = Umma2pCfg<DT, DQK, DV, KS, VS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_u32 + pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int group = p.group;
  const int qpt = 128 / group;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  pdl_wait();  // the previous kernel in the stream is complete from here on
  if (__syncthreads_or(timed_out_before(p.err))) return;

  // Barriers (thread 0) and TMEM (warp 1) first: they do not depend on the
  // tile list, and their latency then hides behind the cu_seqlens loads that
  // warps 4-11 make for the list.
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t q_full = bar0;
  const uint32_t k_full = bar0 + 8;                // [KS]
  const uint32_t k_empty = k_full + 8 * KS;         // [KS]
  const uint32_t v_full = k_empty + 8 * KS;         // [VS]
  const uint32_t v_empty = v_full + 8 * VS;         // [VS]
  const uint32_t s_full = v_empty + 8 * VS;         // [2]
  const uint32_t p_ready = s_full + 16;            // [2]
  const uint32_t o_done = p_ready + 16;            // [2]
  const uint32_t drain = o_done + 16;
  const uint32_t q_empty = sbase + CP::OFF_BAR2;
  const uint32_t o_free = q_empty + 8;              // [2]
  const uint32_t tr_full = sbase + CP::OFF_TRING_BAR;  // [kTileRing]
  const uint32_t tr_empty = tr_full + 8 * kTileRing;    // [kTileRing]
  PTile* tring = reinterpret_cast<PTile*>(smem + CP::OFF_TRING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
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
      mbar_init(o_free + 8 * t, 128);
    }
    // a tile slot is released by the MMA thread and the eight softmax warps
    for (int s = 0; s < kTileRing; ++s) {
      mbar_init(tr_full + 8 * s, 1);
      mbar_init(tr_empty + 8 * s, 9);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + C::OFF_TMEM_SLOT, C::TMEM_COLS);
    tmem_relinquish();
  }

  // ---- the tile list: units (sequence, query pair) that exist, longest first
  uint16_t* units = reinterpret_cast<uint16_t*>(smem + CP::OFF_UNITS);
  int* n_units_s = reinterpret_cast<int*>(smem + CP::OFF_NUNITS);
  {
    int* s_pairs = reinterpret_cast<int*>(smem + CP::OFF_SCRATCH);  // [128]
    int* s_keys = s_pairs + 128;                                     // [128]
    int* s_order = s_keys + 128;                                     // [128] rank -> sequence
    int* s_off = s_order + 128;                                      // [129]
    const int lt = (int)threadIdx.x - 128;  // list builders: warps 4-11 (batch <= 128)
    for (int bb = lt; bb >= 0 && bb < p.batch; bb += blockDim.x - 128) {
      SeqInfo s;
      int pr = 0, key = 0;
      if (load_seq(p, bb, s)) {
        pr = min((s.lq + 2 * qpt - 1) / (2 * qpt), kMaxUnitPairs);
        key = s.lk;
      } else if (blockIdx.x == 0) {
        record_error(p.err, kErrDeviceArg);
      }
      s_pairs[bb] = pr;
      s_keys[bb] = key;
    }
    __syncthreads();
    if (!p.unit_mmajor) {
      // sequences by key count, longest first (ties by index)
      for (int bb = lt; bb >= 0 && bb < p.batch; bb += blockDim.x - 128) {
        int rk = 0;
        for (int c = 0; c < p.batch; ++c)
          rk += (s_keys[c] > s_keys[bb]) | ((s_keys[c] == s_keys[bb]) & (c < bb));
        s_order[rk] = bb;
      }
      __syncthreads();
      if (lt == 0) {
        int acc = 0;
        for (int rk = 0; rk < p.batch; ++rk) {
          s_off[rk] = acc;
          acc += s_pairs[s_order[rk]];
        }
        s_off[p.batch] = acc;
        *n_units_s = min(acc, kMaxUnits);
      }
      __syncthreads();
      for (int rk = lt; rk >= 0 && rk < p.batch; rk += blockDim.x - 128) {
        const int bb = s_order[rk];
        const int pr = s_pairs[bb];
        for (int m = 0; m < pr; ++m) {
          const int at = s_off[rk] + m;
          if (at < kMaxUnits) units[at] = (uint16_t)(bb | ((pr - 1 - m) << 7));
        }
      }
    } else if (warp == 4) {
      // query pairs from the last (most keys under the mask) down, sequences
      // in order within a level
      int maxp = 0;
      for (int bb = lane; bb < p.batch; bb += 32) maxp = max(maxp, s_pairs[bb]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) maxp = max(maxp, __shfl_xor_sync(0xffffffffu, maxp, o));
      int n = 0;
      for (int m = maxp - 1; m >= 0; --m) {
        for (int base = 0; base < p.batch; base += 32) {
          const int bb = base + lane;
          const bool on = bb < p.batch && s_pairs[bb] > m;
          const unsigned bal = __ballot_sync(0xffffffffu, on);
          const int at = n + __popc(bal & ((1u << lane) - 1u));
          if (on && at < kMaxUnits) units[at] = (uint16_t)(bb | (m << 7));
          n += __popc(bal);
        }
      }
      if (lane == 0) *n_units_s = min(n, kMaxUnits);
    }
  }

  tc_fence_before();
  __syncthreads();  // also publishes the tile list (and frees the scratch)
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_units = *n_units_s;
  const int n_tiles = n_units * p.h_kv;

  if (warp < 4) {
    regs_dec<CP::REGS_CTRL>();
    int issued_k = 0, issued_v = 0, issued_q = 0;

    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        const uint64_t pol_q = l2_policy_evict_first();
        const uint64_t pol_kv = l2_policy_evict_last();
        bool ok = true;
        // K block j of tile T into the ring (false if the wait gave up).
        auto load_k = [&](const PTile& T, int j) {
          const int st = issued_k % KS;
          if (issued_k >= KS &&
              !mbar_wait(k_empty + 8 * st, ((issued_k / KS) - 1) & 1, p.err, abort_flag))
            return false;
          const uint32_t dst = sbase + C::OFF_K + st * C::K_STAGE;
          mbar_arrive_expect_tx(k_full + 8 * st, C::K_STAGE);
#pragma unroll
          for (int pk = 0; pk < C::NPQ; ++pk)
            tma_load_3d(dst + pk * C::PANEL, &tmK, k_full + 8 * st, pk * C::PANEL_ELEMS, T.kh,
                        kv_row_ok(p, T.sq.k0 + T.kb0 + j * kBlockN) ? T.sq.k0 + T.kb0 + j * kBlockN : 0,
                        pol_kv);
          ++issued_k;
          return true;
        };
        auto load_v = [&](const PTile& T, int j) {
          const int st = issued_v % VS;
          if (issued_v >= VS &&
              !mbar_wait(v_empty + 8 * st, ((issued_v / VS) - 1) & 1, p.err, abort_flag))
            return false;
          const uint32_t dst = sbase + C::OFF_V + st * C::V_STAGE;
          mbar_arrive_expect_tx(v_full + 8 * st, C::V_STAGE);
#pragma unroll
          for (int pv = 0; pv < C::NPV; ++pv)
            tma_load_3d(dst + pv * C::PANEL, &tmV, v_full + 8 * st, pv * C::PANEL_ELEMS, T.kh,
                        kv_row_ok(p, T.sq.k0 + T.kb0 + j * kBlockN) ? T.sq.k0 + T.kb0 + j * kBlockN : 0,
                        pol_kv);
          ++issued_v;
          return true;
        };
        // Q and the first K/V block of a claimed tile into L2 while the
        // current tile's last blocks run: the tile's own Q load can only start
        // once the current tile's last S MMAs have read the old Q, and then
        // finds it in L2.
        auto prefetch_tile = [&](const PTile& T) {
          const int ntiles = T.nq_b > 0 ? 2 : 1;
          for (int t = 0; t < ntiles; ++t)
#pragma unroll
            for (int pq = 0; pq < C::NPQ; ++pq)
              tma_prefetch_l2_3d(&tmQ, pq * C::PANEL_ELEMS, T.kh * group, T.sq.q0 + T.q_start + t * qpt);
#pragma unroll
          for (int pk = 0; pk < C::NPQ; ++pk)
            tma_prefetch_l2_3d(&tmK, pk * C::PANEL_ELEMS, T.kh, T.sq.k0 + T.kb0);
#pragma unroll
          for (int pv = 0; pv < C::NPV; ++pv)
            tma_prefetch_l2_3d(&tmV, pv * C::PANEL_ELEMS, T.kh, T.sq.k0 + T.kb0);
        };
        // Every CTA's first tile is its own index; each later one is claimed
        // from the ticket counter once the tile before it has issued all its
        // loads, so the tiles (longest first) go to whichever CTA is free.
        int claimed = (int)blockIdx.x < n_tiles ? (int)blockIdx.x : -1;
        for (int k = 0; ok; ++k) {
          const int r = claimed;
          PTile T = {};
          if (r >= 0)
            decode_ptile(p, units, r, n_units, qpt, T);
          else
            T.b = -1;
          // hand the decoded tile (or the end mark) to the MMA and softmax roles
          const int sl = k % kTileRing;
          if (k >= kTileRing &&
              !mbar_wait(tr_empty + 8 * sl, ((k / kTileRing) - 1) & 1, p.err, abort_flag))
            break;
          tring[sl] = T;
          mbar_arrive(tr_full + 8 * sl);
          if (r < 0) break;
          if (T.nblk == 0) {
            claimed = ticket_tile(atomicAdd(p.sched, 1), n_tiles);
            continue;
          }
          // K(0) first: its ring stage frees long before the old Q does
          if (!load_k(T, 0)) break;
          // Q of this tile once the previous tile's S MMAs have read theirs
          if (issued_q > 0 && !mbar_wait(q_empty, (issued_q - 1) & 1, p.err, abort_flag)) break;
          const int ntiles = T.nq_b > 0 ? 2 : 1;
          mbar_arrive_expect_tx(q_full, ntiles * C::NPQ * qpt * group * 128);
          for (int t = 0; t < ntiles; ++t)
#pragma unroll
            for (int pq = 0; pq < C::NPQ; ++pq)
              tma_load_3d(sbase + C::OFF_Q + (t * C::NPQ + pq) * C::PANEL, &tmQ, q_full,
                          pq * C::PANEL_ELEMS, T.kh * group,
                          q_row_ok(p, T.sq.q0 + T.q_start + t * qpt) ? T.sq.q0 + T.q_start + t * qpt : 0,
                          pol_q);
          ++issued_q;
          // K(1), V(0), K(2), V(1), ...: K one block ahead of V.
          for (int j = 1; j <= T.nblk; ++j) {
            if (j < T.nblk && !load_k(T, j)) {
              ok = false;
              break;
            }
            if (!load_v(T, j - 1)) {
              ok = false;
              break;
            }
          }
          // This tile's loads are all issued: claim the next one now, so that
          // no CTA holds a tile it will not start for a while, and bring its
          // Q and first K/V block into L2.
          claimed = ticket_tile(atomicAdd(p.sched, 1), n_tiles);
          if (claimed >= 0) {
            PTile T2;
            decode_ptile(p, units, claimed, n_units, qpt, T2);
            if (T2.nblk > 0) prefetch_tile(T2);
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA
      if (lane == 0) {
        // The operand descriptors are built once per call; a k-step only
        // moves the start address (bits 0-13, in 16-byte units), so it adds
        // to the low word.  This single thread issues every MMA of the CTA
        // while sharing its scheduler with two softmax warps, so its
        // instruction count per MMA shows in the tensor pipe's idle time.
        constexpr uint32_t kHiKmaj = smem_desc_sw128_hi(1024);  // Q, K: K-major
        constexpr uint32_t kHiV = smem_desc_sw128_hi(1024);     // V: MN-major
        auto issue_s = [&](int t, int kst) {
          const uint32_t qd = smem_desc_sw128_lo(sbase + C::OFF_Q + t * C::NPQ * C::PANEL, 16);
          const uint32_t kd = smem_desc_sw128_lo(sbase + C::OFF_K + kst * C::K_STAGE, 16);
#pragma unroll
          for (int ks = 0; ks < C::S_KSTEPS; ++ks) {
            const uint32_t off =
                ((ks / C::KSTEPS_PER_PANEL) * C::PANEL + (ks % C::KSTEPS_PER_PANEL) * 32) >> 4;
            tc_mma_f16(tmem + C::tm_s(t), smem_desc_join(qd + off, kHiKmaj),
                       smem_desc_join(kd + off, kHiKmaj), C::IDESC_S, ks > 0 ? 1u : 0u);
          }
          tc_commit(s_full + 8 * t);
        };
        auto issue_pv = [&](int t, int vst, bool first) {
          const uint32_t vd = smem_desc_sw128_lo(sbase + C::OFF_V + vst * C::V_STAGE, C::PANEL);
#pragma unroll
          for (int ks = 0; ks < C::PV_KSTEPS; ++ks)
            tc_mma_f16_ts(tmem + C::tm_o(t), tmem + C::tm_s(t) + ks * 8,
                          smem_desc_join(vd + ((ks * C::UMMA_K * 128) >> 4), kHiV), C::IDESC_PV,
                          (!first || ks > 0) ? 1u : 0u);
        };
        // Running counts: Q tiles and K/V blocks consumed, ring entries read;
        // per slot (bit t) the parity of its p_ready waits and O tiles, and
        // whether it has held an O tile yet.
        int nq = 0, gk = 0, gv = 0, kr = 0;
        uint32_t pcb = 0, odb = 0, odv = 0;
        bool ok = true;
        auto read_ring = [&](PTile& X) {
          const int sl = kr % kTileRing;
          if (!mbar_wait(tr_full + 8 * sl, (kr / kTileRing) & 1, p.err, abort_flag)) return false;
          X = tring[sl];
          mbar_arrive(tr_empty + 8 * sl);
          ++kr;
          return true;
        };
        // S(0) of the next tile into slot t, once its Q and K(0) have landed
        bool s0_ready = false;
        auto issue_s0 = [&](int t) {
          if (!s0_ready) {
            if (!mbar_wait(q_full, nq & 1, p.err, abort_flag) ||
                !mbar_wait(k_full + 8 * (gk % KS), (gk / KS) & 1, p.err, abort_flag))
              return false;
            tc_fence_after();
            s0_ready = true;
          }
          issue_s(t, gk % KS);
          return true;
        };
        // all S(0) of tile X are issued: K(0) frees once they are done
        auto finish_s0 = [&](const PTile& X) {
          tc_commit(k_empty + 8 * (gk % KS));
          ++gk;
          ++nq;
          s0_ready = false;
          if (X.nblk == 1) tc_commit(q_empty);  // its only S MMAs are issued
        };
        PTile T;
        ok = read_ring(T);
        bool s0_done = false;  // T's S(0) went in behind the previous tile
        while (ok && T.b >= 0) {
          if (T.nblk == 0) {
            ok = read_ring(T);
            s0_done = false;
            continue;
          }
          const int ntiles = T.nq_b > 0 ? 2 : 1;
          if (!s0_done) {
            for (int t = 0; ok && t < ntiles; ++t) ok = issue_s0(t);
            if (!ok) break;
            finish_s0(T);
          }
          // The next ring entry is read at the last block; when it has key
          // blocks, its S(0) goes into each slot right behind that slot's
          // last PV (MMAs run in issue order, so S may overwrite P then), and
          // the softmax warps find it ready when their epilogue ends.  Only
          // one entry ahead: the producer can always publish it.
          PTile N;
          N.b = -1;
          int n_ntiles = 0;
          for (int j = 0; ok && j < T.nblk; ++j) {
            const int vst = gv % VS;
            const bool last = j + 1 == T.nblk;
            uint32_t s0m = 0;  // slots given the next tile's S(0)
            for (int t = 0; t < ntiles; ++t) {
              // Slot A's P, V(j) and K(j+1) are usually all there by now: the
              // three phases are tested together (each test takes about 70
              // cycles, and back to back they overlap), and waited for one
              // by one only when one is not complete.
              bool ready = false;
              if (t == 0)
                ready = mbar_test_wait(p_ready, pcb & 1) &
                        mbar_test_wait(v_full + 8 * vst, (gv / VS) & 1) &
                        (last || mbar_test_wait(k_full + 8 * (gk % KS), (gk / KS) & 1));
              if (!ready) {
                ok = mbar_wait(p_ready + 8 * t, (pcb >> t) & 1, p.err, abort_flag);
                if (ok && t == 0)
                  ok = mbar_wait(v_full + 8 * vst, (gv / VS) & 1, p.err, abort_flag);
                if (ok && t == 0 && !last)
                  ok = mbar_wait(k_full + 8 * (gk % KS), (gk / KS) & 1, p.err, abort_flag);
              }
              pcb ^= 1u << t;
              // the previous tile's O in this slot has been read out of TMEM
              if (ok && j == 0 && ((odv >> t) & 1))
                ok = mbar_wait(o_free + 8 * t, ((odb >> t) & 1) ^ 1u, p.err, abort_flag);
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, vst, j == 0);
              if (!last) {
                issue_s(t, gk % KS);
              } else {
                tc_commit(o_done + 8 * t);
                odb ^= 1u << t;
                odv |= 1u << t;
                if (t == 0) {
                  ok = read_ring(N);
                  if (!ok) break;
                  n_ntiles = (N.b >= 0 && N.nblk > 0) ? (N.nq_b > 0 ? 2 : 1) : 0;
                }
                // the next tile's S(0) into every free slot up to this one
                for (int u = 0; ok && u <= t && u < n_ntiles; ++u)
                  if (!((s0m >> u) & 1)) {
                    ok = issue_s0(u);
                    s0m |= 1u << u;
                  }
                if (!ok) break;
              }
            }
            if (!ok) break;
            if (last)  // a slot this tile left idle
              for (int t = 0; ok && t < n_ntiles; ++t)
                if (!((s0m >> t) & 1)) {
                  ok = issue_s0(t);
                  s0m |= 1u << t;
                }
            if (!ok) break;
            tc_commit(v_empty + 8 * vst);
            ++gv;
            if (!last) {
              tc_commit(k_empty + 8 * (gk % KS));
              ++gk;
            }
            if (j + 2 == T.nblk) tc_commit(q_empty);  // S(nblk-1) of both tiles issued
            if (last && n_ntiles > 0) finish_s0(N);
          }
          s0_done = n_ntiles > 0;
          T = N;
        }
        tc_commit(drain);
        mbar_wait(drain, 0, nullptr, nullptr);
      }
    }
    pdl_launch_dependents();
    // --------------------------------------------------- teardown (TMA/MMA side)
    if (warp == 0 && lane == 0 && *abort_flag) {
      for (int st = 0; st < KS && st < issued_k; ++st) {
        const int j_last = st + ((issued_k - 1 - st) / KS) * KS;
        mbar_wait(k_full + 8 * st, (j_last / KS) & 1, nullptr, nullptr);
      }
      for (int st = 0; st < VS && st < issued_v; ++st) {
        const int j_last = st + ((issued_v - 1 - st) / VS) * VS;
        mbar_wait(v_full + 8 * st, (j_last / VS) & 1, nullptr, nullptr);
      }
      if (issued_q > 0) mbar_wait(q_full, (issued_q - 1) & 1, nullptr, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  } else {
    regs_inc<CP::REGS_SOFTMAX>();
    // ------------------------------------------------------- softmax warps
    const int t = (warp - 4) >> 2;  // tile slot 0 (A): warps 4-7, 1 (B): warps 8-11
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::tm_s(t);
    const uint32_t o_addr = tmem + lane_base + C::tm_o(t);
    const float sl2 = p.scale * 1.4426950408889634f;
    int sc = 0, od = 0;  // s_full waits and O tiles of this slot
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int sl = k % kTileRing;
      ok = mbar_wait(tr_full + 8 * sl, (k / kTileRing) & 1, p.err, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      const PTile T = tring[sl];
      __syncwarp();
      if (lane == 0) mbar_arrive(tr_empty + 8 * sl);
      if (T.b < 0) break;
      const int nq = t == 0 ? T.nq_a : T.nq_b;
      if (nq <= 0) continue;
      const int nrows = nq * group;
      const bool warp_active = quarter * 32 < nrows;
      const bool row_ok = r < nrows;
      const int i = T.q_start + t * qpt + r / group;
      const int h = T.kh * group + (r - (r / group) * group);
      // Rows outside the tile never ask for masking (see fa_umma2.cuh).
      int lo = -(1 << 30), hi = 1 << 30;
      if (row_ok) {
        row_key_range(i, T.sq.lq, T.sq.lk, p.causal, p.window_left, lo, hi);
        lo = max(lo, T.k0);
        hi = min(hi, T.k1);
      }
      float m_run = -CUDART_INF_F, l_run = 0.f;
      for (int j = 0; j < T.nblk; ++j) {
        ok = mbar_wait(s_full + 8 * t, sc & 1, p.err, abort_flag);
        ++sc;
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        if (warp_active) {
          const int kb = T.kb0 + j * kBlockN;
          float s[128];
          float m_new = m_run, alpha = 1.f, rsum = 0.f;
          // Once every row of the warp has a running max, the exponentials
          // are first taken against it without the block max.  A row sum of
          // at most 2^8 means that no probability exceeds 2^8, which the lazy
          // rescale allows without moving the max, so the block max was not
          // needed.  Otherwise (rare after a tile's first block) the scores
          // are read again and the block takes the second pass with its max.
          // Both give the same result bit for bit.
          bool with_max = !__all_sync(0xffffffffu, m_run != -CUDART_INF_F);
#pragma unroll 1
          for (;;) {
            tmem_ld128(s_addr, reinterpret_cast<uint32_t*>(s));
            if (__any_sync(0xffffffffu, !(kb >= lo && kb + kBlockN <= hi))) {
              // Under a causal mask most cut blocks are cut by the right bound
              // alone: one compare per key.  The unmasked instantiation only
              // meets sequence tails and keeps the general form alone.
              bool cut = false;
              if constexpr (MASKED) {
                if (__all_sync(0xffffffffu, kb >= lo)) {
                  const int c_hi = hi - kb;
#pragma unroll
                  for (int c = 0; c < 128; ++c) s[c] = c < c_hi ? s[c] : -CUDART_INF_F;
                  cut = true;
                }
              }
              if (!cut) {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                  const int key = kb + c;
                  s[c] = (key >= lo && key < hi) ? s[c] : -CUDART_INF_F;
                }
              }
            }
            float m_use = m_run;
            if (with_max) {
              float mx[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) mx[u] = -CUDART_INF_F;
#pragma unroll
              for (int c = 0; c < 128; c += 16)
#pragma unroll
                for (int u = 0; u < 8; ++u) mx[u] = fmax3(mx[u], s[c + u], s[c + 8 + u]);
              const float bmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
              m_new = (bmax > m_run + 8.f) ? bmax : m_run;  // lazy rescale, 2^8
              m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
              alpha = m_run == m_new ? 1.f : fast_exp2(m_run - m_use);
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
            const float2 r01 = f2_split(f2_add(f2_add(sm[0], sm[1]), f2_add(sm[2], sm[3])));
            rsum = r01.x + r01.y;
            if (with_max || !__any_sync(0xffffffffu, !(rsum <= 256.f))) break;
            with_max = true;
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
          l_run = l_run * alpha + rsum;
          m_run = m_new;
        }
        tc_fence_before();
        mbar_arrive(p_ready + 8 * t);
      }
      if (!ok) break;

      // ------------------------------------------------------------ epilogue
      if (T.nblk > 0) {
        ok = mbar_wait(o_done + 8 * t, od & 1, p.err, abort_flag);
        ++od;
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
      }
      float inv = 0.f, lse_v = -CUDART_INF_F;
      if (row_ok && l_run > 0.f && m_run != -CUDART_INF_F) {
        inv = 1.f / l_run;
        lse_v = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      }
      const int tok = T.sq.q0 + i;
      // O out of TMEM in one load, released, then scaled and stored
      uint32_t o[DV];
      if (warp_active && T.nblk > 0) {
        if constexpr (DV == 128)
          tmem_ld128(o_addr, o);
        else
          tmem_ld64(o_addr, o);
      } else {
#pragma unroll
        for (int e = 0; e < DV; ++e) o[e] = 0u;
      }
      if (T.nblk > 0) {
        // O has been read out of TMEM: the next tile's first PV may overwrite it
        tc_fence_before();
        mbar_arrive(o_free + 8 * t);
      }
      if (warp_active && row_ok) {
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          const size_t oe = ((size_t)tok * p.h_q + h) * DV + c * 32;
          if (o_ok(p, oe, 32))
            store_o<32, true>(p.out, oe, reinterpret_cast<const float*>(o + 32 * c), inv,
                              p.out_dtype);
        }
      }
      if (warp_active && row_ok && p.lse != nullptr && lse_ok(p, h, tok))
        p.lse[(size_t)h * p.total_q + tok] = lse_v;
    }
    // teardown (softmax side): the TMEM release waits for these warps
    tc_fence_before();
    __syncthreads();
  }
}

}  // namespace fa
