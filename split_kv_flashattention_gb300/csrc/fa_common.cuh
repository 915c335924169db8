// Shared definitions of the split-KV forward path: launch parameters, the
// tile -> (sequence, head, split) decode and the per-split key range.
//
// Packed varlen layout (cutlass "Adds variable sequence lengths to the
// Hopper CuTe DSL FMHA example", section "Interface"): sequence b owns query
// rows cu_q[b] .. cu_q[b+1]-1 of Q [total_q, h_q, d_qk] and O
// [total_q, h_q, d_v], and key rows cu_k[b] .. cu_k[b+1]-1 of
// K [total_k, h_kv, d_qk] and V [total_k, h_kv, d_v].  Query head h reads
// key/value head h / (h_q / h_kv) (GQA).
#pragma once

#include <stdint.h>

#include "fa_ptx.cuh"

namespace fa {

constexpr int kBlockN = 128;    // keys per split block
constexpr int kMaxSplits = 128;
// Tile list of the persistent two-tile kernel: (sequence, 256-row query pair)
// units held in shared memory, 7 bits of sequence and 9 of pair each.  The
// host bounds the units by batch * pairs of the longest sequence.
constexpr int kMaxUnits = 4096;
constexpr int kMaxUnitPairs = 512;
// Slots of the ring through which its producer hands each claimed tile to the
// MMA and softmax roles.
constexpr int kTileRing = 4;
// Workspace bytes of a one-split call: the persistent kernel's ticket counter.
constexpr unsigned kSchedBytes = 16;
constexpr int kMinPage = 32;                 // smallest page of a paged K/V cache
constexpr int kMaxSub = kBlockN / kMinPage;  // page-sized loads per key block, at most

enum DType : int { kBF16 = 0, kFP16 = 1, kE4M3 = 2 };

struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  const int* cu_q;
  const int* cu_k;
  void* out;
  float* lse;       // [h_q, total_q] natural log, may be null
  float* ws_o;      // [ns, slots, h_q, d_v] fp32 partial outputs (ns > 1)
  float* ws_l;      // [ns, slots, h_q]      fp32 partial LSEs    (ns > 1)
  const float* descale_q;
  const float* descale_k;
  const float* descale_v;
  int* err;         // device error word
  int batch, total_q, total_k, max_seqlen_q;
  int h_q, h_kv, group, d_qk, d_v;
  int num_splits;
  int causal;
  int window_left;  // < 0: unbounded
  float scale;      // softmax scale (already resolved from the default)
  int out_dtype;    // DType of O
  int slots;        // batch * max_seqlen_q
  int tile_rows;    // rows (query, head pairs) per CTA tile
  // Paged K/V (page_size > 0): K/V are page pools [num_pages*page_size, h_kv, d];
  // key j of sequence b lives in pool row
  //   block_table[b*max_pages + j/page_size]*page_size + j%page_size
  // and seqlens_k[b] gives the sequence's key count (cu_k is unused).
  const int* block_table;
  const int* seqlens_k;
  int max_pages;
  int page_size;    // 0: contiguous packed K/V addressed through cu_k
  int page_shift;   // log2(page_size)
  int num_sms;      // SMs of the device (0 if unknown)
  int* sched;       // persistent kernel's tile ticket counter, zero at launch
  int kv_head_group;  // persistent kernel: KV heads per group of its tile walk (divides h_kv)
  int unit_mmajor;    // persistent kernel: units m-major (1) or by key count, last pair first (0)
};

struct SeqInfo {
  int q0, lq, k0, lk;
};

// ---- bounds checks of the debug build (FA_DEBUG)
// Every global access of the kernels goes through one of these predicates.
// In a debug build a failed check records FA_ERR_DEVICE_BOUNDS in the error
// word and the caller skips the access; the context stays usable.  In the
// normal build they are constant true and compile away.
#ifdef FA_DEBUG
__device__ __forceinline__ bool dbg_ok(const FwdParams& p, bool ok) {
  if (!ok) record_error(p.err, kErrDeviceBounds);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool dbg_ok(const FwdParams&, bool) { return true; }
#endif
// n elements of O from element `elem` on
__device__ __forceinline__ bool o_ok(const FwdParams& p, size_t elem, int n) {
  return dbg_ok(p, elem + n <= (size_t)p.total_q * p.h_q * p.d_v);
}
__device__ __forceinline__ bool lse_ok(const FwdParams& p, int h, int t) {
  return dbg_ok(p, h >= 0 && h < p.h_q && t >= 0 && t < p.total_q);
}
// n fp32 partials of O from index `idx` on; one partial LSE at `idx`
__device__ __forceinline__ bool ws_o_ok(const FwdParams& p, size_t idx, int n) {
  return dbg_ok(p, p.ws_o != nullptr &&
                       idx + n <= (size_t)p.num_splits * p.slots * p.h_q * p.d_v);
}
__device__ __forceinline__ bool ws_l_ok(const FwdParams& p, size_t idx) {
  return dbg_ok(p, p.ws_l != nullptr && idx < (size_t)p.num_splits * p.slots * p.h_q);
}
// first row of a K/V or Q box (a box may run past the last row: TMA fills zeros)
__device__ __forceinline__ bool kv_row_ok(const FwdParams& p, int row) {
  return dbg_ok(p, row >= 0 && row < p.total_k);
}
__device__ __forceinline__ bool q_row_ok(const FwdParams& p, int row) {
  return dbg_ok(p, row >= 0 && row < p.total_q);
}
__device__ __forceinline__ bool seq_ok_idx(const FwdParams& p, int b) {
  return dbg_ok(p, b >= 0 && b < p.batch);
}

// Reads and validates one sequence's offsets.  A sequence whose lengths are
// negative, exceed max_seqlen_q, or overrun the declared buffers is skipped
// and reported through the error word (never read or written out of range).
__device__ __forceinline__ bool load_seq(const FwdParams& p, int b, SeqInfo& s) {
  if (!seq_ok_idx(p, b)) b = 0;
  s.q0 = __ldg(p.cu_q + b);
  s.lq = __ldg(p.cu_q + b + 1) - s.q0;
  if (p.page_size > 0) {
    s.k0 = 0;
    s.lk = __ldg(p.seqlens_k + b);
    return s.q0 >= 0 && s.lq >= 0 && s.lk >= 0 && s.lq <= p.max_seqlen_q &&
           s.q0 + s.lq <= p.total_q && (long long)s.lk <= (long long)p.max_pages * p.page_size;
  }
  s.k0 = __ldg(p.cu_k + b);
  s.lk = __ldg(p.cu_k + b + 1) - s.k0;
  bool ok = s.q0 >= 0 && s.lq >= 0 && s.k0 >= 0 && s.lk >= 0 && s.lq <= p.max_seqlen_q &&
            s.q0 + s.lq <= p.total_q && s.k0 + s.lk <= p.total_k;
  return ok;
}

// First K/V row of a load of `box` rows starting at key `key` (sequence-
// local) of sequence b.  For paged K/V the caller keeps the load inside one
// page (key % box == 0, box <= page_size, both powers of two).  Loads that
// start past the sequence's keys (tails of the last block; every such row is
// masked) read the sequence's last box instead, so they never index the
// block table past the sequence's pages and always bring finite values.  A
// page index outside the pool reads row 0 and is reported through the error
// word.
//
// The block-table lookups go through a cursor owned by the one producer
// thread, which walks keys in increasing order.  It keeps the key range of
// the page in use and that page's base row, so a load inside the same page
// costs two compares and an add; on entering a page it already fetches the
// next page's entry, so that lookup's latency overlaps a page worth of loads
// instead of stalling the next TMA issue.
struct PageCursor {
  int lo = 0, hi = 0;    // sequence keys [lo, hi) of the page in use
  int base = 0;          // pool row of key lo, minus lo
  int nxt_lp = -1, nxt_pp = 0;  // the following logical page and its pool page
};

__device__ __forceinline__ void page_enter(const FwdParams& p, const SeqInfo& s, int b, int key,
                                        PageCursor& pc) {
  const int lp = key >> p.page_shift;
  const int* row = p.block_table + (size_t)b * p.max_pages;
  int pg = lp == pc.nxt_lp ? pc.nxt_pp : __ldg(row + lp);
  pc.nxt_lp = lp + 1;
  pc.nxt_pp = (long long)(lp + 1) * p.page_size < s.lk ? __ldg(row + lp + 1) : 0;
  if (pg < 0 || (long long)(pg + 1) * p.page_size > p.total_k) {
    if (p.err) atomicCAS(p.err, 0, -6);
    pg = 0;
  }
  pc.lo = lp << p.page_shift;
  pc.hi = pc.lo + p.page_size;
  pc.base = pg * p.page_size - pc.lo;
}

__device__ __forceinline__ int kv_row_walk(const FwdParams& p, const SeqInfo& s, int b, int key,
                                           int box, PageCursor& pc) {
  int row;
  if (p.page_size <= 0) {
    row = s.k0 + key;
  } else {
    if (key >= s.lk) key = (s.lk - 1) & ~(box - 1);
    if (__builtin_expect(key < pc.lo || key >= pc.hi, 0)) page_enter(p, s, b, key, pc);
    row = pc.base + key;
  }
  return kv_row_ok(p, row) ? row : 0;
}

// ---- longest-first dispatch of decode tiles
// The CTAs of a grid start roughly in linear block order (x fastest, then y,
// then z).  A decode CTA's work is its split's share of one sequence's keys,
// so in a varlen batch the grid order leaves long splits for the last wave
// while the other SMs idle.  The CTA's linear index is therefore read as
// (rank, split, KV head, row tile), rank slowest, where rank orders the
// sequences by key count, longest first, ties by index: the launch becomes a
// longest-processing-time-first list schedule of the splits.  The mapping is
// a bijection onto the same (tile, sequence, head, split) set, so the
// results do not change.  Larger batches keep the grid order.  (cutlass
// "Adds variable sequence lengths to the Hopper CuTe DSL FMHA example",
// section "Performance (GH200)": a static assignment over the max-length
// grid balances skewed lengths poorly; a length-aware schedule is the named
// follow-up.)
constexpr int kMaxRankedSeqs = 128;

struct TileIdx {
  int m_blk, b, kh, split;
};

__device__ __forceinline__ int seq_keys(const FwdParams& p, int b) {
  return p.page_size > 0 ? __ldg(p.seqlens_k + b) : __ldg(p.cu_k + b + 1) - __ldg(p.cu_k + b);
}

// Tile of this CTA in plain grid order: x = row tile, y = sequence * h_kv +
// KV head, z = split.
__device__ __forceinline__ TileIdx grid_order_tile(const FwdParams& p) {
  TileIdx t;
  t.m_blk = blockIdx.x;
  t.b = blockIdx.y / p.h_kv;
  t.kh = blockIdx.y - t.b * p.h_kv;
  t.split = blockIdx.z;
  return t;
}

// Tile of a tensor-core CTA: grid x = query tiles, y = sequence * h_kv + KV
// head, z = split.  Query tiles run last tile first.  Without a mask every
// tile of a sequence does the same work, and the x-fastest order keeps the
// tiles of one (sequence, head), which share K/V in L2, together.  With a
// causal or window mask a tile's work grows with its index m and hardly
// depends on the sequence, so the tiles run m-major (all sequences' last
// tiles first): a longest-first order computed from the block index alone.
__device__ __forceinline__ TileIdx query_tile_order_at(const FwdParams& p, int x, int y, int z) {
  TileIdx t;
  if (p.causal || p.window_left >= 0) {
    const int lin = x + gridDim.x * y;
    x = lin / gridDim.y;
    y = lin - x * gridDim.y;
  }
  t.m_blk = gridDim.x - 1 - x;
  t.b = y / p.h_kv;
  t.kh = y - t.b * p.h_kv;
  t.split = z;
  return t;
}

__device__ __forceinline__ TileIdx query_tile_order(const FwdParams& p) {
  return query_tile_order_at(p, blockIdx.x, blockIdx.y, blockIdx.z);
}

// Every thread of the CTA calls this: it holds two barriers.  `keys` and
// `pick` are shared-memory scratch of kMaxRankedSeqs ints and one int.
__device__ __forceinline__ TileIdx longest_first_tile(const FwdParams& p, int* keys, int* pick) {
  const int gx = gridDim.x;
  const int ns = gridDim.z;
  int v = blockIdx.x + gx * (blockIdx.y + gridDim.y * blockIdx.z);
  TileIdx t;
  t.m_blk = v % gx;
  v /= gx;
  t.kh = v % p.h_kv;
  v /= p.h_kv;
  t.split = v % ns;
  const int rank = v / ns;
  t.b = rank;
  if (p.batch > 1 && p.batch <= kMaxRankedSeqs) {  // else the identity order
    for (int i = threadIdx.x; i < p.batch; i += blockDim.x) keys[i] = seq_keys(p, i);
    __syncthreads();
    for (int i = threadIdx.x; i < p.batch; i += blockDim.x) {
      const int li = keys[i];
      int r = 0;
      for (int c = 0; c < p.batch; ++c) r += (keys[c] > li) | ((keys[c] == li) & (c < i));
      if (r == rank) *pick = i;
    }
    __syncthreads();
    t.b = *pick;
  }
  return t;
}

// First key of a tile's load schedule: the split's first key, rounded down to
// the load granularity in paged mode so no load crosses a page.
__device__ __forceinline__ int load_base(const FwdParams& p, int k0, int granularity) {
  return p.page_size > 0 ? k0 & ~(granularity - 1) : k0;
}

// Allowed keys [lo, hi) of query i in a (lq, lk) sequence: everything without
// a mask; bottom-right causal keeps keys <= i + lk - lq; a (window_left, 0)
// window also drops keys < i + lk - lq - window_left.
__device__ __forceinline__ void row_key_range(int i, int lq, int lk, int causal, int wl,
                                              int& lo, int& hi) {
  if (!causal && wl < 0) {
    lo = 0;
    hi = lk;
    return;
  }
  int diag = i + lk - lq;
  hi = min(diag + 1, lk);
  lo = wl >= 0 ? max(diag - wl, 0) : 0;
  if (hi < lo) hi = lo;
}

// Keys [k0, k1) processed by split s of a tile covering queries
// i_lo..i_hi: the union of the rows' ranges is cut into 128-key blocks and
// the blocks into ns_eff = min(ns, nb) nearly equal runs.
__device__ __forceinline__ void tile_split_range(int i_lo, int i_hi, int lq, int lk, int causal,
                                                 int wl, int ns, int s, int& k0, int& k1) {
  k0 = 0;
  k1 = 0;
  if (lk <= 0) return;
  int lo = 0, hi = lk;
  if (causal || wl >= 0) {
    int off = lk - lq;
    hi = min(lk, i_hi + off + 1);
    lo = wl >= 0 ? max(0, i_lo + off - wl) : 0;
  }
  if (hi <= lo) return;
  int b_lo = lo / kBlockN;
  int b_hi = (hi + kBlockN - 1) / kBlockN;
  int nb = b_hi - b_lo;
  int ns_eff = min(ns, nb);
  if (s >= ns_eff) return;
  int b0 = (int)(((long long)s * nb) / ns_eff);
  int b1 = (int)(((long long)(s + 1) * nb) / ns_eff);
  if (b1 <= b0) return;
  k0 = max(lo, (b_lo + b0) * kBlockN);
  k1 = min(hi, (b_lo + b1) * kBlockN);
}

}  // namespace fa
