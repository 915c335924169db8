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

namespace fa {

constexpr int kBlockN = 128;    // keys per split block
constexpr int kMaxSplits = 128;

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
};

struct SeqInfo {
  int q0, lq, k0, lk;
};

// Reads and validates one sequence's offsets.  A sequence whose lengths are
// negative, exceed max_seqlen_q, or overrun the declared buffers is skipped
// and reported through the error word (never read or written out of range).
__device__ __forceinline__ bool load_seq(const FwdParams& p, int b, SeqInfo& s) {
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
__device__ __forceinline__ int kv_row(const FwdParams& p, const SeqInfo& s, int b, int key,
                                      int box) {
  if (p.page_size <= 0) return s.k0 + key;
  if (key >= s.lk) key = (s.lk - 1) - ((s.lk - 1) % box);
  const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + key / p.page_size);
  if (pg < 0 || (long long)(pg + 1) * p.page_size > p.total_k) {
    if (p.err) atomicCAS(p.err, 0, -6);
    return 0;
  }
  return pg * p.page_size + (key & (p.page_size - 1));
}

// First key of a tile's load schedule: the split's first key, rounded down to
// the load granularity in paged mode so no load crosses a page.
__device__ __forceinline__ int load_base(const FwdParams& p, int k0, int granularity) {
  return p.page_size > 0 ? k0 - (k0 % granularity) : k0;
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
