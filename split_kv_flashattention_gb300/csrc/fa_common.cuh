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
  s.k0 = __ldg(p.cu_k + b);
  s.lk = __ldg(p.cu_k + b + 1) - s.k0;
  bool ok = s.q0 >= 0 && s.lq >= 0 && s.k0 >= 0 && s.lk >= 0 && s.lq <= p.max_seqlen_q &&
            s.q0 + s.lq <= p.total_q && s.k0 + s.lk <= p.total_k;
  return ok;
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
