"""Integer split planner and per-split key ranges (the rule the library must
reproduce bit for bit).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages give the inputs of the split choice but not a formula:
[AITER] description ("automatic and explicit split selection") and its review
("auto split-K, up to 16 splits plus a per-call fp32 workspace"); [FA4]
"Benchmarks" (one split is 4.6x slower than 4..32 splits at one query, 32
heads, 131072 keys, because 32 CTAs cannot fill the GPU).  The reading used
here, sized from B * H_kv * ceil(Q * group / 128) work units against the SM
count:

  units  = batch * h_kv * ceil(max_seqlen_q * group / 128)
  explicit num_splits > 0     -> min(num_splits, 128)
  units == 0                  -> 1
  units >= 2 * num_sms        -> 1            (already two full waves)
  otherwise the smallest ns in 1..128 whose wave efficiency
      units*ns / (ceil(units*ns / num_sms) * num_sms) >= 0.9
  (integer test: 10*units*ns >= 9*waves*num_sms), else the first ns with the
  highest efficiency.

Per-split key ranges.  A tile of queries [i_lo, i_hi] of a sequence (Lq, Lk)
attends keys [lo, hi) = union of its rows' allowed ranges ([CUTLASS]
"Implementation": masks get that sequence's lengths; a tile whose key
sequence is empty is skipped).  Keys are grouped in blocks of 128
(BLOCK_N); blocks b_lo = lo // 128 .. b_hi = ceil(hi / 128), nb = b_hi - b_lo.
The split count used by this tile is ns_eff = min(ns, nb) and split s < ns_eff
takes blocks [b_lo + s*nb//ns_eff, b_lo + (s+1)*nb//ns_eff), clipped to
[lo, hi) in keys.  Splits s >= ns_eff are empty (partial LSE = -inf).
"""

from __future__ import annotations

BLOCK_N = 128      # keys per split block
M_TILE = 128       # rows of the tensor-core query tile ([FA4] description: M = 128)
MAX_SPLITS = 128   # largest split count ([FA4] "Benchmarks" sweeps up to 128)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def plan_num_splits(batch: int, max_seqlen_q: int, h_q: int, h_kv: int,
                    num_splits: int, num_sms: int):
    """-> (num_splits, units).  See the module docstring for the rule."""
    group = h_q // h_kv
    m_blocks = _ceil_div(max_seqlen_q * group, M_TILE)
    units = batch * h_kv * m_blocks
    if num_splits > 0:
        return min(num_splits, MAX_SPLITS), units
    if units <= 0:
        return 1, units
    if units >= 2 * num_sms:
        return 1, units
    best_ns, best_num, best_den = 1, 0, 1
    for ns in range(1, MAX_SPLITS + 1):
        work = units * ns
        waves = _ceil_div(work, num_sms)
        den = waves * num_sms
        if 10 * work >= 9 * den:
            return ns, units
        # compare work/den > best_num/best_den without floats
        if work * best_den > best_num * den:
            best_ns, best_num, best_den = ns, work, den
    return best_ns, units


def tile_key_range(i_lo: int, i_hi: int, lq: int, lk: int, causal: bool,
                   window_left: int):
    """Union [lo, hi) of the allowed key ranges of queries i_lo..i_hi
    (inclusive) of one sequence.  Empty ranges come back with hi <= lo."""
    if lk <= 0:
        return 0, 0
    if not causal and window_left < 0:
        return 0, lk
    off = lk - lq
    hi = min(lk, i_hi + off + 1)
    lo = 0 if window_left < 0 else max(0, i_lo + off - window_left)
    return lo, hi


def split_block_range(nb: int, ns: int, s: int):
    """Blocks [b0, b1) of split s when nb blocks are cut into
    ns_eff = min(ns, nb) nearly equal parts."""
    if nb <= 0:
        return 0, 0
    ns_eff = min(ns, nb)
    if s >= ns_eff:
        return 0, 0
    return (s * nb) // ns_eff, ((s + 1) * nb) // ns_eff


def tile_split_key_range(i_lo: int, i_hi: int, lq: int, lk: int, causal: bool,
                         window_left: int, ns: int, s: int):
    """Keys [k0, k1) that split s of the query tile i_lo..i_hi processes
    (k1 <= k0 means the split is empty)."""
    lo, hi = tile_key_range(i_lo, i_hi, lq, lk, causal, window_left)
    if hi <= lo:
        return 0, 0
    b_lo = lo // BLOCK_N
    b_hi = _ceil_div(hi, BLOCK_N)
    b0, b1 = split_block_range(b_hi - b_lo, ns, s)
    if b1 <= b0:
        return 0, 0
    k0 = max(lo, (b_lo + b0) * BLOCK_N)
    k1 = min(hi, (b_lo + b1) * BLOCK_N)
    return k0, k1


def workspace_bytes(batch: int, max_seqlen_q: int, h_q: int, d_v: int, ns: int) -> int:
    """fp32 split workspace: partial O [ns, batch*max_seqlen_q, h_q, d_v] then
    partial LSE [ns, batch*max_seqlen_q, h_q]; none when ns == 1."""
    if ns <= 1:
        return 0
    slots = batch * max_seqlen_q * h_q
    return 4 * ns * slots * (d_v + 1)
