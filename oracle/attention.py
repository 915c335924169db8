"""Float64 CPU definition of the forward attention that split-KV computes.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed (the plain definition; split-KV reaches it by exact
re-association):

  for every packed sequence b, query head h (key/value head kh = h // group)
  and query i < Lq_b, over the keys j the mask allows:

      s_j  = scale * dq * dk * <Q[t_i, h, :], K[u_j, kh, :]>
      LSE  = log(sum_j exp(s_j))                      (natural log)
      O    = dv * sum_j exp(s_j - LSE) * V[u_j, kh, :]

  [FA4] description and [AITER] description: forward attention returning the
  output and its log-sum-exp.  [CUTLASS] "Interface": Q/K/V/O/LSE packed
  along the sequence axis, sequence b's rows are cu_seqlens[b] ..
  cu_seqlens[b+1]-1.  dq, dk, dv are per-tensor FP8 descales ([AITER]
  description: FP8 FMHA); they are 1 for 16-bit inputs.

Readings where the pages are silent:

* LSE is the natural log and includes the softmax scale.
* LSE is laid out [h_q, total_q].
* A query row with no allowed key (empty key sequence, or a causal row that
  sees no key) has O = 0 and LSE = -inf.  [CUTLASS] "Implementation" leaves
  such rows unwritten; this oracle defines them.
* Causal is bottom-right aligned ([CUTLASS] "Tests": bottom-right causal for
  different q/k lengths): query i may see key j iff j <= i + Lk - Lq.
* A window (wl, 0) ([CUTLASS] "Tests": window (128, 0)) additionally needs
  j >= i + Lk - Lq - wl; the right bound is 0, so a window implies causal.
* The default scale is 1/sqrt(head dim of Q/K) ([CUTLASS] "Implementation",
  the default softmax scale bullet).
"""

from __future__ import annotations

import math

import numpy as np
import torch

NEG_INF = float("-inf")


def default_softmax_scale(d_qk: int) -> float:
    """1/sqrt(d_qk): [CUTLASS] "Implementation", default softmax scale uses
    the head dimension, not the (possibly packed) sequence length."""
    return 1.0 / math.sqrt(d_qk)


def decode_inputs_f64(x, descale: float = 1.0) -> np.ndarray:
    """Widen a bf16 / fp16 / float8_e4m3fn / float tensor to float64 exactly,
    then apply a per-tensor descale.  Every 16-bit and 8-bit value is exactly
    representable in float64, so the widening itself is exact."""
    if isinstance(x, torch.Tensor):
        arr = x.detach().to("cpu").to(torch.float64).numpy()
    else:
        arr = np.asarray(x, dtype=np.float64)
    if descale != 1.0:
        arr = arr * float(descale)
    return arr


def allowed_key_range(i: int, lq: int, lk: int, causal: bool, window_left: int):
    """Keys query i of a (lq, lk) sequence may attend, as [lo, hi).

    [CUTLASS] "Tests": no mask, bottom-right causal, window (128, 0).
    The diagonal of query i sits at key i + lk - lq (bottom-right alignment).
    A window of (wl, 0) keeps keys diag - wl .. diag inclusive.
    """
    if not causal and window_left < 0:
        return 0, lk
    diag = i + lk - lq
    hi = diag + 1
    lo = diag - window_left if window_left >= 0 else 0
    lo = max(lo, 0)
    hi = min(hi, lk)
    if hi < lo:
        hi = lo
    return lo, hi


def allowed_mask(lq: int, lk: int, causal: bool, window_left: int) -> np.ndarray:
    """Boolean [lq, lk] matrix of allowed (query, key) pairs."""
    m = np.zeros((lq, lk), dtype=bool)
    for i in range(lq):
        lo, hi = allowed_key_range(i, lq, lk, causal, window_left)
        m[i, lo:hi] = True
    return m


def _softmax_rows(s: np.ndarray, v: np.ndarray):
    """Rows of s (already masked with -inf) -> (O, LSE) with a max-subtracted
    log-sum-exp.  Rows with no finite entry give O = 0 and LSE = -inf."""
    lq = s.shape[0]
    d_v = v.shape[1]
    o = np.zeros((lq, d_v), dtype=np.float64)
    lse = np.full((lq,), NEG_INF, dtype=np.float64)
    if s.shape[1] == 0:
        return o, lse
    m = s.max(axis=1)
    ok = np.isfinite(m)
    if not ok.any():
        return o, lse
    sm = s[ok] - m[ok][:, None]
    p = np.exp(sm)  # exp(-inf) = 0 for masked keys
    l = p.sum(axis=1)
    lse[ok] = m[ok] + np.log(l)
    o[ok] = (p @ v) / l[:, None]
    return o, lse


def attention_forward(q, k, v, cu_seqlens_q, cu_seqlens_k, h_q: int, h_kv: int,
                      scale: float | None = None, causal: bool = False,
                      window_left: int = -1, descale_q: float = 1.0,
                      descale_k: float = 1.0, descale_v: float = 1.0):
    """O [total_q, h_q, d_v] and LSE [h_q, total_q], float64.

    q: [total_q, h_q, d_qk], k: [total_k, h_kv, d_qk], v: [total_k, h_kv, d_v]
    as torch tensors (any dtype) or arrays.  cu_seqlens_*: int [B+1].
    The full score matrix of every (sequence, head) is materialised.
    GQA: query head h reads key/value head h // (h_q // h_kv)
    ([CUTLASS] "Interface": GQA/MQA).
    """
    qf = decode_inputs_f64(q)
    kf = decode_inputs_f64(k)
    vf = decode_inputs_f64(v)
    cq = [int(x) for x in (cu_seqlens_q.tolist() if hasattr(cu_seqlens_q, "tolist") else cu_seqlens_q)]
    ck = [int(x) for x in (cu_seqlens_k.tolist() if hasattr(cu_seqlens_k, "tolist") else cu_seqlens_k)]
    assert len(cq) == len(ck)
    assert h_q % h_kv == 0
    group = h_q // h_kv
    total_q = qf.shape[0]
    d_qk = qf.shape[2]
    d_v = vf.shape[2]
    if scale is None or scale <= 0:
        scale = default_softmax_scale(d_qk)
    s_eff = float(scale) * float(descale_q) * float(descale_k)
    out = np.zeros((total_q, h_q, d_v), dtype=np.float64)
    lse = np.full((h_q, total_q), NEG_INF, dtype=np.float64)
    for b in range(len(cq) - 1):
        q0, q1 = cq[b], cq[b + 1]
        k0, k1 = ck[b], ck[b + 1]
        lq, lk = q1 - q0, k1 - k0
        if lq <= 0:
            continue
        mask = allowed_mask(lq, lk, causal, window_left)
        for h in range(h_q):
            kh = h // group
            s = s_eff * (qf[q0:q1, h, :] @ kf[k0:k1, kh, :].T)
            s = np.where(mask, s, NEG_INF)
            o_bh, lse_bh = _softmax_rows(s, vf[k0:k1, kh, :])
            out[q0:q1, h, :] = float(descale_v) * o_bh
            lse[h, q0:q1] = lse_bh
    return out, lse


def partial_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, h_q: int, h_kv: int,
                      key_ranges, scale: float | None = None, causal: bool = False,
                      window_left: int = -1, descale_q: float = 1.0,
                      descale_k: float = 1.0, descale_v: float = 1.0):
    """Attention restricted to one key sub-range per sequence: the per-split
    partial result of split-KV ([FA4] description, [AITER] description).

    key_ranges[b] = (j0, j1) in sequence-local key indices.  Returns the
    partial O_s (normalised over its own keys) and lse_s, with O_s = 0 and
    lse_s = -inf where the range holds no allowed key.
    """
    qf = decode_inputs_f64(q)
    kf = decode_inputs_f64(k)
    vf = decode_inputs_f64(v)
    cq = [int(x) for x in (cu_seqlens_q.tolist() if hasattr(cu_seqlens_q, "tolist") else cu_seqlens_q)]
    ck = [int(x) for x in (cu_seqlens_k.tolist() if hasattr(cu_seqlens_k, "tolist") else cu_seqlens_k)]
    group = h_q // h_kv
    total_q, _, d_qk = qf.shape
    d_v = vf.shape[2]
    if scale is None or scale <= 0:
        scale = default_softmax_scale(d_qk)
    s_eff = float(scale) * float(descale_q) * float(descale_k)
    out = np.zeros((total_q, h_q, d_v), dtype=np.float64)
    lse = np.full((h_q, total_q), NEG_INF, dtype=np.float64)
    for b in range(len(cq) - 1):
        q0, q1 = cq[b], cq[b + 1]
        k0, k1 = ck[b], ck[b + 1]
        lq, lk = q1 - q0, k1 - k0
        if lq <= 0:
            continue
        j0, j1 = key_ranges[b]
        j0, j1 = max(0, j0), min(lk, j1)
        mask = allowed_mask(lq, lk, causal, window_left)
        sub = np.zeros_like(mask)
        if j1 > j0:
            sub[:, j0:j1] = True
        mask = mask & sub
        for h in range(h_q):
            kh = h // group
            s = s_eff * (qf[q0:q1, h, :] @ kf[k0:k1, kh, :].T)
            s = np.where(mask, s, NEG_INF)
            o_bh, lse_bh = _softmax_rows(s, vf[k0:k1, kh, :])
            out[q0:q1, h, :] = float(descale_v) * o_bh
            lse[h, q0:q1] = lse_bh
    return out, lse


def combine_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """LSE-weighted merge of split partials ([AITER] timing note: attention
    and split combine; [FA4] split-KV).

    o_parts: [ns, ..., d_v], lse_parts: [ns, ...] (natural-log LSE of each
    split).  With M = max_s lse_s:
        LSE = M + log(sum_s exp(lse_s - M))
        O   = sum_s exp(lse_s - LSE) * O_s
    Positions where every split is empty (M = -inf) give O = 0, LSE = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    ok = np.isfinite(m)
    m_safe = np.where(ok, m, 0.0)
    w = np.exp(lse_parts - m_safe[None])  # exp(-inf) = 0 for empty splits
    total = w.sum(axis=0)
    lse = np.where(ok, m_safe + np.log(np.where(ok, total, 1.0)), NEG_INF)
    lse_safe = np.where(ok, lse, 0.0)
    coef = np.where(ok[None], np.exp(lse_parts - lse_safe[None]), 0.0)
    o = (coef[..., None] * o_parts).sum(axis=0)
    return o, lse


def split_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, h_q: int, h_kv: int,
                    ranges_per_split, scale: float | None = None,
                    causal: bool = False, window_left: int = -1,
                    descale_q: float = 1.0, descale_k: float = 1.0,
                    descale_v: float = 1.0):
    """Split-KV as the two steps the pages name: a partial attention per
    split, then the LSE-weighted combine.  ranges_per_split[s][b] = (j0, j1).
    Equal to attention_forward up to float64 rounding whenever the ranges of
    each sequence partition its keys."""
    o_parts, l_parts = [], []
    for ranges in ranges_per_split:
        o_s, l_s = partial_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, h_q, h_kv,
                                     ranges, scale, causal, window_left,
                                     descale_q, descale_k, descale_v)
        o_parts.append(o_s)
        l_parts.append(l_s.T)  # -> [total_q, h_q] to line up with O
    o, lse_t = combine_partials(np.stack(o_parts), np.stack(l_parts))
    return o, lse_t.T
