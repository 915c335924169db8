"""Pins for the float64 oracle: hand-worked fixtures, closed forms, special
cases, brute force and an independent library routine.  CPU only.

Each test names the mistake class it guards against, so a plausible bug in
the oracle (dropped scale, wrong GQA index, transposed operand, wrong
causal alignment, missing max-subtraction, wrong combine weights) fails at
least one of them.  ``test_planted_mistakes_are_caught`` plants such bugs in
a copy of the oracle and checks that the pins reject every one.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A
from workloads import cu_seqlens, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

_SYMBOLS = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4),
            "ln10": math.log(10), "2ln3": 2 * math.log(3), "-inf": -math.inf}


def _num(x):
    if isinstance(x, str):
        return _SYMBOLS[x]
    if isinstance(x, list):
        return [_num(y) for y in x]
    return float(x)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _run_case(c, fwd=None):
    fwd = fwd or A.attention_forward
    q = np.array(_num(c["q"]))
    k = np.array(_num(c["k"]))
    v = np.array(_num(c["v"]))
    o, lse = fwd(q, k, v, cu_seqlens(c["lens_q"]), cu_seqlens(c["lens_k"]),
                 c["h_q"], c["h_kv"], c["scale"], c["causal"], c["window_left"],
                 c.get("descale_q", 1.0), c.get("descale_k", 1.0), c.get("descale_v", 1.0))
    return o, lse


# ---------------------------------------------------------------- fixtures

@pytest.mark.parametrize("case", _load("attention_worked_examples.json")["cases"],
                         ids=lambda c: c["name"])
def test_worked_examples(case):
    o, lse = _run_case(case)
    np.testing.assert_allclose(o, np.array(_num(case["o"])), rtol=0, atol=1e-12)
    exp_lse = np.array(_num(case["lse"]))
    assert np.array_equal(np.isinf(lse), np.isinf(exp_lse))
    fin = np.isfinite(exp_lse)
    np.testing.assert_allclose(lse[fin], exp_lse[fin], rtol=0, atol=1e-12)


# ------------------------------------------------------------ closed forms

def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("causal,wl", [(False, -1), (True, -1), (False, 5), (True, 0)])
def test_uniform_scores_give_mean_and_log_count(causal, wl):
    """Equal scores s: O = mean of allowed V rows, LSE = log(n) + s."""
    lq, lk, d = 7, 19, 5
    kvec = _rand((d,), 1)
    k = np.tile(kvec, (lk, 1))[:, None, :]
    q = _rand((lq, 1, d), 2)
    v = _rand((lk, 1, 3), 3)
    scale = 0.37
    o, lse = A.attention_forward(q, k, v, [0, lq], [0, lk], 1, 1, scale, causal, wl)
    for i in range(lq):
        lo, hi = A.allowed_key_range(i, lq, lk, causal, wl)
        s = scale * float(q[i, 0] @ kvec)
        if hi <= lo:
            assert lse[0, i] == -math.inf and np.all(o[i] == 0)
            continue
        np.testing.assert_allclose(o[i, 0], v[lo:hi, 0].mean(axis=0), atol=1e-12)
        assert abs(lse[0, i] - (math.log(hi - lo) + s)) < 1e-12


def test_one_hot_huge_score_selects_row():
    lk, d = 33, 4
    k = np.zeros((lk, 1, d))
    k[17, 0, 0] = 1.0
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 1e4
    v = _rand((lk, 1, 6), 4)
    o, lse = A.attention_forward(q, k, v, [0, 1], [0, lk], 1, 1, 1.0)
    np.testing.assert_allclose(o[0, 0], v[17, 0], atol=1e-12)
    assert abs(lse[0, 0] - 1e4) < 1e-9


def test_single_key_and_empty_and_no_queries():
    d = 3
    q = _rand((2, 2, d), 5)
    k = _rand((1, 2, d), 6)
    v = _rand((1, 2, 4), 7)
    # sequence 0: one query, one key; sequence 1: one query, no keys;
    # sequence 2: no queries, no keys.
    o, lse = A.attention_forward(q, k, v, [0, 1, 2, 2], [0, 1, 1, 1], 2, 2, 0.5)
    for h in range(2):
        np.testing.assert_allclose(o[0, h], v[0, h], atol=1e-14)
        assert abs(lse[h, 0] - 0.5 * float(q[0, h] @ k[0, h])) < 1e-12
        assert np.all(o[1, h] == 0) and lse[h, 1] == -math.inf
    assert o.shape == (2, 2, 4) and lse.shape == (2, 2)


def test_score_shift_moves_lse_only():
    """Adding c to every score (extra dim with k=1, q=c/scale) leaves O and
    shifts LSE by exactly c: LSE includes the scale, O is normalised."""
    lq, lk, d = 3, 11, 4
    q = _rand((lq, 1, d), 8)
    k = _rand((lk, 1, d), 9)
    v = _rand((lk, 1, 5), 10)
    scale, c = 0.3, 2.5
    o1, l1 = A.attention_forward(q, k, v, [0, lq], [0, lk], 1, 1, scale)
    q2 = np.concatenate([q, np.full((lq, 1, 1), c / scale)], axis=2)
    k2 = np.concatenate([k, np.ones((lk, 1, 1))], axis=2)
    o2, l2 = A.attention_forward(q2, k2, v, [0, lq], [0, lk], 1, 1, scale)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + c, atol=1e-12)


def test_large_scores_do_not_overflow():
    """Max-subtraction: scores near 1e3 would overflow exp without it."""
    q = np.full((1, 1, 1), 1000.0)
    k = np.array([[[1.0]], [[1.0 - 1e-3]]])
    v = np.array([[[1.0]], [[3.0]]])
    o, lse = A.attention_forward(q, k, v, [0, 1], [0, 2], 1, 1, 1.0)
    w1 = 1.0 / (1.0 + math.exp(-1.0))
    assert abs(o[0, 0, 0] - (w1 * 1 + (1 - w1) * 3)) < 1e-12
    assert abs(lse[0, 0] - (1000.0 + math.log(1 + math.exp(-1.0)))) < 1e-9


# ---------------------------------------------------- special-case reductions

def _sdpa_f64(q, k, v, scale, is_causal):
    """Independent library routine: torch SDPA in float64 on [h, L, d]."""
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2)
    vt = torch.from_numpy(v).permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=is_causal, scale=scale)
    s = scale * (qt @ kt.transpose(1, 2))
    if is_causal:
        L = s.shape[1]
        s = s.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), -math.inf)
    return o.permute(1, 0, 2).numpy(), torch.logsumexp(s, dim=2).numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(causal):
    L, h, d, dv = 37, 3, 16, 8
    q, k, v = _rand((L, h, d), 11), _rand((L, h, d), 12), _rand((L, h, dv), 13)
    scale = 1 / math.sqrt(d)
    o, lse = A.attention_forward(q, k, v, [0, L], [0, L], h, h, None, causal)
    o_ref, lse_ref = _sdpa_f64(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_noncausal_lq_ne_lk_matches_sdpa():
    lq, lk, h, d = 5, 23, 2, 8
    q, k, v = _rand((lq, h, d), 14), _rand((lk, h, d), 15), _rand((lk, h, d), 16)
    o, lse = A.attention_forward(q, k, v, [0, lq], [0, lk], h, h, 0.25)
    o_ref, lse_ref = _sdpa_f64(q, k, v, 0.25, False)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_gqa_equals_repeated_kv_heads():
    lq, lk, hq, hkv, d = 4, 9, 8, 2, 6
    q, k, v = _rand((lq, hq, d), 17), _rand((lk, hkv, d), 18), _rand((lk, hkv, d), 19)
    o, lse = A.attention_forward(q, k, v, [0, lq], [0, lk], hq, hkv, 0.4, True)
    k_rep = np.repeat(k, hq // hkv, axis=1)
    v_rep = np.repeat(v, hq // hkv, axis=1)
    o2, lse2 = A.attention_forward(q, k_rep, v_rep, [0, lq], [0, lk], hq, hq, 0.4, True)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)


def test_varlen_packing_equals_separate_sequences():
    lens_q, lens_k = [3, 0, 5, 1], [4, 2, 7, 0]
    hq, hkv, d = 4, 2, 5
    q = _rand((sum(lens_q), hq, d), 20)
    k = _rand((sum(lens_k), hkv, d), 21)
    v = _rand((sum(lens_k), hkv, 3), 22)
    cq, ck = cu_seqlens(lens_q).tolist(), cu_seqlens(lens_k).tolist()
    o, lse = A.attention_forward(q, k, v, cq, ck, hq, hkv, 0.5, True)
    for b in range(4):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        ob, lb = A.attention_forward(q[q0:q1], k[k0:k1], v[k0:k1], [0, q1 - q0],
                                     [0, k1 - k0], hq, hkv, 0.5, True)
        np.testing.assert_allclose(o[q0:q1], ob, atol=1e-14)
        np.testing.assert_allclose(lse[:, q0:q1], lb, atol=1e-14)


def test_window_covering_everything_equals_causal():
    L, d = 9, 4
    q, k, v = _rand((L, 1, d), 23), _rand((L, 1, d), 24), _rand((L, 1, d), 25)
    o1, l1 = A.attention_forward(q, k, v, [0, L], [0, L], 1, 1, 0.5, True, -1)
    o2, l2 = A.attention_forward(q, k, v, [0, L], [0, L], 1, 1, 0.5, False, L)
    np.testing.assert_allclose(o1, o2, atol=0)
    np.testing.assert_allclose(l1, l2, atol=0)


def test_window_is_banded_by_hand_count():
    """window (128, 0) on 300 keys: query i sees min(i'+1, 129) keys."""
    L = 300
    m = A.allowed_mask(L, L, False, 128)
    for i in range(L):
        assert m[i].sum() == min(i + 1, 129)
        assert m[i, i] and (i + 1 >= L or not m[i, i + 1])


def test_brute_force_tiny_scalar_loops():
    """Scalar Python loops (no numpy, no max-subtraction) on tiny shapes."""
    rng = np.random.default_rng(26)
    for trial in range(20):
        lq, lk, d, dv = rng.integers(1, 5), rng.integers(1, 5), rng.integers(1, 5), rng.integers(1, 4)
        causal = bool(trial % 2)
        q, k, v = rng.standard_normal((lq, 1, d)), rng.standard_normal((lk, 1, d)), rng.standard_normal((lk, 1, dv))
        o, lse = A.attention_forward(q, k, v, [0, lq], [0, lk], 1, 1, 0.7, causal)
        for i in range(lq):
            num = [0.0] * dv
            den = 0.0
            for j in range(lk):
                if causal and j > i + lk - lq:
                    continue
                e = math.exp(0.7 * sum(q[i, 0, t] * k[j, 0, t] for t in range(d)))
                den += e
                for c in range(dv):
                    num[c] += e * v[j, 0, c]
            if den == 0.0:
                assert lse[0, i] == -math.inf
                continue
            assert abs(lse[0, i] - math.log(den)) < 1e-12
            for c in range(dv):
                assert abs(o[i, 0, c] - num[c] / den) < 1e-12


# --------------------------------------------------------- split-KV identity

def test_split_invariance_any_partition():
    rng = np.random.default_rng(27)
    lens_q, lens_k = [2, 3, 1], [50, 7, 0]
    hq, hkv, d = 4, 2, 8
    q = rng.standard_normal((sum(lens_q), hq, d))
    k = rng.standard_normal((sum(lens_k), hkv, d))
    v = rng.standard_normal((sum(lens_k), hkv, 5))
    for causal, wl in [(False, -1), (True, -1), (False, 9)]:
        o_ref, l_ref = A.attention_forward(q, k, v, cu_seqlens(lens_q), cu_seqlens(lens_k), hq, hkv, 0.3, causal, wl)
        for ns in (1, 2, 3, 7):
            ranges = []
            cuts = [sorted(rng.integers(0, lk + 1, size=ns - 1).tolist()) for lk in lens_k]
            for s in range(ns):
                rs = []
                for b, lk in enumerate(lens_k):
                    edges = [0] + cuts[b] + [lk]
                    rs.append((edges[s], edges[s + 1]))
                ranges.append(rs)
            o, l = A.split_attention(q, k, v, cu_seqlens(lens_q), cu_seqlens(lens_k), hq, hkv,
                                     ranges, 0.3, causal, wl)
            np.testing.assert_allclose(o, o_ref, atol=1e-12)
            assert np.array_equal(np.isinf(l), np.isinf(l_ref))
            fin = np.isfinite(l_ref)
            np.testing.assert_allclose(l[fin], l_ref[fin], atol=1e-12)


def test_combine_closed_form_two_parts():
    """lse (ln 1, ln 3) -> weights 1/4, 3/4 and LSE = ln 4."""
    o_parts = np.array([[[4.0]], [[8.0]]])
    lse_parts = np.array([[0.0], [math.log(3)]])
    o, l = A.combine_partials(o_parts, lse_parts)
    assert abs(o[0, 0] - 7.0) < 1e-14 and abs(l[0] - math.log(4)) < 1e-14


def test_combine_with_empty_and_all_empty_splits():
    o_parts = np.array([[[np.nan], [np.nan]], [[2.0], [np.nan]], [[np.nan], [np.nan]]])
    o_parts = np.nan_to_num(o_parts, nan=0.0)
    lse_parts = np.array([[-np.inf, -np.inf], [1.5, -np.inf], [-np.inf, -np.inf]])
    o, l = A.combine_partials(o_parts, lse_parts)
    assert o[0, 0] == 2.0 and l[0] == 1.5
    assert o[1, 0] == 0.0 and l[1] == -np.inf


def test_combine_is_associative():
    rng = np.random.default_rng(28)
    o_p = rng.standard_normal((5, 6, 4))
    l_p = rng.standard_normal((5, 6)) * 10
    o_all, l_all = A.combine_partials(o_p, l_p)
    o_a, l_a = A.combine_partials(o_p[:2], l_p[:2])
    o_b, l_b = A.combine_partials(o_p[2:], l_p[2:])
    o2, l2 = A.combine_partials(np.stack([o_a, o_b]), np.stack([l_a, l_b]))
    np.testing.assert_allclose(o2, o_all, atol=1e-12)
    np.testing.assert_allclose(l2, l_all, atol=1e-12)


# ------------------------------------------------------------- input decode

def test_e4m3_decode_closed_form_all_codes():
    """Every e4m3 (fn) code widened by the oracle equals the format's closed
    form: sign, 4-bit exponent with bias 7, 3-bit mantissa, subnormals at
    exponent 0, and only S.1111.111 as NaN."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
    got = A.decode_inputs_f64(codes)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert math.isnan(got[c])
            continue
        val = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        assert got[c] == (-val if s else val)


def test_bf16_decode_is_exact_widening():
    x = torch.tensor([1.0, -2.5, 3.140625, 1e-3, 65504.0], dtype=torch.float32).to(torch.bfloat16)
    raw = x.view(torch.int16).numpy().astype(np.uint32) & 0xFFFF
    want = (raw << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    assert np.array_equal(A.decode_inputs_f64(x), want)


def test_fp8_workload_descale_reconstructs_draw():
    inp = make_inputs([3], [40], 2, 2, 16, 8, "e4m3", seed=3)
    deq = A.decode_inputs_f64(inp.k, inp.descale_k)
    assert np.abs(deq).max() <= 448.0 * inp.descale_k * (1 + 1e-7)
    assert np.abs(A.decode_inputs_f64(inp.k)).max() == 448.0


# ----------------------------------------------------------------- planner

@pytest.mark.parametrize("case", _load("planner_cases.json")["cases"],
                         ids=lambda c: "_".join(str(a) for a in c["args"]))
def test_planner_hand_cases(case):
    ns, units = oracle.plan_num_splits(*case["args"])
    assert (ns, units) == (case["ns"], case["units"]), case["derivation"]


@pytest.mark.parametrize("case", _load("split_ranges_cases.json")["cases"],
                         ids=lambda c: "_".join(str(a) for a in c["args"]))
def test_split_ranges_hand_cases(case):
    i_lo, i_hi, lq, lk, causal, wl, ns = case["args"]
    got = [list(oracle.tile_split_key_range(i_lo, i_hi, lq, lk, bool(causal), wl, ns, s))
           for s in range(ns)]
    assert got == case["ranges"], case["derivation"]


def test_split_ranges_partition_allowed_keys():
    """Splits of a tile partition exactly the union of its rows' allowed keys,
    in order, with min(ns, nb) non-empty parts whose block counts differ by
    at most one."""
    rng = np.random.default_rng(29)
    for _ in range(400):
        lq = int(rng.integers(1, 40))
        lk = int(rng.integers(0, 3000))
        causal = bool(rng.integers(0, 2))
        wl = int(rng.choice([-1, 0, 5, 128, 1000]))
        i_lo = int(rng.integers(0, lq))
        i_hi = int(rng.integers(i_lo, lq))
        ns = int(rng.integers(1, 20))
        union = set()
        for i in range(i_lo, i_hi + 1):
            lo, hi = A.allowed_key_range(i, lq, lk, causal, wl)
            union.update(range(lo, hi))
        got = []
        for s in range(ns):
            k0, k1 = oracle.tile_split_key_range(i_lo, i_hi, lq, lk, causal, wl, ns, s)
            if k1 > k0:
                got.append((k0, k1))
        covered = [j for k0, k1 in got for j in range(k0, k1)]
        assert covered == sorted(covered) and len(covered) == len(set(covered))
        if union:
            assert set(covered) == set(range(min(union), max(union) + 1))
            nb = -(-(max(union) + 1) // 128) - min(union) // 128
            assert len(got) == min(ns, nb)
            blocks = [oracle.split_block_range(nb, ns, s) for s in range(min(ns, nb))]
            sizes = [b1 - b0 for b0, b1 in blocks]
            assert max(sizes) - min(sizes) <= 1
        else:
            assert not got


def test_workspace_bytes():
    assert oracle.workspace_bytes(1, 1, 32, 128, 1) == 0
    assert oracle.workspace_bytes(1, 1, 32, 128, 9) == 4 * 9 * 32 * 129
    assert oracle.workspace_bytes(2, 70, 12, 128, 12) == 4 * 12 * 2 * 70 * 12 * 129


def test_default_scale_pins_head_dim():
    """Default scale uses the Q/K head dim for non-square shapes: a packed
    query side of 129 rows with head_dim 64 gives 1/8, and 129 vs 128 gives
    1/sqrt(128) -- never 1/sqrt(seqlen) or 1/sqrt(d_v)."""
    assert oracle.default_softmax_scale(64) == 0.125
    assert oracle.default_softmax_scale(128) == 1 / math.sqrt(128)
    assert oracle.default_softmax_scale(192) == 1 / math.sqrt(192)


# --------------------------------------------------------- planted mistakes

def _mutants():
    """Oracle variants with one plausible mistake each."""
    def drop_scale(q, k, v, cq, ck, hq, hkv, scale=None, causal=False, wl=-1, dq=1, dk=1, dv=1):
        return A.attention_forward(q, k, v, cq, ck, hq, hkv, 1.0, causal, wl, dq, dk, dv)

    def gqa_modulo(q, k, v, cq, ck, hq, hkv, scale=None, causal=False, wl=-1, dq=1, dk=1, dv=1):
        hkv_ = k.shape[1]
        idx = [h % hkv_ for h in range(hq)]
        return A.attention_forward(q, k[:, idx], v[:, idx], cq, ck, hq, hq, scale, causal, wl, dq, dk, dv)

    def top_left_causal(q, k, v, cq, ck, hq, hkv, scale=None, causal=False, wl=-1, dq=1, dk=1, dv=1):
        orig = A.allowed_key_range

        def tl(i, lq, lk, c, w):
            if not c and w < 0:
                return 0, lk
            hi = min(i + 1, lk)
            lo = max(0, i - w) if w >= 0 else 0
            return lo, max(lo, hi)
        A.allowed_key_range = tl
        try:
            return A.attention_forward(q, k, v, cq, ck, hq, hkv, scale, causal, wl, dq, dk, dv)
        finally:
            A.allowed_key_range = orig

    def lse_without_scale_shift(q, k, v, cq, ck, hq, hkv, scale=None, causal=False, wl=-1, dq=1, dk=1, dv=1):
        o, lse = A.attention_forward(q, k, v, cq, ck, hq, hkv, scale, causal, wl, dq, dk, dv)
        return o, np.where(np.isfinite(lse), lse / (scale if scale and scale > 0 else 1.0), lse)

    def ignore_dv(q, k, v, cq, ck, hq, hkv, scale=None, causal=False, wl=-1, dq=1, dk=1, dv=1):
        return A.attention_forward(q, k, v, cq, ck, hq, hkv, scale, causal, wl, dq, dk, 1.0)

    def scale_from_dv(q, k, v, cq, ck, hq, hkv, scale=None, causal=False, wl=-1, dq=1, dk=1, dv=1):
        if scale is None or scale <= 0:
            scale = 1 / math.sqrt(np.asarray(v).shape[2])
        return A.attention_forward(q, k, v, cq, ck, hq, hkv, scale, causal, wl, dq, dk, dv)

    def window_exclusive(q, k, v, cq, ck, hq, hkv, scale=None, causal=False, wl=-1, dq=1, dk=1, dv=1):
        return A.attention_forward(q, k, v, cq, ck, hq, hkv, scale, causal, wl - 1 if wl > 0 else wl, dq, dk, dv)

    return [drop_scale, gqa_modulo, top_left_causal, lse_without_scale_shift,
            ignore_dv, scale_from_dv, window_exclusive]


@pytest.mark.parametrize("mutant", _mutants(), ids=lambda f: f.__name__)
def test_planted_mistakes_are_caught(mutant):
    """At least one worked example rejects each planted mistake."""
    caught = False
    for c in _load("attention_worked_examples.json")["cases"]:
        o, lse = _run_case(c, fwd=mutant)
        exp_o = np.array(_num(c["o"]))
        exp_l = np.array(_num(c["lse"]))
        if o.shape != exp_o.shape or not np.allclose(o, exp_o, atol=1e-9):
            caught = True
            break
        if not np.array_equal(np.isinf(lse), np.isinf(exp_l)) or not np.allclose(
                lse[np.isfinite(exp_l)], exp_l[np.isfinite(exp_l)], atol=1e-9):
            caught = True
            break
    assert caught, mutant.__name__


# ------------------------------------------------------------- paged K/V

def test_gather_paged_kv_inverts_a_scatter():
    """Scatter packed K/V into pages in a shuffled order (written here as a
    separate procedure), then the oracle's gather must give the packed K/V
    back exactly, with the sequences' cu_seqlens."""
    rng = np.random.default_rng(30)
    lens = [5, 0, 17, 8]
    page_size, h, d = 4, 2, 3
    total = sum(lens)
    k = torch.from_numpy(rng.standard_normal((total, h, d)))
    v = torch.from_numpy(rng.standard_normal((total, h, d + 1)))
    need = [-(-n // page_size) for n in lens]
    num_pages = sum(need) + 2
    perm = rng.permutation(num_pages)
    kc = torch.full((num_pages, page_size, h, d), float("nan"), dtype=torch.float64)
    vc = torch.full((num_pages, page_size, h, d + 1), float("nan"), dtype=torch.float64)
    table = np.zeros((len(lens), max(need)), dtype=np.int32)
    used, start = 0, 0
    for b, n in enumerate(lens):
        for pi in range(need[b]):
            page = int(perm[used])
            used += 1
            table[b, pi] = page
            rows = range(pi * page_size, min(n, (pi + 1) * page_size))
            for r, j in enumerate(rows):
                kc[page, r] = k[start + j]
                vc[page, r] = v[start + j]
        start += n
    kg, vg, cu = oracle.gather_paged_kv(kc, vc, table, lens)
    assert torch.equal(kg, k) and torch.equal(vg, v)
    assert cu.tolist() == [0, 5, 5, 22, 30]


def test_gather_paged_kv_hand_case():
    """Page size 2, two sequences: seq 0 keys 0..2 in pages (3, 0); seq 1 key
    0 in page 1."""
    kc = torch.arange(4 * 2 * 1 * 1, dtype=torch.float64).view(4, 2, 1, 1)
    vc = -kc
    k, v, cu = oracle.gather_paged_kv(kc, vc, [[3, 0], [1, 0]], [3, 1])
    assert k.flatten().tolist() == [6.0, 7.0, 0.0, 2.0]
    assert v.flatten().tolist() == [-6.0, -7.0, -0.0, -2.0]
    assert cu.tolist() == [0, 3, 4]
