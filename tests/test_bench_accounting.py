"""The benchmark's roofline numerators, checked on the CPU: the attended
(query, key) pairs behind the prefill FLOP count against closed forms and
against the oracle's own mask, the metric's bytes for the long decode, and
the number of input copies that keeps a replayed graph's inputs out of L2."""

import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from workloads import PREFILL_LENGTHS, cu_seqlens  # noqa: E402


def _seqs(lens_q, lens_k):
    return SimpleNamespace(cu_seqlens_q=cu_seqlens(lens_q), cu_seqlens_k=cu_seqlens(lens_k))


def test_prefill_pairs_closed_forms():
    """No mask: sum of L^2; causal with Lq = Lk: sum of L(L+1)/2."""
    inp = _seqs(PREFILL_LENGTHS, PREFILL_LENGTHS)
    assert bench.attended_pairs(inp, False) == sum(n * n for n in PREFILL_LENGTHS) == 42_991_616
    assert bench.attended_pairs(inp, True) == sum(n * (n + 1) // 2 for n in PREFILL_LENGTHS) == 21_504_000
    # 2 (d_qk + d_v) FLOPs per pair and query head
    assert bench.flops(SimpleNamespace(**vars(inp), d_qk=128, d_v=128, h_q=16), True) == \
        512 * 16 * 21_504_000


@pytest.mark.parametrize("seed", range(4))
def test_pairs_match_the_oracle_mask(seed):
    """Random Lq != Lk (bottom-right causal rows may see no key at all)."""
    rng = np.random.default_rng(seed)
    lens_q = [int(x) for x in rng.integers(0, 200, size=5)]
    lens_k = [int(x) for x in rng.integers(0, 200, size=5)]
    inp = _seqs(lens_q, lens_k)
    for causal in (False, True):
        want = sum(int(oracle.allowed_mask(lq, lk, causal, -1).sum())
                   for lq, lk in zip(lens_q, lens_k))
        assert bench.attended_pairs(inp, causal) == want


def test_long_decode_metric_bytes():
    """K + V + Q + O at storage width for B=1, K=131072, H=32/32, D=128, bf16."""
    inp = SimpleNamespace(k=torch.empty((131072, 32, 128), device="meta"),
                          q=torch.empty((1, 32, 128), device="meta"),
                          h_kv=32, h_q=32, d_qk=128, d_v=128, dtype="bf16")
    assert bench.metric_bytes(inp) == 2 * 131072 * 32 * 128 * 2 + 32 * 128 * 2 * 2 == 2_147_500_032


def test_input_copies_keep_l2_cold():
    """Inputs of 256 MB (twice the L2) or more run as they are; smaller ones
    rotate over enough copies that 256 MB is read between two uses of one."""
    big = bench.L2_FLUSH_BYTES
    assert bench.copies_for(big) == 1 and bench.copies_for(4 * big) == 1
    fp8_prefix = 63_075_856
    n = bench.copies_for(fp8_prefix)
    assert n == 6 and (n - 1) * fp8_prefix >= big
    for size in (1, 1000, 10 << 20, 100 << 20, big - 1):
        n = bench.copies_for(size)
        assert (n - 1) * size >= big or n == 512
