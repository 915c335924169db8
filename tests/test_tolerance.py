"""Pins of the output comparison rule (tests/tolerance.py), on the CPU.

The tolerance of the cutlass varlen page ("Tests": fp16/bf16 atol 1e-2)
bounds the value the kernel computes; the stored O is that value rounded to
the 16-bit output type.  These tests fix what the rule must accept and
reject, using torch's round-to-nearest-even conversions as the rounding."""

import numpy as np
import torch

from tolerance import excess, rounding_slack

ATOL = 1e-2


def _to(x, dtype):
    """float32 values rounded to a 16-bit type, back in float64."""
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(dtype).double().numpy()


def test_exact_value_rounded_to_bf16_can_miss_atol():
    # an oracle value of the edge workload (seed 55): its nearest bf16 value
    # is 0.0107 away, so no bf16 output meets atol 1e-2 against it unrounded
    r = -4.166917848620204
    o = _to([r], torch.bfloat16)[0]
    assert o == -4.15625
    assert abs(o - r) > ATOL
    assert excess(o, r, ATOL, 0.0, "bf16") <= 0


def test_rounded_reference_is_no_remedy():
    # 1e-3 apart, either side of the midpoint between two bf16 values on
    # [2, 4): they round to neighbours 2^-6 = 0.0156 apart, beyond 1e-2
    mid = 2.2421875
    a, b = _to([mid - 5e-4, mid + 5e-4], torch.bfloat16)
    assert abs(a - b) == 2.0 ** -6 > ATOL
    # the rule accepts either stored value against either exact value
    for o in (a, b):
        for r in (mid - 5e-4, mid + 5e-4):
            assert excess(o, r, ATOL, 0.0, "bf16") <= 0


def test_accepts_every_rounding_of_a_value_within_atol():
    rng = np.random.default_rng(0)
    for dtype, fmt in ((torch.bfloat16, "bf16"), (torch.float16, "fp16")):
        r = rng.uniform(-8.0, 8.0, 200_000)
        r = np.concatenate([r, rng.uniform(-1e-3, 1e-3, 20_000), [0.0, 4.0, -2.0, 1.0]])
        z = (r + rng.uniform(-ATOL, ATOL, r.size)).astype(np.float32).astype(np.float64)
        keep = np.abs(z - r) <= ATOL
        o = _to(z[keep], dtype)
        assert excess(o, r[keep], ATOL, 0.0, fmt).max() <= 0


def test_rejects_values_no_rounding_reaches():
    # 0.3 + 0.02: beyond atol plus half a bf16 gap near 0.32 (2^-9)
    o = _to([0.32], torch.bfloat16)[0]
    assert excess(o, 0.3, ATOL, 0.0, "bf16") > 0
    # one and two bf16 steps above 4.0 (2^-5 apart on [4, 8)): values within
    # 1e-2 of 4.0 round to 4.0 only
    assert excess(4.03125, 4.0, ATOL, 0.0, "bf16") > 0
    assert excess(4.0625, 4.0, ATOL, 0.0, "bf16") > 0
    # fp16 steps are 2^-8 on [4, 8): 4.0 + 2^-8 * 3 is 0.0117 from 4.0,
    # within 1e-2 + 2^-9
    assert excess(4.0 + 3 * 2.0 ** -8, 4.0, ATOL, 0.0, "fp16") <= 0
    assert excess(4.0 + 4 * 2.0 ** -8, 4.0, ATOL, 0.0, "fp16") > 0


def test_gap_below_a_power_of_two_is_half():
    # below 4.0 bf16 steps are 2^-6, above it 2^-5, so values from
    # 4 - 2^-7 = 3.9921875 up round to 4.0: an exact 3.985 has such values
    # within 1e-2 of it, an exact 3.980 has none (with the gap above 4.0
    # used on both sides the rule would accept it)
    assert rounding_slack(4.0, 3.985, "bf16") == 2.0 ** -7
    assert rounding_slack(4.0, 4.02, "bf16") == 2.0 ** -6
    assert excess(4.0, 3.985, ATOL, 0.0, "bf16") <= 0
    assert excess(4.0, 3.980, ATOL, 0.0, "bf16") > 0
    assert abs(4.0 - 3.980) <= ATOL + 2.0 ** -6
    # and the value that does round to 4.0 from below is accepted
    z = 4.0 - 2.0 ** -7 + 1e-6
    assert _to([z], torch.bfloat16)[0] == 4.0
    assert excess(4.0, z - ATOL, ATOL, 0.0, "bf16") <= 0


def test_slack_at_zero_and_subnormals():
    assert rounding_slack(0.0, 1e-3, "fp16") == 2.0 ** -25
    s = rounding_slack(2.0 ** -20, 0.0, "fp16")  # an fp16 subnormal
    assert s == 2.0 ** -25


def test_planted_mistakes_fail():
    # 4.0155 rounds to the bf16 value 4.0, 0.0155 away
    r = 4.0155
    o = _to([r], torch.bfloat16)[0]
    assert o == 4.0 and excess(o, r, ATOL, 0.0, "bf16") <= 0
    # no rounding slack at all: the correctly rounded exact value fails
    assert np.abs(o - r) - ATOL > 0
    # the fp16 gap used for a bf16 output: it fails too
    assert excess(o, r, ATOL, 0.0, "fp16") > 0
