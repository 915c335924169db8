"""How a 16-bit output is compared with the float64 oracle.

cutlass "Adds variable sequence lengths to the Hopper CuTe DSL FMHA example",
section "Tests", checks O against a PyTorch reference with atol 1e-2 for
fp16/bf16 (0.13 for fp8, rtol 1e-5).  The kernels store O in a 16-bit type,
and the oracle's O is float64.  Rounding alone separates the two: bf16 keeps
8 significant bits, so on [4, 8) its values are 2^-5 apart and the exact
result, correctly rounded, can land 2^-6 = 0.0156 from itself, beyond 1e-2.
Comparing against the oracle rounded to the output type does not help
either: two values 1e-3 apart on either side of a rounding midpoint on
[2, 4) round to bf16 neighbours 0.0156 apart.

Reading used by the tests: the tolerance bounds the value the kernel
computes, and the stored output is that value rounded to the output type.
So a stored value o is accepted against the oracle's r when some y with
|y - r| <= atol + rtol |r| rounds to o, that is when o lies within the
tolerance plus half the gap between o and its neighbour on r's side.
"""

from __future__ import annotations

import numpy as np

# (significant bits, smallest normal exponent) of the 16-bit output types
FORMATS = {"bf16": (8, -126), "fp16": (11, -14)}


def rounding_slack(o, r, fmt: str) -> np.ndarray:
    """Half the gap between each stored value o (a value of the format
    `fmt`, held in float32/64) and its neighbour on the side of r: the
    farthest an exact value that rounds to o can lie from o towards r."""
    bits, emin = FORMATS[fmt]
    o = np.asarray(o, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    a = np.abs(o)
    m, e = np.frexp(a)  # a = m * 2^e, m in [0.5, 1)
    ulp = np.ldexp(1.0, np.maximum(e - bits, emin + 1 - bits))
    # from a power of two towards zero the next value is half as far
    ulp = np.where((m == 0.5) & (np.abs(r) < a) & (e - 1 > emin), ulp / 2, ulp)
    ulp = np.where(a == 0, np.ldexp(1.0, emin + 1 - bits), ulp)
    return 0.5 * ulp


def excess(o, r, atol: float, rtol: float, fmt: str | None) -> np.ndarray:
    """How far each |o - r| lies beyond the allowed error (<= 0 passes).
    fmt None: o is compared as it is (no output rounding)."""
    o = np.asarray(o, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    allow = atol + rtol * np.abs(r)
    if fmt is not None:
        allow = allow + rounding_slack(o, r, fmt)
    return np.abs(o - r) - allow
