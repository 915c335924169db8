"""Oracle for split-KV flash attention: plain, slow, CPU-only, float64.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this package.  The only permitted users are ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``.  It shares no code with the CUDA library (no kernels,
headers, helpers, tables or constants); the two meet only at the seeded input
generators in ``workloads.py``, which contain none of the method's arithmetic.

Sources (pages as titled; sections named, not lines):

* [FA4] flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference"
  -- split-KV forward with a single 128-row query tile, sections
  "Benchmarks" (the num_splits sweep) and the description.
* [AITER] ROCm aiter PR "[FlyDSL] Enable FP8 FMHA split-K for short
  cached-prefix queries" -- split-K with automatic/explicit split selection,
  return_lse, an fp32 split workspace and the attention + split-combine pair.
* [CUTLASS] NVIDIA cutlass "Adds variable sequence lengths to the Hopper CuTe
  DSL FMHA example" -- sections "Interface" (cu_seqlens, packed layout),
  "Implementation" (tile skipping, tails, masks, default softmax scale),
  "Tests" (length matrix, masks, tolerances).

Modules:

* ``attention``  -- the definition softmax(Q K^T * scale) V with its
  log-sum-exp, per packed varlen sequence, with the no-mask, bottom-right
  causal and sliding-window masks; partial attention over a key sub-range and
  the LSE-weighted combine of partials (the split-KV identity).
* ``planner``    -- the integer split planner and per-split key ranges, the
  host/device rule that the library must reproduce bit for bit.
* ``paged``      -- the paged K/V layout as plain indexing (gather pages back
  into packed K/V), for the paged-cache entry point.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, hand-worked fixtures in ``tests/golden/``, brute force
and an independent library routine (torch scaled_dot_product_attention in
float64).  No function is "parity unpinned".
"""

from .attention import (  # noqa: F401
    NEG_INF,
    allowed_key_range,
    allowed_mask,
    attention_forward,
    combine_partials,
    decode_inputs_f64,
    default_softmax_scale,
    partial_attention,
    split_attention,
)
from .paged import gather_paged_kv  # noqa: F401
from .planner import (  # noqa: F401
    BLOCK_N,
    M_TILE,
    MAX_SPLITS,
    plan_num_splits,
    split_block_range,
    tile_key_range,
    tile_split_key_range,
    workspace_bytes,
)
