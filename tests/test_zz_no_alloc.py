"""fa_fwd_splitkv_noalloc: the forward entry point for callers that cannot
allocate device memory (code running under a runtime that owns every device
allocation, a plugin without an allocator handle, or a path where
cudaMalloc's device synchronisation is not allowed).  It takes its split
workspace from a fixed array inside the library instead of from the caller.

Each case runs the existing entry point fa_fwd_splitkv_ex with a workspace
the test allocates, then calls the no-alloc entry point twice in a row
through the C ABI: the second call finds the first call's leftovers in the
shared array and must still agree.  Both calls are compared with the
float64 oracle at the parity tolerances (cutlass varlen page, "Tests":
O atol 1e-2, LSE atol 1e-3) and with the workspace path.

This file is collected last so that a stop at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""

import numpy as np
import pytest
import torch

import split_kv_flashattention_gb300 as fa
from gpu_harness import assert_close, reference
from workloads import make_inputs, workload

pytestmark = pytest.mark.gpu

O_ATOL, LSE_ATOL = 1e-2, 1e-3


def _to_dev(inp):
    dev = torch.device("cuda:0")
    return (inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens_q.to(dev),
            inp.cu_seqlens_k.to(dev))


def _outputs(inp, q):
    out = torch.full((q.shape[0], inp.h_q, inp.d_v), float("nan"), dtype=q.dtype, device=q.device)
    lse = torch.full((inp.h_q, q.shape[0]), float("nan"), dtype=torch.float32, device=q.device)
    return out, lse


CASES = {
    "decode_mha_7_splits": (lambda: workload("long_decode", kv=5000, h=4), dict(num_splits=7)),
    "gqa_varlen_auto_splits": (
        lambda: make_inputs([1] * 6, [2000, 17, 0, 3000, 1, 999], 16, 4, 128, 128, "bf16", seed=11),
        dict(num_splits=0)),
    "causal_prefix_3_splits": (
        lambda: make_inputs([3, 40, 1], [200, 300, 64], 8, 2, 128, 128, "bf16", seed=12),
        dict(num_splits=3, causal=True)),
    # one split: the persistent prefill kernel, its tile counter in the array
    "causal_prefill_persistent": (
        lambda: make_inputs([700, 300, 520], [700, 300, 520], 4, 2, 128, 128, "bf16", seed=13),
        dict(num_splits=1, causal=True, kernel=fa.FA_KID_UMMA2_PERSISTENT)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_caller_workspace_path(name):
    make, kw = CASES[name]
    inp = make()
    q, k, v, cq, ck = _to_dev(inp)

    ref_out, ref_lse = _outputs(inp, q)
    ns = kw.get("num_splits", 0)
    nbytes = fa.fa_fwd_splitkv_workspace_size(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv,
                                              inp.d_v, ns)
    assert 0 < nbytes <= fa.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
    fa.fa_fwd_splitkv_ex(q, k, v, cq, ck, inp.max_seqlen_q, ref_out, ref_lse, ws,
                         causal=kw.get("causal", False), num_splits=ns)
    torch.cuda.synchronize()
    ref_o = ref_out.float().cpu().numpy()
    ref_l = ref_lse.cpu().numpy()
    assert np.isfinite(ref_o).all()
    o_oracle, l_oracle = reference(inp, 0.0, kw.get("causal", False))
    assert_close(inp, ref_o, ref_l, o_oracle, l_oracle)

    for call in range(2):
        out, lse = _outputs(inp, q)
        fa.fa_fwd_splitkv_noalloc(q, k, v, cq, ck, inp.max_seqlen_q, out, lse,
                                  causal=kw.get("causal", False), num_splits=ns)
        if "kernel" in kw:
            assert fa.fa_debug_last_kernel() == kw["kernel"]
        torch.cuda.synchronize()
        assert fa.fa_get_device_error(clear=True) == 0
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.isfinite(o).all(), f"call {call}: unwritten or non-finite output"
        assert_close(inp, o, l, o_oracle, l_oracle)
        assert np.abs(o - ref_o).max() <= O_ATOL, f"call {call}"
        assert np.array_equal(np.isneginf(l), np.isneginf(ref_l)), f"call {call}"
        fin = np.isfinite(ref_l)
        assert np.abs(l[fin] - ref_l[fin]).max() <= LSE_ATOL, f"call {call}"


def test_noalloc_rejects_problems_larger_than_its_scratch():
    """A workspace need above the fixed array is refused before any launch."""
    inp = workload("long_decode", kv=256, h=4)
    q, k, v, cq, ck = _to_dev(inp)
    out, lse = _outputs(inp, q)
    max_q = 5000  # 16 splits * 5000 slots * 4 heads * 129 floats > 8 MiB
    assert fa.fa_fwd_splitkv_workspace_size(1, max_q, 4, 4, 128, 16) > fa.NOALLOC_SCRATCH_BYTES
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_splitkv_noalloc(q, k, v, cq, ck, max_q, out, lse, num_splits=16)
    assert e.value.status == -3
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
