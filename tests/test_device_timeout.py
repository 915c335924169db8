"""The bounded-wait path on the GPU, without a fault: a wait that nothing
completes gives up, the device error word reports FA_ERR_DEVICE_TIMEOUT, the
forward kernels skip their work while it is set, and after clearing it the
context computes correctly again."""

import time

import numpy as np
import pytest
import torch

import split_kv_flashattention_gb300 as fa
from gpu_harness import assert_close, reference, run_gpu
from workloads import workload

FA_ERR_DEVICE_TIMEOUT = -5


@pytest.mark.gpu
def test_bounded_wait_times_out_and_context_survives():
    dev = torch.device("cuda:0")
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    try:
        t0 = time.monotonic()
        fa.fa_debug_wait_timeout(50)
        torch.cuda.synchronize()
        elapsed = time.monotonic() - t0
        assert 0.04 <= elapsed < 5.0
        assert fa.fa_get_device_error() == FA_ERR_DEVICE_TIMEOUT

        # While the timeout is recorded, the forward kernels leave at once:
        # the outputs keep their sentinels and the error stays.
        inp = workload("tiny_decode", device=dev)
        q, k, v = inp.q, inp.k, inp.v
        cq, ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev)
        out = torch.full((q.shape[0], inp.h_q, inp.d_v), float("nan"), dtype=q.dtype, device=dev)
        lse = torch.full((inp.h_q, q.shape[0]), float("nan"), dtype=torch.float32, device=dev)
        nbytes = fa.fa_fwd_splitkv_workspace_size(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv,
                                                 inp.d_v, 4)
        ws = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
        fa.fa_fwd_splitkv_ex(q, k, v, cq, ck, inp.max_seqlen_q, out, lse, ws, 0.0, False, -1, 4)
        torch.cuda.synchronize()
        assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
        assert fa.fa_get_device_error() == FA_ERR_DEVICE_TIMEOUT
    finally:
        fa.fa_get_device_error(clear=True)

    # Cleared: the same context computes correctly.
    inp = workload("tiny_decode")
    out, lse = run_gpu(inp, num_splits=4)
    o_ref, l_ref = reference(inp)
    assert_close(inp, out, lse, o_ref, l_ref)
