"""The host-buffer entry point fa_fwd_splitkv_host: its device-buffer size and
argument checks on the CPU; on the GPU, its results against the oracle and,
bit for bit, against the device-buffer call on the same inputs."""

import ctypes

import numpy as np
import pytest
import torch

import split_kv_flashattention_gb300 as fa
from gpu_harness import assert_close, reference, run_gpu
from workloads import make_inputs

FA_ERR_INVALID_ARG, FA_ERR_WORKSPACE = -1, -3


def _align(x):
    return (x + 255) // 256 * 256


def test_buffer_size_is_the_sum_of_aligned_regions():
    """Q, K, V, the two offset arrays, the descales, O, LSE and the split
    workspace, each rounded up to 256 bytes (explicit split count: host only)."""
    b, tq, tk, mq, hq, hkv, dqk, dv, ns = 3, 70, 5000, 40, 8, 2, 192, 128, 4
    ws = fa.fa_fwd_splitkv_workspace_size(b, mq, hq, hkv, dv, ns)
    assert ws == 4 * ns * b * mq * hq * (dv + 1)
    for in_dt, es in ((torch.bfloat16, 2), (torch.float8_e4m3fn, 1)):
        want = (_align(tq * hq * dqk * es) + _align(tk * hkv * dqk * es) + _align(tk * hkv * dv * es)
                + 2 * _align((b + 1) * 4) + _align(12) + _align(tq * hq * dv * 2)
                + _align(hq * tq * 4) + _align(ws))
        assert fa.fa_fwd_splitkv_host_buffer_size(b, tq, tk, mq, hq, hkv, dqk, dv, in_dt,
                                                  torch.bfloat16, ns) == want


def test_buffer_size_rejects_invalid_sizes():
    bad = [dict(h_q=6, h_kv=4), dict(num_splits=129), dict(total_k=-1), dict(d_v=0)]
    for kw in bad:
        args = dict(batch=1, total_q=1, total_k=10, max_seqlen_q=1, h_q=4, h_kv=4, d_qk=128,
                    d_v=128, in_dtype=torch.bfloat16, out_dtype=torch.bfloat16, num_splits=2)
        args.update(kw)
        assert fa.fa_fwd_splitkv_host_buffer_size(**args) == 0, kw


def test_host_call_refuses_a_missing_or_misaligned_buffer_before_any_copy():
    """Checked on the host before any CUDA call, so no device is needed."""
    lib = fa.library()
    q = np.zeros((1, 4, 128), dtype=np.uint16)
    k = np.zeros((64, 4, 128), dtype=np.uint16)
    cq = np.array([0, 1], dtype=np.int32)
    ck = np.array([0, 64], dtype=np.int32)
    out = np.zeros((1, 4, 128), dtype=np.uint16)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    need = fa.fa_fwd_splitkv_host_buffer_size(1, 1, 64, 1, 4, 4, 128, 128, torch.bfloat16,
                                              torch.bfloat16, 2)

    def call(buf, nbytes):
        return lib.fa_fwd_splitkv_host(vp(q), vp(k), vp(k), vp(cq), vp(ck), 1, 1, 64, 1, 4, 4, 128,
                                       128, 0.0, 0, -1, 2, vp(out), None, buf, nbytes, 0, 0, None,
                                       None, None, 0, None)

    assert call(None, need) == FA_ERR_INVALID_ARG
    assert call(ctypes.c_void_p(4096 + 16), need) == FA_ERR_INVALID_ARG  # not 256-byte aligned
    assert call(ctypes.c_void_p(4096), need - 1) == FA_ERR_WORKSPACE


def _host_call(inp, causal=False, num_splits=0, with_lse=True):
    """fa_fwd_splitkv_host on pinned copies of `inp`; returns (O, LSE)."""
    dev = torch.device("cuda:0")
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    q, k, v = pin(inp.q), pin(inp.k), pin(inp.v)
    cq, ck = pin(inp.cu_seqlens_q), pin(inp.cu_seqlens_k)
    out_dtype = torch.bfloat16 if inp.dtype == "e4m3" else q.dtype
    out = torch.full((q.shape[0], inp.h_q, inp.d_v), float("nan"), dtype=out_dtype).pin_memory()
    lse = (torch.full((inp.h_q, q.shape[0]), float("nan"), dtype=torch.float32).pin_memory()
           if with_lse else None)
    dsc = [None] * 3
    if inp.dtype == "e4m3":
        dsc = [torch.tensor([d], dtype=torch.float32) for d in
               (inp.descale_q, inp.descale_k, inp.descale_v)]
    nbytes = fa.fa_fwd_splitkv_host_buffer_size(
        inp.batch, q.shape[0], k.shape[0], inp.max_seqlen_q, inp.h_q, inp.h_kv, q.shape[2],
        inp.d_v, q.dtype, out_dtype, num_splits)
    assert nbytes > 0
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    fa.fa_fwd_splitkv_host(q, k, v, cq, ck, inp.max_seqlen_q, out, lse, buf, causal=causal,
                           num_splits=num_splits, descale_q=dsc[0], descale_k=dsc[1],
                           descale_v=dsc[2], stream=s)
    s.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    return out.float().numpy(), (lse.numpy() if with_lse else None)


CASES = {
    "gqa_decode": (lambda: make_inputs([1, 1, 1], [2500, 700, 4100], 16, 4, 128, 128, "bf16",
                                       seed=90), False),
    "fp8_prefix": (lambda: make_inputs([70], [3000], 4, 4, 192, 128, "e4m3", seed=91), False),
    "prefill_causal": (lambda: make_inputs([300, 129], [300, 129], 4, 4, 128, 128, "fp16",
                                           seed=92), True),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(CASES))
def test_host_entry_matches_oracle_and_device_call(case):
    make, causal = CASES[case]
    inp = make()
    ns = 1 if case == "prefill_causal" else 0
    out, lse = _host_call(inp, causal=causal, num_splits=ns)
    o_ref, l_ref = reference(inp, 0.0, causal)
    assert_close(inp, out, lse, o_ref, l_ref)
    out_d, lse_d = run_gpu(inp, causal=causal, num_splits=ns)
    assert np.array_equal(out, out_d, equal_nan=True) and np.array_equal(lse, lse_d, equal_nan=True)


@pytest.mark.gpu
def test_host_entry_without_lse():
    inp = CASES["gqa_decode"][0]()
    out, _ = _host_call(inp, with_lse=False)
    o_ref, l_ref = reference(inp)
    assert_close(inp, out, None, o_ref, l_ref)
