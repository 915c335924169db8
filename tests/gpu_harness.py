"""Shared helpers of the GPU parity tests: run the C-ABI path on seeded
inputs and compare with the float64 oracle element by element."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import split_kv_flashattention_gb300 as fa
from tolerance import excess

# Tolerances: cutlass "Adds variable sequence lengths to the Hopper CuTe DSL
# FMHA example", section "Tests" (fp16/bf16 atol 1e-2; fp8 atol 0.13,
# rtol 1e-5); LSE atol 1e-3 for every dtype.  They bound the value the
# kernel computes; the stored 16-bit O is that value rounded to its type
# (tests/tolerance.py).
TOL = {"bf16": (1e-2, 0.0), "fp16": (1e-2, 0.0), "e4m3": (0.13, 1e-5)}
LSE_ATOL = 1e-3
# output type of each input type when the call leaves it to the library
OUT_FMT = {"bf16": "bf16", "fp16": "fp16", "e4m3": "bf16"}


def device():
    return torch.device("cuda:0")


def run_gpu(inp, scale=0.0, causal=False, window_left=-1, num_splits=0, flags=0,
            with_lse=True, guard_rows=0, out_dtype=None, ws_guard=0, out_offset=0, ws_offset=0):
    """Runs fa_fwd_splitkv_ex on `inp` (workloads.Inputs).  Output rows past
    the packed queries (guard_rows of them) and ws_guard floats past the
    workspace are filled with NaN sentinels and must stay untouched.  O starts
    out_offset bytes into its allocation, the workspace ws_offset bytes into
    its own; the bytes before either must stay NaN."""
    dev = device()
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    cq, ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev)
    total_q = q.shape[0] + guard_rows
    if guard_rows:
        qpad = torch.zeros((total_q,) + tuple(q.shape[1:]), dtype=q.dtype, device=dev)
        qpad[: q.shape[0]] = q
        q = qpad
    if out_dtype is None:
        out_dtype = torch.bfloat16 if inp.dtype == "e4m3" else q.dtype
    n_out = total_q * inp.h_q * inp.d_v
    pre = out_offset // torch.empty((), dtype=out_dtype).element_size()
    out_buf = torch.full((pre + n_out,), float("nan"), dtype=out_dtype, device=dev)
    out = out_buf[pre:].view(total_q, inp.h_q, inp.d_v)
    lse = (torch.full((inp.h_q, total_q), float("nan"), dtype=torch.float32, device=dev)
           if with_lse else None)
    ns_bytes = fa.fa_fwd_splitkv_workspace_size(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv,
                                               inp.d_v, num_splits)
    ws = ws_buf = None
    ws_pre = ws_offset // 4
    if ns_bytes:
        ws_buf = torch.full((ws_pre + ns_bytes // 4 + ws_guard,), float("nan"), dtype=torch.float32,
                            device=dev)
        ws = ws_buf[ws_pre:]
    dq = dk = dv = None
    if inp.dtype == "e4m3":
        dq = torch.tensor([inp.descale_q], dtype=torch.float32, device=dev)
        dk = torch.tensor([inp.descale_k], dtype=torch.float32, device=dev)
        dv = torch.tensor([inp.descale_v], dtype=torch.float32, device=dev)
    fa.fa_fwd_splitkv_ex(q, k, v, cq, ck, inp.max_seqlen_q, out, lse, ws, scale, causal,
                         window_left, num_splits, dq, dk, dv, flags)
    torch.cuda.synchronize()
    err = fa.fa_get_device_error(clear=True)
    assert err == 0, fa.fa_status_string(err)
    if ws is not None and ws_guard:
        assert torch.isnan(ws[ns_bytes // 4:]).all(), "workspace guard overwritten"
    if pre:
        assert torch.isnan(out_buf[:pre].float()).all(), "bytes before O overwritten"
    if ws_pre and ws_buf is not None:
        assert torch.isnan(ws_buf[:ws_pre]).all(), "bytes before the workspace overwritten"
    return out.float().cpu().numpy(), (lse.cpu().numpy() if lse is not None else None)


def reference(inp, scale=0.0, causal=False, window_left=-1, heads=None):
    """Oracle O [total_q, h_q, d_v] and LSE [h_q, total_q] (optionally for a
    subset of query heads, computed from the matching KV heads only)."""
    if heads is None:
        return oracle.attention_forward(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k,
                                        inp.h_q, inp.h_kv, scale, causal, window_left,
                                        inp.descale_q, inp.descale_k, inp.descale_v)
    group = inp.h_q // inp.h_kv
    outs, lses = {}, {}
    for h in heads:
        kh = h // group
        o, l = oracle.attention_forward(inp.q[:, h:h + 1], inp.k[:, kh:kh + 1],
                                        inp.v[:, kh:kh + 1], inp.cu_seqlens_q, inp.cu_seqlens_k,
                                        1, 1, scale, causal, window_left, inp.descale_q,
                                        inp.descale_k, inp.descale_v)
        outs[h], lses[h] = o[:, 0], l[0]
    return outs, lses


def assert_close(inp, out, lse, o_ref, l_ref, heads=None):
    atol, rtol = TOL[inp.dtype]
    tq = inp.q.shape[0]
    hs = range(inp.h_q) if heads is None else heads
    for h in hs:
        o_h = out[:tq, h]
        r_h = o_ref[:, h] if heads is None else o_ref[h]
        assert np.isfinite(o_h).all(), f"head {h}: non-finite or unwritten output"
        err = excess(o_h, r_h, atol, rtol, OUT_FMT[inp.dtype])
        assert err.max() <= 0, (f"head {h}: max|dO|={np.abs(o_h - r_h).max():.4g}, "
                                f"beyond the tolerance by {err.max():.3g}")
        if lse is not None:
            l_h = lse[h, :tq]
            lr = l_ref[h] if heads is None else l_ref[h]
            assert np.array_equal(np.isneginf(l_h), np.isneginf(lr)), f"head {h}: -inf rows differ"
            fin = np.isfinite(lr)
            assert np.isfinite(l_h[fin]).all()
            if fin.any():
                d = np.abs(l_h[fin] - lr[fin]).max()
                assert d <= LSE_ATOL, f"head {h}: max|dLSE|={d:.4g}"


def run_gpu_paged(inp, scale=0.0, causal=False, window_left=-1, num_splits=0, flags=0):
    """fa_fwd_splitkv_paged on workloads.PagedInputs; returns (O, LSE)."""
    dev = device()
    q = inp.q.to(dev)
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    cq = inp.cu_seqlens_q.to(dev)
    sk, bt = inp.seqlens_k.to(dev), inp.block_table.to(dev)
    out_dtype = torch.bfloat16 if inp.dtype == "e4m3" else q.dtype
    out = torch.full((q.shape[0], inp.h_q, inp.d_v), float("nan"), dtype=out_dtype, device=dev)
    lse = torch.full((inp.h_q, q.shape[0]), float("nan"), dtype=torch.float32, device=dev)
    nbytes = fa.fa_fwd_splitkv_workspace_size(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv,
                                             inp.d_v, num_splits)
    ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device=dev) if nbytes else None
    dq = dk = dv = None
    if inp.dtype == "e4m3":
        dq = torch.tensor([inp.descale_q], dtype=torch.float32, device=dev)
        dk = torch.tensor([inp.descale_k], dtype=torch.float32, device=dev)
        dv = torch.tensor([inp.descale_v], dtype=torch.float32, device=dev)
    fa.fa_fwd_splitkv_paged(q, kc, vc, cq, sk, bt, inp.max_seqlen_q, out, lse, ws, scale, causal,
                            window_left, num_splits, dq, dk, dv, flags=flags)
    torch.cuda.synchronize()
    err = fa.fa_get_device_error(clear=True)
    assert err == 0, fa.fa_status_string(err)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def reference_paged(inp, scale=0.0, causal=False, window_left=-1):
    """The oracle on the paged cache gathered back into packed K/V."""
    k, v, cu_k = oracle.gather_paged_kv(inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens_k)
    return oracle.attention_forward(inp.q, k, v, inp.cu_seqlens_q, cu_k, inp.h_q, inp.h_kv,
                                    scale, causal, window_left, inp.descale_q, inp.descale_k,
                                    inp.descale_v)
