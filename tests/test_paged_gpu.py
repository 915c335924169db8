"""GPU parity of the paged K/V entry point against the oracle (pages
gathered back into packed K/V)."""

import numpy as np
import pytest
import torch

import split_kv_flashattention_gb300 as fa
from gpu_harness import assert_close, reference, reference_paged, run_gpu_paged
from workloads import Inputs, gqa_decode_lengths, make_paged_inputs

pytestmark = pytest.mark.gpu

KERNELS = [fa.FA_KERNEL_SIMT, fa.FA_KERNEL_UMMA, fa.FA_KERNEL_UMMA2]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("page_size", [32, 64, 128, 256])
def test_paged_decode_gqa(kernel, page_size):
    """Decode (one query per sequence), GQA 4:2, ragged key counts including
    an empty and a one-key sequence, shuffled pages, automatic splits."""
    inp = make_paged_inputs([1] * 5, [1000, 0, 1, 2049, 300], 8, 2, 128, 128, page_size, seed=20)
    out, lse = run_gpu_paged(inp, flags=kernel)
    o_ref, l_ref = reference_paged(inp)
    assert_close(inp, out, lse, o_ref, l_ref)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("mask", ["none", "causal", "window"])
def test_paged_prefix_masks(kernel, mask):
    """Several queries per sequence (cached prefix), masks, 3 splits."""
    causal = mask == "causal"
    wl = 100 if mask == "window" else -1
    inp = make_paged_inputs([3, 40, 130], [700, 333, 1290], 4, 2, 128, 128, 64, seed=21)
    out, lse = run_gpu_paged(inp, causal=causal, window_left=wl, num_splits=3, flags=kernel)
    o_ref, l_ref = reference_paged(inp, 0.0, causal, wl)
    assert_close(inp, out, lse, o_ref, l_ref)


@pytest.mark.parametrize("kernel", [fa.FA_KERNEL_SIMT, fa.FA_KERNEL_UMMA])
@pytest.mark.parametrize("d_qk,page_size", [(192, 32), (192, 64), (128, 128)])
def test_paged_fp8(kernel, d_qk, page_size):
    """e4m3 K/V pages (d_v = 128) with a few queries per sequence, ragged key
    counts and shuffled pages; bf16 output against the oracle."""
    inp = make_paged_inputs([1, 3, 70], [1500, 333, 2100], 6, 6, d_qk, 128, page_size,
                            dtype="e4m3", seed=25)
    out, lse = run_gpu_paged(inp, num_splits=4, flags=kernel)
    o_ref, l_ref = reference_paged(inp)
    assert_close(inp, out, lse, o_ref, l_ref)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype,d", [("fp16", 64), ("bf16", 256)])
def test_paged_other_head_dims(kernel, dtype, d):
    """Head dims 64 (fp16) and 256 (bf16) through the page cursor, causal."""
    if kernel == fa.FA_KERNEL_UMMA2 and d == 256:
        pytest.skip("the two-tile kernel takes head dims up to 128")
    inp = make_paged_inputs([2, 1, 9], [900, 64, 1700], 8, 2, d, d, 64, dtype=dtype, seed=26)
    out, lse = run_gpu_paged(inp, causal=True, num_splits=3, flags=kernel)
    o_ref, l_ref = reference_paged(inp, 0.0, True)
    assert_close(inp, out, lse, o_ref, l_ref)


def test_paged_equals_packed_path():
    """The same keys through the paged and the packed entry points agree."""
    from gpu_harness import run_gpu
    from workloads import Inputs
    import oracle
    inp = make_paged_inputs([1, 1], [5000, 777], 32, 8, 128, 128, 128, seed=22)
    out_p, lse_p = run_gpu_paged(inp, num_splits=4)
    k, v, cu_k = oracle.gather_paged_kv(inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens_k)
    packed = Inputs(q=inp.q, k=k, v=v, cu_seqlens_q=inp.cu_seqlens_q,
                    cu_seqlens_k=torch.from_numpy(cu_k), max_seqlen_q=inp.max_seqlen_q,
                    h_q=inp.h_q, h_kv=inp.h_kv, dtype=inp.dtype)
    out_c, lse_c = run_gpu(packed, num_splits=4)
    assert np.abs(out_p - out_c[: out_p.shape[0]]).max() <= 1e-2
    assert np.abs(lse_p - lse_c[:, : lse_p.shape[1]]).max() <= 1e-3


def test_paged_bad_page_index_is_reported():
    """A block-table entry outside the pool is skipped and flagged."""
    inp = make_paged_inputs([1], [100], 2, 2, 128, 128, 64, seed=23)
    inp.block_table[0, 0] = 10_000
    dev = torch.device("cuda:0")
    out = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device=dev)
    fa.fa_fwd_splitkv_paged(inp.q.to(dev), inp.k_cache.to(dev), inp.v_cache.to(dev),
                            inp.cu_seqlens_q.to(dev), inp.seqlens_k.to(dev),
                            inp.block_table.to(dev), 1, out, None, None, num_splits=1)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == -6


def test_full_paged_gqa_decode_sampled_heads():
    """The GQA decode batch at full size (B=32, H_q=32, H_kv=8, D=128, K
    lengths U[1024, 32768], seed 0; 2.3 GB of K/V) in a pool of 64-key pages
    handed out in a shuffled order, through the paged entry point in the
    benchmark's launch configuration (automatic splits); 4 of 32 query heads
    against the oracle on the keys gathered back from the pages."""
    import oracle
    lens_k = gqa_decode_lengths(0)
    inp = make_paged_inputs([1] * len(lens_k), lens_k, 32, 8, 128, 128, 64, seed=24)
    out, lse = run_gpu_paged(inp)
    k, v, cu_k = oracle.gather_paged_kv(inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens_k)
    packed = Inputs(q=inp.q, k=k, v=v, cu_seqlens_q=inp.cu_seqlens_q,
                    cu_seqlens_k=torch.from_numpy(cu_k), max_seqlen_q=inp.max_seqlen_q,
                    h_q=inp.h_q, h_kv=inp.h_kv, dtype=inp.dtype)
    heads = [0, 9, 22, 31]
    o_ref, l_ref = reference(packed, heads=heads)
    assert_close(packed, out, lse, o_ref, l_ref, heads=heads)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
