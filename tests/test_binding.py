"""CPU tests of the Python binding's argument checks.  The C library sees only
addresses and sizes, so the binding refuses, before any call, tensors whose
layout it would misread: strided views, wrong dtypes or shapes, and host
memory.  Every case here fails in the binding; nothing reaches a GPU."""

import pytest
import torch

import split_kv_flashattention_gb300 as fa


def _args(**over):
    """A consistent decode-shaped call on host tensors (B=1, Lq=2, Lk=8,
    H_q=4, H_kv=2, d=64), with some arguments replaced."""
    a = dict(
        q=torch.zeros(2, 4, 64, dtype=torch.bfloat16),
        k=torch.zeros(8, 2, 64, dtype=torch.bfloat16),
        v=torch.zeros(8, 2, 64, dtype=torch.bfloat16),
        cu_seqlens_q=torch.tensor([0, 2], dtype=torch.int32),
        cu_seqlens_k=torch.tensor([0, 8], dtype=torch.int32),
        max_seqlen_q=2,
        out=torch.zeros(2, 4, 64, dtype=torch.bfloat16),
        lse=torch.zeros(4, 2, dtype=torch.float32),
    )
    a.update(over)
    return a


def _strided(t):
    """The same shape as t, not contiguous."""
    return t.transpose(0, 1).contiguous().transpose(0, 1)


@pytest.mark.parametrize("over, message", [
    (dict(q=_strided(torch.zeros(2, 4, 64, dtype=torch.bfloat16))), "q must be contiguous"),
    (dict(k=torch.zeros(8, 2, 64, dtype=torch.float16)), "k has dtype"),
    (dict(q=torch.zeros(2, 4, 64, dtype=torch.float32)), "q has dtype"),
    (dict(v=torch.zeros(7, 2, 64, dtype=torch.bfloat16)), "differ before the head dim"),
    (dict(k=torch.zeros(8, 2, 128, dtype=torch.bfloat16),
          v=torch.zeros(8, 2, 128, dtype=torch.bfloat16)), "head dims differ"),
    (dict(q=torch.zeros(2, 256, dtype=torch.bfloat16)), "3-D"),
    (dict(cu_seqlens_k=torch.tensor([0, 8], dtype=torch.int64)), "cu_seqlens_k has dtype"),
    (dict(cu_seqlens_k=torch.tensor([0, 4, 8], dtype=torch.int32)), "cu_seqlens_k has shape"),
    (dict(cu_seqlens_q=torch.zeros(1, 2, dtype=torch.int32)), "cu_seqlens_q must be 1-D"),
    (dict(out=torch.zeros(2, 4, 32, dtype=torch.bfloat16)), "out has shape"),
    (dict(out=torch.zeros(2, 4, 64, dtype=torch.float32)), "out has dtype"),
    (dict(lse=torch.zeros(2, 4, dtype=torch.float32)), "lse has shape"),
    (dict(lse=torch.zeros(4, 2, dtype=torch.float64)), "lse has dtype"),
    (dict(workspace=_strided(torch.zeros(4, 4))), "workspace must be contiguous"),
    (dict(descale_q=torch.ones(1, dtype=torch.float16)), "descale_q has dtype"),
    (dict(), "must be CUDA tensors"),
    (dict(lse=None), "must be CUDA tensors"),
])
def test_forward_arguments_are_checked_before_the_call(over, message):
    with pytest.raises(ValueError, match=message):
        fa.fa_fwd_splitkv_ex(**_args(**over))


@pytest.mark.parametrize("entry", ["fa_fwd_splitkv", "fa_fwd_splitkv_noalloc"])
def test_other_entry_points_check_their_arguments(entry):
    fn = getattr(fa, entry)
    with pytest.raises(ValueError, match="out has shape"):
        fn(**_args(out=torch.zeros(2, 4, 32, dtype=torch.bfloat16)))
    with pytest.raises(ValueError, match="must be CUDA tensors"):
        fn(**_args())


def test_bf16_shorthand_refuses_other_dtypes():
    f16 = dict(q=torch.zeros(2, 4, 64, dtype=torch.float16),
               k=torch.zeros(8, 2, 64, dtype=torch.float16),
               v=torch.zeros(8, 2, 64, dtype=torch.float16),
               out=torch.zeros(2, 4, 64, dtype=torch.float16))
    with pytest.raises(ValueError, match="must be CUDA tensors|bf16"):
        fa.fa_fwd_splitkv(**_args(**f16))


def _paged_args(**over):
    a = dict(
        q=torch.zeros(1, 4, 64, dtype=torch.bfloat16),
        k_cache=torch.zeros(3, 32, 2, 64, dtype=torch.bfloat16),
        v_cache=torch.zeros(3, 32, 2, 64, dtype=torch.bfloat16),
        cu_seqlens_q=torch.tensor([0, 1], dtype=torch.int32),
        seqlens_k=torch.tensor([70], dtype=torch.int32),
        block_table=torch.tensor([[2, 0, 1]], dtype=torch.int32),
        max_seqlen_q=1,
        out=torch.zeros(1, 4, 64, dtype=torch.bfloat16),
    )
    a.update(over)
    return a


@pytest.mark.parametrize("over, message", [
    (dict(k_cache=torch.zeros(3, 32, 2, 64, dtype=torch.float16)), "k has dtype"),
    (dict(k_cache=torch.zeros(96, 2, 64, dtype=torch.bfloat16),
          v_cache=torch.zeros(96, 2, 64, dtype=torch.bfloat16)), "4-D"),
    (dict(seqlens_k=torch.tensor([0, 70], dtype=torch.int32)), "seqlens_k has shape"),
    (dict(block_table=torch.tensor([2, 0, 1], dtype=torch.int32)), "block_table must be"),
    (dict(block_table=torch.tensor([[2, 0, 1]], dtype=torch.int64)), "block_table has dtype"),
    (dict(), "must be CUDA tensors"),
])
def test_paged_arguments_are_checked_before_the_call(over, message):
    with pytest.raises(ValueError, match=message):
        fa.fa_fwd_splitkv_paged(**_paged_args(**over))


def test_split_ranges_hook_checks_its_offsets():
    cq = torch.tensor([0, 1], dtype=torch.int32)
    with pytest.raises(ValueError, match="cu_seqlens_k has dtype"):
        fa.fa_debug_split_ranges(cq, torch.tensor([0, 9]), 1, False, -1, 2, 128)
    with pytest.raises(ValueError, match="must be CUDA tensors"):
        fa.fa_debug_split_ranges(cq, torch.tensor([0, 9], dtype=torch.int32), 1, False, -1, 2, 128)
