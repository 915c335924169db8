"""Paged K/V layout, written out as plain indexing.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages this library follows do not describe a paged cache; the layout is
the common serving convention: a pool of pages [num_pages, page_size, h_kv,
d], a block table [batch, max_pages] whose entry (b, i) names the page that
holds keys i*page_size .. (i+1)*page_size - 1 of sequence b, and the key
count of each sequence.  Attention over a paged cache is, by definition,
attention over the keys gathered back into one packed buffer, so the oracle
gathers and then applies ``attention.attention_forward``.
"""

from __future__ import annotations

import numpy as np
import torch


def gather_paged_kv(k_cache, v_cache, block_table, seqlens_k):
    """-> (k, v, cu_seqlens_k): the keys/values of every sequence, in order,
    packed along the token axis (cu_seqlens_k int32 [batch+1])."""
    kc = k_cache.detach().cpu() if isinstance(k_cache, torch.Tensor) else torch.as_tensor(k_cache)
    vc = v_cache.detach().cpu() if isinstance(v_cache, torch.Tensor) else torch.as_tensor(v_cache)
    bt = [list(map(int, row)) for row in (block_table.tolist() if hasattr(block_table, "tolist") else block_table)]
    lens = [int(x) for x in (seqlens_k.tolist() if hasattr(seqlens_k, "tolist") else seqlens_k)]
    page_size = int(kc.shape[1])
    ks, vs, cu = [], [], [0]
    for b, n in enumerate(lens):
        for j in range(n):
            page = bt[b][j // page_size]
            ks.append(kc[page, j % page_size])
            vs.append(vc[page, j % page_size])
        cu.append(cu[-1] + n)
    if ks:
        k = torch.stack(ks)
        v = torch.stack(vs)
    else:
        k = kc.new_empty((0,) + tuple(kc.shape[2:]))
        v = vc.new_empty((0,) + tuple(vc.shape[2:]))
    return k, v, np.asarray(cu, dtype=np.int32)
