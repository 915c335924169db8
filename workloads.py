"""Seeded synthetic inputs for split-KV attention.

This module is the one piece shared by the oracle side (tests, CPU baseline)
and the CUDA side (tests, bench): it only draws random numbers and packs
them.  It holds none of the attention arithmetic.

Recipe (same for every workload):
* torch.Generator on the CPU (or, for the large workloads the GPU tests and
  the benchmark use, on the CUDA device: same recipe, the device's Philox
  generator), manual_seed(seed), drawing Q, then K, then V as float32
  N(0, 1), in chunks of CHUNK elements, each chunk cast to the storage dtype.
  Both sides always see the same tensor: the oracle gets a host copy of it.
* Packed varlen layout: Q [total_q, h_q, d_qk], K [total_k, h_kv, d_qk],
  V [total_k, h_kv, d_v], cu_seqlens int32 [B+1] exclusive prefix sums.
* FP8 e4m3: the float32 draw x of a whole tensor gives descale = amax/448 and
  stored codes e4m3(x / descale) (round to nearest even); the descale is a
  float32 scalar.  Quantisation is input preparation, not part of the path.

Named workloads mirror the shapes the pages measure.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

CHUNK = 1 << 22
E4M3_MAX = 448.0

DTYPES = {
    "bf16": torch.bfloat16,
    "fp16": torch.float16,
    "e4m3": torch.float8_e4m3fn,
}


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    cu_seqlens_q: torch.Tensor
    cu_seqlens_k: torch.Tensor
    max_seqlen_q: int
    h_q: int
    h_kv: int
    dtype: str
    descale_q: float = 1.0
    descale_k: float = 1.0
    descale_v: float = 1.0

    @property
    def batch(self) -> int:
        return int(self.cu_seqlens_q.numel()) - 1

    @property
    def d_qk(self) -> int:
        return int(self.q.shape[2])

    @property
    def d_v(self) -> int:
        return int(self.v.shape[2])


def _randn_chunked(gen: torch.Generator, shape, out_dtype) -> torch.Tensor:
    n = 1
    for s in shape:
        n *= int(s)
    dev = gen.device
    out = torch.empty(n, dtype=out_dtype, device=dev)
    for s0 in range(0, n, CHUNK):
        s1 = min(n, s0 + CHUNK)
        out[s0:s1] = torch.randn(s1 - s0, generator=gen, dtype=torch.float32,
                                 device=dev).to(out_dtype)
    return out.view(*shape)


def _randn_e4m3(gen: torch.Generator, shape):
    x = _randn_chunked(gen, shape, torch.float32)
    amax = float(x.abs().max()) if x.numel() else 1.0
    descale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
    codes = (x / descale).to(torch.float8_e4m3fn)
    return codes, descale


def cu_seqlens(lengths) -> torch.Tensor:
    c = [0]
    for n in lengths:
        c.append(c[-1] + int(n))
    return torch.tensor(c, dtype=torch.int32)


def make_inputs(lens_q, lens_k, h_q: int, h_kv: int, d_qk: int, d_v: int,
                dtype: str = "bf16", seed: int = 0, device: str = "cpu") -> Inputs:
    """Q/K/V on `device` (cu_seqlens always on the host)."""
    assert len(lens_q) == len(lens_k)
    total_q, total_k = int(sum(lens_q)), int(sum(lens_k))
    gen = torch.Generator(device=device).manual_seed(seed)
    if dtype == "e4m3":
        q, dq = _randn_e4m3(gen, (total_q, h_q, d_qk))
        k, dk = _randn_e4m3(gen, (total_k, h_kv, d_qk))
        v, dv = _randn_e4m3(gen, (total_k, h_kv, d_v))
    else:
        t = DTYPES[dtype]
        q = _randn_chunked(gen, (total_q, h_q, d_qk), t)
        k = _randn_chunked(gen, (total_k, h_kv, d_qk), t)
        v = _randn_chunked(gen, (total_k, h_kv, d_v), t)
        dq = dk = dv = 1.0
    return Inputs(q=q, k=k, v=v, cu_seqlens_q=cu_seqlens(lens_q),
                  cu_seqlens_k=cu_seqlens(lens_k),
                  max_seqlen_q=max([int(x) for x in lens_q] + [0]),
                  h_q=h_q, h_kv=h_kv, dtype=dtype,
                  descale_q=dq, descale_k=dk, descale_v=dv)


# ----------------------------------------------------------------------------
# Named workloads (shapes from the pages).

def gqa_decode_lengths(seed: int = 0, batch: int = 32):
    """Per-sequence key lengths uniform in [1024, 32768] from the seed."""
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(1024, 32768, endpoint=True, size=batch)]


PREFILL_LENGTHS = (4096, 512, 3072, 1024, 2560, 1536, 2048, 1536)
EDGE_LENGTHS = (1, 0, 63, 64, 65, 128, 129, 700)


def workload(name: str, seed: int = 0, device: str = "cpu", **kw) -> Inputs:
    """The named workloads; keyword overrides resize them for tests."""
    if name == "tiny_decode":
        kv = kw.get("kv", 1024)
        return make_inputs([1], [kv], 4, 4, 64, 64, "bf16", seed, device)
    if name == "long_decode":
        kv = kw.get("kv", 131072)
        h = kw.get("h", 32)
        d = kw.get("d", 128)
        return make_inputs([1], [kv], h, h, d, d, "bf16", seed, device)
    if name == "gqa_decode":
        batch = kw.get("batch", 32)
        lens_k = kw.get("lens_k") or gqa_decode_lengths(seed, batch)
        return make_inputs([1] * len(lens_k), lens_k, 32, 8, 128, 128, "bf16", seed, device)
    if name == "fp8_prefix":
        kv = kw.get("kv", 16384)
        q = kw.get("q", 70)
        h = kw.get("h", 12)
        return make_inputs([q], [kv], h, h, 192, 128, "e4m3", seed, device)
    if name == "prefill":
        lens = kw.get("lens", PREFILL_LENGTHS)
        d = kw.get("d", 128)
        return make_inputs(lens, lens, 16, kw.get("h_kv", 16), d, d,
                           kw.get("dtype", "bf16"), seed, device)
    if name == "edge":
        lens = kw.get("lens", EDGE_LENGTHS)
        return make_inputs(lens, lens, 8, 2, 128, 128, kw.get("dtype", "bf16"), seed, device)
    raise KeyError(name)


@dataclasses.dataclass
class PagedInputs:
    q: torch.Tensor
    k_cache: torch.Tensor       # [num_pages, page_size, h_kv, d_qk]
    v_cache: torch.Tensor       # [num_pages, page_size, h_kv, d_v]
    block_table: torch.Tensor   # int32 [batch, max_pages]
    seqlens_k: torch.Tensor     # int32 [batch]
    cu_seqlens_q: torch.Tensor
    max_seqlen_q: int
    h_q: int
    h_kv: int
    dtype: str
    page_size: int
    descale_q: float = 1.0
    descale_k: float = 1.0
    descale_v: float = 1.0

    @property
    def batch(self) -> int:
        return int(self.cu_seqlens_q.numel()) - 1

    @property
    def d_v(self) -> int:
        return int(self.v_cache.shape[3])


def make_paged_inputs(lens_q, lens_k, h_q: int, h_kv: int, d_qk: int, d_v: int,
                      page_size: int, dtype: str = "bf16", seed: int = 0,
                      spare_pages: int = 3) -> PagedInputs:
    """Q packed as usual; K/V in a pool of pages (the sequences' pages plus
    `spare_pages` unused ones) handed out in a seeded random order; unused
    block-table slots hold page 0."""
    need = [-(-int(n) // page_size) for n in lens_k]
    num_pages = sum(need) + spare_pages
    max_pages = max(need + [1])
    gen = torch.Generator().manual_seed(seed)
    t = DTYPES[dtype]
    q = _randn_chunked(gen, (int(sum(lens_q)), h_q, d_qk), t)
    k_cache = _randn_chunked(gen, (num_pages, page_size, h_kv, d_qk), t)
    v_cache = _randn_chunked(gen, (num_pages, page_size, h_kv, d_v), t)
    order = np.random.default_rng(seed).permutation(num_pages).tolist()
    table = np.zeros((len(lens_k), max_pages), dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = order[pos:pos + n]
        pos += n
    return PagedInputs(q=q, k_cache=k_cache, v_cache=v_cache,
                       block_table=torch.from_numpy(table),
                       seqlens_k=torch.tensor([int(n) for n in lens_k], dtype=torch.int32),
                       cu_seqlens_q=cu_seqlens(lens_q),
                       max_seqlen_q=max([int(x) for x in lens_q] + [0]), h_q=h_q, h_kv=h_kv,
                       dtype=dtype, page_size=page_size)
