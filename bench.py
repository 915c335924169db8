#!/usr/bin/env python
"""Benchmark of the split-KV attention forward on GB300.

Default workload: long-context decode, B=1, Q=1, K=131072, H_q=H_kv=32,
D=128, bf16 N(0,1) inputs, automatic split count (the split sweep workload of
flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference",
"Benchmarks").  One step = one pass of the whole path: the split partial
kernel plus the combine kernel.  The metric is HBM throughput in TB/s with
the bytes counted as that page counts them (K + V + Q + O at the storage
width), divided by the device time of a step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload long_decode|gqa_decode|fp8_prefix|fp8_prefix_11k]
                  [--num-splits S] [--kernel auto|simt|umma]

With N > 1 (torchrun) every rank runs its own replica of the workload
(independent problems: weak scaling, no collective on the data path) and
rank 0 prints the aggregate.  `--impl reference` times the float64 CPU
oracle on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import workload  # noqa: E402

METRIC = "decode attn HBM TB/s (K=128K, Q=1) & varlen prefill TFLOPS, % of roofline"
L2_FLUSH_BYTES = 256 << 20  # twice GB300's 129 MB L2
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "split_kv_flashattention_gb300", "csrc")

WORKLOADS = {
    "long_decode": dict(name="long_decode", kw={},
                        desc="long-context decode MHA: B=1, Q=1, K=131072, H_q=H_kv=32, D=128, bf16"),
    "gqa_decode": dict(name="gqa_decode", kw={},
                       desc="batched GQA decode varlen: B=32, Q=1, H_q=32, H_kv=8, D=128, "
                            "K lengths U[1024,32768] seed 0, bf16"),
    "fp8_prefix": dict(name="fp8_prefix", kw={"kv": 16384},
                       desc="short cached-prefix FP8: B=1, Q=70, H=12, D_qk=192, D_v=128, KV=16384, e4m3"),
    "fp8_prefix_11k": dict(name="fp8_prefix", kw={"kv": 11008},
                           desc="short cached-prefix FP8: B=1, Q=70, H=12, D_qk=192, D_v=128, KV=11008, e4m3"),
    "prefill": dict(name="prefill", kw={"h_kv": 16}, causal=False, kind="tensor",
                    desc="varlen prefill: 16384 tokens (4096,512,3072,1024,2560,1536,2048,1536), "
                         "H_q=H_kv=16, D=128, bf16, no mask"),
    "prefill_causal": dict(name="prefill", kw={"h_kv": 16}, causal=True, kind="tensor",
                           desc="varlen prefill: 16384 tokens (4096,512,3072,1024,2560,1536,2048,1536), "
                                "H_q=H_kv=16, D=128, bf16, causal"),
    "prefill_gqa": dict(name="prefill", kw={"h_kv": 4}, causal=False, kind="tensor",
                        desc="varlen prefill: 16384 tokens, H_q=16, H_kv=4, D=128, bf16, no mask"),
    "prefill_d256": dict(name="prefill", kw={"h_kv": 16, "d": 256}, causal=False, kind="tensor",
                         desc="varlen prefill: 16384 tokens, H_q=H_kv=16, D=256, bf16, no mask"),
    "decode_d256": dict(name="long_decode", kw={"kv": 65536, "h": 16, "d": 256},
                        desc="long-context decode MHA: B=1, Q=1, K=65536, H_q=H_kv=16, D=256, bf16"),
    "paged_decode": dict(name="gqa_decode", kw={}, paged=64,
                         desc="batched GQA decode varlen over a paged K/V cache: B=32, Q=1, H_q=32, "
                              "H_kv=8, D=128, K lengths U[1024,32768] seed 0, 64-key pages, bf16"),
    "prefill_gqa_causal": dict(name="prefill", kw={"h_kv": 4}, causal=True, kind="tensor",
                               desc="varlen prefill: 16384 tokens, H_q=16, H_kv=4, D=128, bf16, causal"),
    "prefill_fp16": dict(name="prefill", kw={"h_kv": 16, "dtype": "fp16"}, causal=False, kind="tensor",
                         desc="varlen prefill: 16384 tokens, H_q=H_kv=16, D=128, fp16, no mask"),
    "prefill_causal_fp16": dict(name="prefill", kw={"h_kv": 16, "dtype": "fp16"}, causal=True,
                                kind="tensor",
                                desc="varlen prefill: 16384 tokens, H_q=H_kv=16, D=128, fp16, causal"),
}


def attended_pairs(inp, causal):
    """(query, key) pairs the mask allows, summed over sequences (the FLOP
    count of the cutlass varlen page: attended pairs only)."""
    cq = inp.cu_seqlens_q.tolist()
    ck = inp.cu_seqlens_k.tolist()
    total = 0
    for b in range(len(cq) - 1):
        lq, lk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
        if not causal:
            total += lq * lk
        else:
            for i in range(lq):
                total += max(0, min(lk, i + lk - lq + 1))
    return total


def flops(inp, causal):
    return 2 * (inp.d_qk + inp.d_v) * inp.h_q * attended_pairs(inp, causal)


def measured_tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0) or 0), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def prefill_secondary(fa, dev, steps, warmup):
    """Varlen prefill TFLOPS (the metric's second part) for no-mask and causal."""
    res = {}
    peak, _, src = measured_tensor_peak()
    for name in ("prefill", "prefill_causal"):
        spec = WORKLOADS[name]
        inp = workload(spec["name"], device=str(dev), **spec["kw"])
        causal = spec["causal"]
        out = torch.empty((inp.q.shape[0], inp.h_q, inp.d_v), dtype=inp.q.dtype, device=dev)
        lse = torch.empty((inp.h_q, inp.q.shape[0]), dtype=torch.float32, device=dev)
        cq, ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev)
        stream = torch.cuda.current_stream(dev)
        ws_bytes = fa.fa_fwd_splitkv_workspace_size(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv,
                                                   inp.d_v, 0)
        ws = torch.empty(max(ws_bytes, 16) // 4, dtype=torch.float32, device=dev) if ws_bytes else None

        def step():
            fa.fa_fwd_splitkv_ex(inp.q, inp.k, inp.v, cq, ck, inp.max_seqlen_q, out, lse, ws,
                                 0.0, causal, -1, 0, None, None, None, 0, stream)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        # inputs (201 MB) are less than twice the L2: overwrite it between
        # steps, outside the timed spans
        flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush_buf.zero_()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        del flush_buf
        tf = flops(inp, causal) / (ms * 1e-3) / 1e12
        res[name] = {"ms": ms, "tflops": tf, "frac": tf / peak, "flops": flops(inp, causal)}
    res["peak_tflops"] = peak
    res["peak_source"] = src + " bf16 dense (burst)"
    res["workload"] = WORKLOADS["prefill"]["desc"].replace(", no mask", "")
    res["l2"] = "L2 overwritten between steps (256 MB write, untimed)"
    return res


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's value (the step time the job waited for);
    plain value at world size 1.  Works with the nccl and gloo backends."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job rate: every rank processes its own replica of the workload
    (weak scaling), so the units of all ranks are divided by the slowest
    rank's step time.  Returned per second, in units / 1e12."""
    return world * units_per_rank / (ms_per_step * 1e-3) / 1e12


def to_paged(inp, page_size, dev):
    """Scatter the packed K/V of `inp` into a pool of pages handed out in a
    seeded random order; returns (k_cache, v_cache, block_table, seqlens_k)."""
    import numpy as np
    cu = inp.cu_seqlens_k.tolist()
    lens = [cu[b + 1] - cu[b] for b in range(len(cu) - 1)]
    need = [-(-n // page_size) for n in lens]
    num_pages = sum(need)
    order = torch.from_numpy(np.random.default_rng(0).permutation(num_pages)).to(dev)
    kc = torch.zeros((num_pages, page_size) + tuple(inp.k.shape[1:]), dtype=inp.k.dtype, device=dev)
    vc = torch.zeros((num_pages, page_size) + tuple(inp.v.shape[1:]), dtype=inp.v.dtype, device=dev)
    table = torch.zeros((len(lens), max(need)), dtype=torch.int32)
    pos = 0
    for b, n in enumerate(lens):
        pages = order[pos:pos + need[b]]
        table[b, :need[b]] = pages.cpu().to(torch.int32)
        for i in range(need[b]):
            rows = min(page_size, n - i * page_size)
            kc[pages[i], :rows] = inp.k[cu[b] + i * page_size: cu[b] + i * page_size + rows]
            vc[pages[i], :rows] = inp.v[cu[b] + i * page_size: cu[b] + i * page_size + rows]
        pos += need[b]
    return kc, vc, table.to(dev), torch.tensor(lens, dtype=torch.int32, device=dev)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_decode", choices=sorted(WORKLOADS))
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "umma", "umma2"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the varlen prefill TFLOPS measurement of the default line")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--kv", type=int, default=0, help="override the key length (long_decode)")
    return ap.parse_args()


def byte_counts(inp, ns):
    """Algorithmic bytes: the metric's (K+V+Q+O at storage width) and the
    partial kernel's (K+V+Q read, workspace or O+LSE written)."""
    es = 1 if inp.dtype == "e4m3" else 2
    tq, tk = inp.q.shape[0], inp.k.shape[0]
    kv = tk * inp.h_kv * (inp.d_qk + inp.d_v) * es
    q = tq * inp.h_q * inp.d_qk * es
    o = tq * inp.h_q * inp.d_v * 2
    metric = kv + q + o
    if ns > 1:
        partial = kv + q + ns * tq * inp.h_q * (inp.d_v + 1) * 4
    else:
        partial = kv + q + o + tq * inp.h_q * 4
    return metric, partial


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_TAGS = {1: "simt_splitkv", 2: "umma_splitkv", 3: "umma2_splitkv", 4: "umma2p_splitkv"}

KERNEL_SOURCES = {
    "simt_splitkv": ("fa_simt.cuh", "fa_simt_launch.cuh", "fa_simt_bf16.cu",
                     "fa_simt_bf16_ordered.cu", "fa_common.cuh", "fa_ptx.cuh", "fa_convert.cuh"),
    "umma_splitkv": ("fa_umma.cuh", "fa_umma_launch.cuh", "fa_umma_bf16.cu", "fa_umma_e4m3.cu",
                     "fa_common.cuh", "fa_ptx.cuh", "fa_convert.cuh"),
    "umma2p_splitkv": ("fa_umma2p.cuh", "fa_umma2p_launch.cuh", "fa_umma2p_bf16.cu", "fa_umma2.cuh",
                       "fa_common.cuh", "fa_ptx.cuh", "fa_convert.cuh"),
    "umma2_splitkv": ("fa_umma2.cuh", "fa_umma2_launch.cuh", "fa_umma2_bf16.cu", "fa_common.cuh",
                      "fa_ptx.cuh", "fa_convert.cuh"),
}


def kernel_source_hash(kernel_tag):
    """Hash of the sources a kernel is built from (its ncu counters are only
    valid for these exact sources)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel_tag]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag, workload_name):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when absent or taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload_name}.txt")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"^source_hash:\s*(\S+)", text, re.M)
    m_t = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not m_hash or not m_t or m_hash.group(1) != kernel_source_hash(kernel_tag):
        return None
    return float(m_t.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.error = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # pragma: no cover
            self.error = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.error or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": self.error or "no nvidia-smi samples"}
        inside = [p for t, p in self.samples if t0 <= t <= t1] or [p for _, p in self.samples]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


def cpu_baseline(inp_cpu, budget_s=12.0, heads=2, causal=False, kind="hbm"):
    """The float64 oracle on `heads` query heads of the workload, repeated for
    about budget_s seconds on the host cores; reported in the metric's unit."""
    import oracle

    group = inp_cpu.h_q // inp_cpu.h_kv
    hs = list(range(heads))
    kvs = sorted({h // group for h in hs})
    q = inp_cpu.q[:, hs]
    k = inp_cpu.k[:, kvs]
    v = inp_cpu.v[:, kvs]
    es = 1 if inp_cpu.dtype == "e4m3" else 2
    tq, tk = q.shape[0], k.shape[0]
    if kind == "tensor":
        sample_work = 2 * (inp_cpu.d_qk + inp_cpu.d_v) * heads * attended_pairs(inp_cpu, causal)
        unit = "TFLOPS"
    else:
        sample_work = (tk * len(kvs) * (inp_cpu.d_qk + inp_cpu.d_v) * es
                       + tq * heads * (inp_cpu.d_qk * es + inp_cpu.d_v * 2))
        unit = "TB/s"
    reps, t_total = 0, 0.0
    while t_total < budget_s or reps == 0:
        t = time.perf_counter()
        oracle.attention_forward(q, k, v, inp_cpu.cu_seqlens_q, inp_cpu.cu_seqlens_k,
                                 heads, len(kvs), 0.0, causal, -1, inp_cpu.descale_q,
                                 inp_cpu.descale_k, inp_cpu.descale_v)
        t_total += time.perf_counter() - t
        reps += 1
    return {"value": sample_work * reps / t_total / 1e12, "unit": unit,
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{heads} of {inp_cpu.h_q} query heads (all keys), float64 oracle, "
                      f"{reps} repetitions in {t_total:.1f} s, numpy/BLAS default threads",
            "seconds": round(t_total, 2)}


def inp_host(inp):
    import dataclasses
    return dataclasses.replace(inp, q=inp.q.cpu(), k=inp.k.cpu(), v=inp.v.cpu())


def run_reference(args, spec, rank):
    """The oracle as the reference arm: one oracle call on a bounded sample
    (one query head, all keys) per step, on the host cores."""
    if rank != 0:
        return
    kind = spec.get("kind", "hbm")
    causal = spec.get("causal", False)
    kw = dict(spec["kw"])
    if args.kv:
        kw["kv"] = args.kv
    inp = workload(spec["name"], **kw)
    vals = []
    cb = None
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(inp, budget_s=0.0, heads=1, causal=causal, kind=kind)
        if i >= args.warmup:
            vals.append(cb["value"])
    value = statistics.median(vals) if vals else cb["value"]
    unit = cb["unit"]
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": spec["desc"]},
        "cpu_baseline": {"value": value, "unit": unit, "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": "1 of %d query heads (all keys), one float64 oracle call per step"
                                   % inp.h_q},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    spec = WORKLOADS[args.workload]
    kind = spec.get("kind", "hbm")
    causal = spec.get("causal", False)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, spec, rank)
        return

    import split_kv_flashattention_gb300 as fa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    kernel_flag = {"auto": fa.FA_KERNEL_AUTO, "simt": fa.FA_KERNEL_SIMT,
                   "umma": fa.FA_KERNEL_UMMA, "umma2": fa.FA_KERNEL_UMMA2}[args.kernel]
    kw = dict(spec["kw"])
    if args.kv:
        kw["kv"] = args.kv
    inp = workload(spec["name"], device=str(dev), **kw)
    q, k, v = inp.q, inp.k, inp.v
    cq, ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev)
    paged = spec.get("paged", 0)
    if paged:
        # the same keys, scattered into a shuffled page pool
        kc, vc, bt, sk = to_paged(inp, paged, dev)
    out_dtype = torch.bfloat16 if inp.dtype == "e4m3" else q.dtype
    out = torch.empty((q.shape[0], inp.h_q, inp.d_v), dtype=out_dtype, device=dev)
    lse = torch.empty((inp.h_q, q.shape[0]), dtype=torch.float32, device=dev)
    ns, _ = fa.fa_plan(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv, args.num_splits)
    ws_bytes = fa.fa_fwd_splitkv_workspace_size(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv,
                                               inp.d_v, args.num_splits)
    ws = torch.empty(max(ws_bytes, 16) // 4, dtype=torch.float32, device=dev) if ws_bytes else None
    dq = dk = dv = None
    if inp.dtype == "e4m3":
        dq = torch.tensor([inp.descale_q], dtype=torch.float32, device=dev)
        dk = torch.tensor([inp.descale_k], dtype=torch.float32, device=dev)
        dv = torch.tensor([inp.descale_v], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    def call(flags):
        if paged:
            fa.fa_fwd_splitkv_paged(q, kc, vc, cq, sk, bt, inp.max_seqlen_q, out, lse, ws, 0.0,
                                    causal, -1, args.num_splits, dq, dk, dv, flags, stream)
            return
        fa.fa_fwd_splitkv_ex(q, k, v, cq, ck, inp.max_seqlen_q, out, lse, ws, 0.0, causal, -1,
                             args.num_splits, dq, dk, dv, flags, stream)

    def partial():
        call(kernel_flag | fa.FA_RUN_PARTIAL_ONLY)

    def combine():
        if ns > 1:
            call(kernel_flag | fa.FA_RUN_COMBINE_ONLY)

    sampler = ClockSampler(local_rank)
    sampler.start()
    for _ in range(args.warmup):
        partial()
        combine()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_error(clear=True) != 0:
        raise RuntimeError("device error during warm-up")
    # the partial kernel the library chose (the last call above enqueued it)
    partial()
    kern_tag = KERNEL_TAGS[fa.fa_debug_last_kernel()]
    torch.cuda.synchronize(dev)

    # Timed region: K whole steps (partial + combine, as one call makes them,
    # so the combine's programmatic launch overlaps the partial's tail).
    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1)

    # Workloads that fit in L2 are timed step by step with L2 overwritten in
    # between (outside the timed spans); larger ones run back to back.
    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, v))
    flush_l2 = in_bytes < L2_FLUSH_BYTES
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if flush_l2 else None

    def timed_flushed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        for a, b in evs:
            flush_buf.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        return sum(a.elapsed_time(b) for a, b in evs)

    run = timed_flushed if flush_l2 else timed
    t_wall0 = time.time()
    total_ms = run(lambda: call(kernel_flag), args.steps)
    t_wall1 = time.time()
    # The dominant (partial) kernel alone, K launches, for its roofline; then
    # the combine alone over the same workspace.
    partial_ms = run(partial, args.steps) / args.steps
    combine_ms = run(combine, args.steps) / args.steps if ns > 1 else 0.0
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    err = fa.fa_get_device_error(clear=True)
    if err != 0:
        raise RuntimeError(f"device error {fa.fa_status_string(err)}")

    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    metric_bytes, partial_bytes = byte_counts(inp, ns)
    work_flops = flops(inp, causal)
    if kind == "tensor":
        unit = "TFLOPS"
        value = job_throughput(work_flops, world, ms_per_step)
    else:
        unit = "TB/s"
        value = job_throughput(metric_bytes, world, ms_per_step)

    # ---- end to end through the public call with host buffers
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    # the step's inputs: Q and cu_seqlens_q, and K/V with their index arrays
    dev_in = [q, cq] + ([kc, vc, bt, sk] if paged else [k, v, ck])
    host_in = [x.cpu().pin_memory() for x in dev_in]
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

    def e2e_step():
        for d_t, h_t in zip(dev_in, host_in):
            d_t.copy_(h_t, non_blocking=True)
        call(kernel_flag)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    e2e_value = job_throughput(work_flops if kind == "tensor" else metric_bytes, world, e2e_ms)

    secondary = None
    if kind == "hbm" and world == 1 and not args.no_prefill:
        secondary = prefill_secondary(fa, dev, steps=max(3, min(args.steps, 30)),
                                      warmup=max(3, min(args.warmup, 5)))

    if rank == 0:
        if kind == "tensor":
            peak, peak_sus, src = measured_tensor_peak()
            achieved = work_flops / (partial_ms * 1e-3) / 1e12
            same_rate = "" if inp.dtype == "bf16" else f"; {inp.dtype} dense at the bf16 nominal rate (1:1)"
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "peak_source": src + " bf16 dense (burst)" + same_rate,
                    "traffic": profiled_traffic(kern_tag, args.workload),
                    "kernel": f"{kern_tag} partial kernel", "partial_ms": partial_ms,
                    "timing": "K partial-only launches, CUDA events",
                    "algorithmic_flops_per_launch": work_flops}
        else:
            peak_gbs, peak_src = measured_peaks()
            achieved_gbs = partial_bytes / (partial_ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": peak_gbs, "unit": "GB/s",
                    "frac": achieved_gbs / peak_gbs, "peak_source": peak_src,
                    "traffic": profiled_traffic(kern_tag, args.workload),
                    "kernel": f"{kern_tag} partial kernel", "partial_ms": partial_ms,
                    "combine_ms": combine_ms,
                    "timing": "K partial-only launches, CUDA events",
                    "algorithmic_bytes_per_launch": partial_bytes}
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if inp.dtype == "bf16" else inp.dtype, "data": "synthetic",
            "config": {"workload": spec["desc"], "num_splits": ns,
                       "num_splits_requested": args.num_splits, "kernel": kern_tag,
                       "l2": ("L2 overwritten between steps (256 MB write, untimed); Q+K+V %.3f GB"
                              if flush_l2 else "inputs larger than L2 (Q+K+V %.2f GB)") % (in_bytes / 1e9),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * (2 if ns > 1 else 1),
            "clocks": clocks,
        }
        if secondary is not None:
            line["prefill"] = secondary
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(inp_host(inp), causal=causal, kind=kind)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
