#!/usr/bin/env python
"""Benchmark of the split-KV attention forward on GB300.

Default workload: long-context decode, B=1, Q=1, K=131072, H_q=H_kv=32,
D=128, bf16 N(0,1) inputs, automatic split count (the split sweep workload of
flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference",
"Benchmarks").  One step = one pass of the whole path: the split partial
kernel plus the combine kernel.  The metric is HBM throughput in TB/s with
the bytes counted as that page counts them (K + V + Q + O at the storage
width), divided by the device time of a step.  The K timed steps are one
CUDA graph of K library calls, replayed once.

The default line also carries flat fields for every configuration of the
metric (cfg1_* tiny decode, cfg2_* the long-decode split sweep 1..128 and
auto, cfg3_* batched GQA decode, cfg4_* the FP8 cached prefix at 16384 and
11008 keys, cfg5_* varlen prefill in bf16/fp16, H_kv 16/4, no mask/causal),
each the median of 7 rounds of 100 CUDA-graph replays of one call (the
timing of aiter PR "[FlyDSL] Enable FP8 FMHA split-K for short cached-prefix
queries"), with a roofline fraction against the measured peaks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--num-splits S] [--kernel auto|simt|umma|umma2]
                  [--no-configs] [--no-cpu-baseline]

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


# ----------------------------------------------------------------------------
# Graph-replay timing of the five configurations (flat fields of the line)

ROUNDS, REPS = 7, 100
SWEEP_SPLITS = (1, 2, 4, 8, 16, 32, 64, 128)


class Case:
    """One workload set up for timing: `copies` copies of its inputs (same
    values, distinct memory) so that consecutive calls of a replayed graph
    read inputs that are not in L2; shared outputs and workspace."""

    def __init__(self, fa, dev, spec, num_splits=0, flags=0, rotate=True, kw_extra=None):
        kw = dict(spec["kw"])
        kw.update(kw_extra or {})
        self.spec = spec
        self.fa = fa
        self.inp = inp = workload(spec["name"], device=str(dev), **kw)
        self.causal = spec.get("causal", False)
        self.num_splits = num_splits
        self.flags = flags
        self.copies = [(inp.q, inp.k, inp.v)]
        self.in_bytes = sum(x.numel() * x.element_size() for x in self.copies[0])
        for _ in range(copies_for(self.in_bytes) - 1 if rotate else 0):
            self.copies.append((inp.q.clone(), inp.k.clone(), inp.v.clone()))
        self.cq, self.ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev)
        out_dtype = torch.bfloat16 if inp.dtype == "e4m3" else inp.q.dtype
        self.out = torch.empty((inp.q.shape[0], inp.h_q, inp.d_v), dtype=out_dtype, device=dev)
        self.lse = torch.empty((inp.h_q, inp.q.shape[0]), dtype=torch.float32, device=dev)
        self.ns, _ = fa.fa_plan(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv, num_splits)
        nbytes = fa.fa_fwd_splitkv_workspace_size(inp.batch, inp.max_seqlen_q, inp.h_q, inp.h_kv,
                                                  inp.d_v, num_splits)
        self.ws = (torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device=dev)
                   if nbytes else None)
        self.dq = self.dk = self.dv = None
        if inp.dtype == "e4m3":
            self.dq = torch.tensor([inp.descale_q], dtype=torch.float32, device=dev)
            self.dk = torch.tensor([inp.descale_k], dtype=torch.float32, device=dev)
            self.dv = torch.tensor([inp.descale_v], dtype=torch.float32, device=dev)

    def call(self, i, stream, extra_flags=0):
        q, k, v = self.copies[i % len(self.copies)]
        self.fa.fa_fwd_splitkv_ex(q, k, v, self.cq, self.ck, self.inp.max_seqlen_q, self.out,
                                  self.lse, self.ws, 0.0, self.causal, -1, self.num_splits,
                                  self.dq, self.dk, self.dv, self.flags | extra_flags, stream)


def copies_for(in_bytes):
    """Input copies a replayed graph cycles through: inputs of 256 MB (twice
    the L2) or more need none; smaller ones get enough copies that the calls
    between two uses of one copy read at least 256 MB."""
    if in_bytes >= L2_FLUSH_BYTES:
        return 1
    return min(512, -(-L2_FLUSH_BYTES // max(1, in_bytes)) + 1)


def graph_times(case, dev, rounds=ROUNDS, reps=REPS, extra_flags=0):
    """Per-call milliseconds of `rounds` replays of one CUDA graph holding
    `reps` calls (cycling through the case's input copies), after two warm
    replays; CUDA events on the replay stream."""
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for i in range(3):
            case.call(i, s, extra_flags)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(reps):
            case.call(i, s, extra_flags)
    times = []
    with torch.cuda.stream(s):
        for r in range(rounds + 2):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            s.synchronize()
            if r >= 2:
                times.append(e0.elapsed_time(e1) / reps)
    del g
    return times


def metric_bytes(inp):
    """K + V + Q + O at storage width (the flash-attention PR's `bw`)."""
    es = 1 if inp.dtype == "e4m3" else 2
    return (inp.k.shape[0] * inp.h_kv * (inp.d_qk + inp.d_v) * es
            + inp.q.shape[0] * inp.h_q * inp.d_qk * es + inp.q.shape[0] * inp.h_q * inp.d_v * 2)


CONFIG_FIELDS = [
    # (field prefix, workload spec, num_splits, kind)
    ("cfg1_tiny_decode", dict(name="tiny_decode", kw={}), 4, "latency"),
    ("cfg3_gqa_decode", dict(name="gqa_decode", kw={}), 0, "hbm"),
    ("cfg4_fp8_prefix_16384", dict(name="fp8_prefix", kw={"kv": 16384}), 0, "hbm"),
    ("cfg4_fp8_prefix_11008", dict(name="fp8_prefix", kw={"kv": 11008}), 0, "hbm"),
] + [
    (f"cfg5_prefill_{dt}_hkv{hkv}_{'causal' if c else 'nomask'}",
     dict(name="prefill", kw={"h_kv": hkv, "dtype": dt}, causal=c), 0, "tensor")
    for dt in ("bf16", "fp16") for hkv in (16, 4) for c in (False, True)
]


def config_fields(fa, dev, hbm_peak, tensor_peak):
    """Flat fields for the five configurations: the long-decode split sweep,
    tiny decode, GQA decode, the FP8 cached prefix at both key lengths and the
    varlen prefill variants; each the median of ROUNDS rounds of REPS
    CUDA-graph replays of one library call (partial + combine)."""
    out = {}

    def med(ts):
        return statistics.median(ts)

    sweep = [("cfg2_long_decode_auto", 0)] + [(f"cfg2_long_decode_ns{n}", n) for n in SWEEP_SPLITS]
    case = Case(fa, dev, dict(name="long_decode", kw={}))
    mb = metric_bytes(case.inp)
    for name, ns in sweep:
        case.num_splits = ns
        nbytes = fa.fa_fwd_splitkv_workspace_size(case.inp.batch, 1, case.inp.h_q, case.inp.h_kv,
                                                  case.inp.d_v, ns)
        if case.ws is None or case.ws.numel() * 4 < nbytes:
            case.ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device=dev)
        ms = med(graph_times(case, dev))
        out[name + "_us"] = ms * 1e3
        out[name + "_tbs"] = mb / (ms * 1e-3) / 1e12
        out[name + "_frac"] = mb / (ms * 1e-3) / 1e9 / hbm_peak
        if ns == 0:
            out[name + "_ns"] = fa.fa_plan(1, 1, 32, 32, 0)[0]
    del case
    torch.cuda.empty_cache()

    for prefix, spec, ns, kind in CONFIG_FIELDS:
        case = Case(fa, dev, spec, num_splits=ns)
        ms = med(graph_times(case, dev))
        kern_tag = KERNEL_TAGS.get(fa.fa_debug_last_kernel(), "?")
        out[prefix + "_us"] = ms * 1e3
        if kind == "hbm":
            mb = metric_bytes(case.inp)
            out[prefix + "_tbs"] = mb / (ms * 1e-3) / 1e12
            out[prefix + "_frac"] = mb / (ms * 1e-3) / 1e9 / hbm_peak
            out[prefix + "_ns"] = case.ns
            out[prefix + "_kernel"] = kern_tag
        elif kind == "tensor":
            tf = flops(case.inp, case.causal) / (ms * 1e-3) / 1e12
            out[prefix + "_tflops"] = tf
            out[prefix + "_frac"] = tf / tensor_peak
        del case
        torch.cuda.empty_cache()
    out["cfg_timing"] = (f"median of {ROUNDS} rounds x {REPS} CUDA-graph replays of one library call "
                         "(partial + combine), CUDA events; inputs under 256 MB rotated over copies so "
                         "that 256 MB (twice the L2) is read between two uses of one copy")
    out["cfg_frac_peaks"] = {"hbm_gbs": hbm_peak, "bf16_tflops": tensor_peak}
    return out


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
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration fields of the default line")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--kv", type=int, default=0, help="override the key length (long_decode)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch (gqa_decode, paged_decode): a smaller case for ncu")
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
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""
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
                 "--format=csv,noheader,nounits", "-lms", "50"],
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
        # a window shorter than the sampling interval is widened to the
        # samples around it, and the line says so
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        widened = 0.0
        while not inside and widened < 2.0:
            widened += 0.1
            inside = [p for t, p in self.samples if t0 - widened <= t <= t1 + widened]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[3 + i] == "Active"})
        res = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "samples": len(inside), "window_s": round(t1 - t0, 4)}
        if widened:
            res["widened_s"] = round(widened, 1)
        return res


def cpu_baseline(inp_cpu, budget_s=12.0, heads=2, causal=False, kind="hbm"):
    """The float64 oracle on `heads` query heads of the workload, repeated for
    about budget_s seconds on the host cores; reported in the metric's unit."""
    import oracle

    group = inp_cpu.h_q // inp_cpu.h_kv
    hs = list(range(heads))
    kvs = sorted({h // group for h in hs})
    def heads_of(x, idx):  # through bytes: CPU indexing of e4m3 tensors is not implemented
        if x.dtype == torch.float8_e4m3fn:
            return x.view(torch.uint8)[:, idx].view(x.dtype)
        return x[:, idx]

    q = heads_of(inp_cpu.q, hs)
    k = heads_of(inp_cpu.k, kvs)
    v = heads_of(inp_cpu.v, kvs)
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
    kw = {"kv": args.kv} if args.kv else {}
    if args.batch:
        kw["batch"] = args.batch
    paged = spec.get("paged", 0)
    case = Case(fa, dev, spec, num_splits=args.num_splits, flags=kernel_flag, rotate=not paged,
                kw_extra=kw)
    inp = case.inp
    ns = case.ns
    stream = torch.cuda.current_stream(dev)
    if paged:
        # the same keys, scattered into a shuffled page pool
        kc, vc, bt, sk = to_paged(inp, paged, dev)

        def call(i, s, extra=0):
            fa.fa_fwd_splitkv_paged(inp.q, kc, vc, case.cq, sk, bt, inp.max_seqlen_q, case.out,
                                    case.lse, case.ws, 0.0, causal, -1, args.num_splits, case.dq,
                                    case.dk, case.dv, kernel_flag | extra, s)
    else:
        call = case.call

    def graph_of(n, extra):
        """A CUDA graph of n calls (cycling through the input copies)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(n):
                call(i, side, extra)
        return g

    sampler = ClockSampler(local_rank)
    sampler.start()
    for i in range(args.warmup):
        call(i, stream)
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_error(clear=True) != 0:
        raise RuntimeError("device error during warm-up")
    # the partial kernel the library chose (the last call above enqueued it)
    kern_tag = KERNEL_TAGS[fa.fa_debug_last_kernel()]
    has_combine = ns > 1  # the split combine runs after the partial kernel

    # Timed region: exactly K steps (one library call each: partial kernel,
    # then the combine as its programmatic dependent when ns > 1), captured
    # in one CUDA graph so that no host work sits between them, replayed
    # once between a barrier and a synchronize.  Inputs under 256 MB rotate
    # over copies, so every step reads inputs that are not in L2.
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    graphs = {"step": graph_of(args.steps, 0),
              "partial": graph_of(args.steps, fa.FA_RUN_PARTIAL_ONLY)}
    if has_combine:
        graphs["combine"] = graph_of(args.steps, fa.FA_RUN_COMBINE_ONLY)

    def replay(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(side):
            e0.record(side)
            g.replay()
            e1.record(side)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1)

    # the partial graph replays once untimed first: its first replay pays
    # the graph upload
    replay(graphs["partial"])
    t_wall0 = time.time()
    total_ms = replay(graphs["step"])
    t_wall1 = time.time()
    # The dominant (partial) kernel alone, K launches, for its roofline; then
    # the combine alone over the same workspace.
    partial_ms = replay(graphs["partial"]) / args.steps
    combine_ms = replay(graphs["combine"]) / args.steps if has_combine else 0.0
    err = fa.fa_get_device_error(clear=True)
    if err != 0:
        raise RuntimeError(f"device error {fa.fa_status_string(err)}")
    del graphs

    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    metric_b, partial_bytes = byte_counts(inp, ns)
    work_flops = flops(inp, causal)
    if kind == "tensor":
        unit = "TFLOPS"
        value = job_throughput(work_flops, world, ms_per_step)
    else:
        unit = "TB/s"
        value = job_throughput(metric_b, world, ms_per_step)

    # ---- end to end with host buffers: packed K/V through the library's
    # host-buffer call (fa_fwd_splitkv_host: the copies to and from the
    # device are part of the call); paged K/V (no host-buffer call) copied
    # around the device call
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    q, k, v = case.copies[0]
    # the step's inputs: Q and cu_seqlens_q, and K/V with their index arrays
    dev_in = [q, case.cq] + ([kc, vc, bt, sk] if paged else [k, v, case.ck])
    host_in = [x.cpu().pin_memory() for x in dev_in]
    h_out = torch.empty(case.out.shape, dtype=case.out.dtype).pin_memory()
    h_lse = torch.empty(case.lse.shape, dtype=case.lse.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    dev_buf = None
    if paged:
        def e2e_step():
            for d_t, h_t in zip(dev_in, host_in):
                d_t.copy_(h_t, non_blocking=True)
            call(0, stream)
            h_out.copy_(case.out, non_blocking=True)
            h_lse.copy_(case.lse, non_blocking=True)
    else:
        hq, hcq, hk, hv, hck = host_in
        h_dsc = [None] * 3
        if inp.dtype == "e4m3":
            h_dsc = [d.cpu().pin_memory() for d in (case.dq, case.dk, case.dv)]
            h2d += 3 * 4
        nbuf = fa.fa_fwd_splitkv_host_buffer_size(
            inp.batch, hq.shape[0], hk.shape[0], inp.max_seqlen_q, inp.h_q, inp.h_kv, hq.shape[2],
            inp.d_v, hq.dtype, h_out.dtype, args.num_splits)
        dev_buf = torch.empty(nbuf, dtype=torch.uint8, device=dev)

        def e2e_step():
            fa.fa_fwd_splitkv_host(hq, hk, hv, hcq, hck, inp.max_seqlen_q, h_out, h_lse, dev_buf,
                                   0.0, causal, -1, args.num_splits, h_dsc[0], h_dsc[1], h_dsc[2],
                                   kernel_flag, stream)

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
    e2e_value = job_throughput(work_flops if kind == "tensor" else metric_b, world, e2e_ms)
    del case, host_in, e2e_step
    dev_buf = None
    torch.cuda.empty_cache()

    peak_gbs, peak_src = measured_peaks()
    tpeak, _, tpeak_src = measured_tensor_peak()
    cfg = None
    t_cfg0 = t_cfg1 = None
    if world == 1 and not args.no_configs and args.workload == "long_decode" and not args.kv \
            and not args.batch:
        t_cfg0 = time.time()
        cfg = config_fields(fa, dev, peak_gbs, tpeak)
        t_cfg1 = time.time()
        if fa.fa_get_device_error(clear=True) != 0:
            raise RuntimeError("device error during the configuration sweep")
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    if t_cfg0 is not None:
        clocks["all_timed_regions"] = sampler.summary(t_wall0, t_cfg1)

    if rank == 0:
        if kind == "tensor":
            achieved = work_flops / (partial_ms * 1e-3) / 1e12
            same_rate = "" if inp.dtype == "bf16" else f"; {inp.dtype} dense at the bf16 nominal rate (1:1)"
            roof = {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": achieved / tpeak,
                    "peak_source": tpeak_src + " bf16 dense (burst)" + same_rate,
                    "traffic": profiled_traffic(kern_tag, args.workload),
                    "kernel": f"{kern_tag} partial kernel", "partial_ms": partial_ms,
                    "timing": "K partial-only launches in one CUDA graph, CUDA events",
                    "algorithmic_flops_per_launch": work_flops}
        else:
            achieved_gbs = partial_bytes / (partial_ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": peak_gbs, "unit": "GB/s",
                    "frac": achieved_gbs / peak_gbs, "peak_source": peak_src,
                    "traffic": profiled_traffic(kern_tag, args.workload),
                    "kernel": f"{kern_tag} partial kernel", "partial_ms": partial_ms,
                    "combine_ms": combine_ms,
                    "timing": "K partial-only launches in one CUDA graph, CUDA events",
                    "algorithmic_bytes_per_launch": partial_bytes}
        in_bytes = sum(x.numel() * x.element_size() for x in (inp.q, inp.k, inp.v))
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if inp.dtype == "bf16" else inp.dtype, "data": "synthetic",
            "config": {"workload": spec["desc"], "num_splits": ns,
                       "num_splits_requested": args.num_splits, "kernel": kern_tag,
                       "l2": ("inputs larger than L2 (Q+K+V %.2f GB)" % (in_bytes / 1e9)
                              if in_bytes >= L2_FLUSH_BYTES else
                              "Q+K+V %.3f GB rotated over %d copies (256 MB read between two "
                              "uses of one copy)" % (in_bytes / 1e9, copies_for(in_bytes))),
                       "timing": "K steps captured in one CUDA graph, replayed once; CUDA events",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * (2 if has_combine else 1),
            "clocks": clocks,
        }
        if cfg is not None:
            line.update(cfg)
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(inp_host(inp), causal=causal, kind=kind)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
