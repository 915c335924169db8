"""CPU tests of the C ABI: the library loads, exports every symbol the header
declares, plans splits exactly like the oracle's integer rule and rejects bad
arguments synchronously.  No compute call touches a GPU here."""

import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_splitkv.h")


@pytest.fixture(scope="module")
def fa():
    import split_kv_flashattention_gb300 as pkg
    if not os.path.exists(pkg.LIB_PATH):
        from split_kv_flashattention_gb300 import build
        build.build()
    pkg.library()
    return pkg


def _declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_expected_entry_points():
    syms = _declared_symbols()
    for s in ("fa_fwd_splitkv", "fa_fwd_splitkv_ex", "fa_fwd_splitkv_workspace_size",
              "fa_plan", "fa_get_device_error", "fa_status_string", "fa_debug_split_ranges"):
        assert s in syms


# What a declaration's comment must name: one of the pages the library
# follows, or the statement that the pages have no counterpart.
PAGE_NAMES = ('flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference"',
              'aiter PR "[FlyDSL] Enable FP8 FMHA split-K for short cached-prefix queries"',
              'cutlass "Adds variable sequence lengths to the Hopper CuTe DSL FMHA example"')
NO_COUNTERPART = ("no counterpart", "do not describe")


def test_every_declaration_cites_a_page_or_says_it_has_none():
    text = open(HEADER).read()
    # the comment text between the previous declaration (or the top of the
    # file's declarations) and each FA_API declaration, whitespace collapsed
    decls = list(re.finditer(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text))
    assert decls
    prev_end = text.index("extern \"C\"")
    for m in decls:
        block = " ".join(text[prev_end:m.start()].replace("*", " ").split())
        page = any(" ".join(p.split()) in block for p in PAGE_NAMES)
        short = any(k in block for k in ('flash-attention PR', 'aiter PR', 'cutlass PR'))
        none = any(k in block for k in NO_COUNTERPART)
        assert page or short or none, f"{m.group(1)}: no page cited"
        prev_end = text.index(";", m.end())


def test_library_exports_every_declared_symbol(fa):
    lib = ctypes.CDLL(fa.LIB_PATH)
    for s in _declared_symbols():
        assert hasattr(lib, s), s
    assert set(_declared_symbols()) == set(fa.EXPORTED)


def test_status_strings(fa):
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(-1) == "FA_ERR_INVALID_ARG"
    assert fa.fa_status_string(-3) == "FA_ERR_WORKSPACE"
    assert fa.fa_status_string(-5) == "FA_ERR_DEVICE_TIMEOUT"
    assert fa.fa_status_string(-7) == "FA_ERR_DEVICE_BOUNDS"
    assert fa.fa_status_string(12345) == "FA_UNKNOWN_STATUS"


def test_plan_matches_golden_cases(fa):
    with open(os.path.join(ROOT, "tests", "golden", "planner_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert fa.fa_plan(*c["args"]) == (c["ns"], c["units"]), c


def test_plan_bit_exact_against_oracle_sweep(fa):
    rng = np.random.default_rng(0)
    for _ in range(3000):
        h_kv = int(rng.choice([1, 2, 4, 8, 12, 16, 32]))
        group = int(rng.choice([1, 2, 3, 4, 8, 16]))
        args = (int(rng.integers(0, 64)), int(rng.integers(0, 5000)), h_kv * group, h_kv,
                int(rng.choice([0, 0, 0, 1, 3, 16, 128, 200])), int(rng.choice([132, 148, 152, 160])))
        assert fa.fa_plan(*args) == oracle.plan_num_splits(*args), args


def test_workspace_size_explicit_splits(fa):
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 32, 32, 128, 1) == 16  # tile counter
    for ns in (2, 9, 128):
        assert fa.fa_fwd_splitkv_workspace_size(3, 70, 12, 4, 128, ns) == \
            oracle.workspace_bytes(3, 70, 12, 128, ns)
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 32, 32, 128, 129) == 0  # invalid
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 3, 2, 128, 4) == 0      # h_q % h_kv


def _call_ex(fa, **kw):
    """fa_fwd_splitkv_ex with fake (never dereferenced) aligned pointers."""
    a = dict(q=0x1000, k=0x2000, v=0x3000, cu_q=0x4000, cu_k=0x5000, batch=2, total_q=2,
             total_k=100, max_seqlen_q=1, h_q=8, h_kv=2, d_qk=128, d_v=128, scale=0.0,
             causal=0, window_left=-1, num_splits=1, out=0x6000, lse=0x7000, ws=0,
             ws_bytes=0, in_dtype=0, out_dtype=0, dq=0, dk=0, dv=0, flags=0, stream=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return fa.library().fa_fwd_splitkv_ex(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["cu_q"]), vp(a["cu_k"]), a["batch"],
        a["total_q"], a["total_k"], a["max_seqlen_q"], a["h_q"], a["h_kv"], a["d_qk"], a["d_v"],
        a["scale"], a["causal"], a["window_left"], a["num_splits"], vp(a["out"]), vp(a["lse"]),
        vp(a["ws"]), a["ws_bytes"], a["in_dtype"], a["out_dtype"], vp(a["dq"]), vp(a["dk"]),
        vp(a["dv"]), a["flags"], vp(a["stream"]))


@pytest.mark.parametrize("kw,status", [
    (dict(h_q=6, h_kv=4), -1),                     # heads not divisible
    (dict(h_q=258, h_kv=1), -1),                   # group > 128
    (dict(num_splits=-1), -1),
    (dict(num_splits=129), -1),                    # more than 128 splits
    (dict(batch=-1), -1),
    (dict(d_qk=96, d_v=96), -2),                   # unsupported head dim
    (dict(d_qk=256, d_v=128), -2),                 # unequal 16-bit dims
    (dict(d_qk=256, d_v=256, flags=3), -2),        # two-tile kernel: head dim <= 128
    (dict(d_qk=192, d_v=128), -2),                 # 192 only for e4m3
    (dict(in_dtype=0, out_dtype=1), -2),           # bf16 in, fp16 out
    (dict(in_dtype=7), -1),
    (dict(out_dtype=3), -1),                       # unknown output type
    (dict(in_dtype=1, out_dtype=0), -2),           # fp16 in, bf16 out
    (dict(q=0x1008), -1),                          # unaligned q
    (dict(out=0x6004), -1),                        # unaligned out
    (dict(lse=0x7002), -1),                        # unaligned lse
    (dict(q=0), -1),                               # null input
    (dict(in_dtype=2, out_dtype=0, d_qk=192), -1),  # fp8 without descales
    (dict(scale=float("nan")), -1),
    (dict(flags=3, in_dtype=2, out_dtype=0, d_qk=192, dq=0x9000, dk=0x9000, dv=0x9000), -2),
    (dict(flags=16), -1),                          # unknown flag bit
    (dict(flags=12), -1),                          # partial-only and combine-only
    (dict(num_splits=4, ws=0), -3),                # split without workspace
    (dict(num_splits=4, ws=0x8000, ws_bytes=16), -3),  # workspace too small
    (dict(num_splits=4, ws=0x8004, ws_bytes=1 << 20), -3),  # unaligned workspace
])
def test_argument_errors_are_synchronous(fa, kw, status):
    assert _call_ex(fa, **kw) == status
    assert fa.fa_debug_last_kernel() == fa.FA_KID_NONE  # nothing enqueued


def test_empty_problem_is_a_noop(fa):
    assert _call_ex(fa, batch=0) == 0
    assert fa.fa_debug_last_kernel() == fa.FA_KID_NONE
    assert _call_ex(fa, max_seqlen_q=0) == 0
    assert _call_ex(fa, total_q=0) == 0


def _call_paged(fa, **kw):
    a = dict(q=0x1000, kc=0x2000, vc=0x3000, cu_q=0x4000, seqlens=0x5000, table=0x5800, batch=2,
             total_q=2, num_pages=8, page_size=64, max_pages=4, max_seqlen_q=1, h_q=8, h_kv=2,
             d_qk=128, d_v=128, scale=0.0, causal=0, window_left=-1, num_splits=1, out=0x6000,
             lse=0x7000, ws=0, ws_bytes=0, in_dtype=0, out_dtype=0, flags=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return fa.library().fa_fwd_splitkv_paged(
        vp(a["q"]), vp(a["kc"]), vp(a["vc"]), vp(a["cu_q"]), vp(a["seqlens"]), vp(a["table"]),
        a["batch"], a["total_q"], a["num_pages"], a["page_size"], a["max_pages"],
        a["max_seqlen_q"], a["h_q"], a["h_kv"], a["d_qk"], a["d_v"], a["scale"], a["causal"],
        a["window_left"], a["num_splits"], vp(a["out"]), vp(a["lse"]), vp(a["ws"]), a["ws_bytes"],
        a["in_dtype"], a["out_dtype"], vp(0), vp(0), vp(0), a["flags"], vp(0))


@pytest.mark.parametrize("kw,status", [
    (dict(page_size=48), -1),        # not a power of two
    (dict(page_size=16), -1),        # below the 32-row load granularity
    (dict(table=0), -1),             # no block table
    (dict(seqlens=0), -1),           # no key counts
    (dict(num_pages=0), -1),         # empty pool
    (dict(max_pages=0), -1),
    (dict(d_qk=96, d_v=96), -2),
    (dict(kc=0x2008), -1),           # unaligned cache
])
def test_paged_argument_errors(fa, kw, status):
    assert _call_paged(fa, **kw) == status


def test_paged_empty_problem_is_a_noop(fa):
    assert _call_paged(fa, batch=0) == 0


@pytest.mark.parametrize("timeout_ms", [0, 10001])
def test_wait_timeout_hook_rejects_bad_timeouts(fa, timeout_ms):
    """The bounded-wait test hook validates its timeout before any CUDA call."""
    assert fa.library().fa_debug_wait_timeout(timeout_ms, None) == -1
