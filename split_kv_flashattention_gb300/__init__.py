"""Split-KV flash-attention forward for GB300 (sm_103a).

Python binding of ``libfa_splitkv.so`` (C ABI in ``include/fa_splitkv.h``).
The functions here only marshal arguments: they read shapes and device
pointers off torch tensors and call the C entry points of the same name.
Every step of the computation runs in the library's CUDA kernels; there is
no fallback.  If the library has not been built the first call raises
``FaLibraryMissing``.

Build:  ``python -m split_kv_flashattention_gb300.build``
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "FaError", "FaLibraryMissing", "library", "fa_fwd_splitkv_ex", "fa_fwd_splitkv",
    "fa_fwd_splitkv_workspace_size", "fa_plan", "fa_debug_split_ranges", "fa_debug_wait_timeout",
    "fa_debug_last_kernel", "FA_KID_NONE", "FA_KID_SIMT", "FA_KID_UMMA", "FA_KID_UMMA2",
    "FA_KID_UMMA2_PERSISTENT",
    "fa_get_device_error", "fa_status_string", "fa_version", "forward",
    "FA_KERNEL_AUTO", "FA_KERNEL_SIMT", "FA_KERNEL_UMMA", "FA_KERNEL_UMMA2", "FA_RUN_PARTIAL_ONLY",
    "FA_RUN_COMBINE_ONLY", "DTYPE_CODES", "fa_fwd_splitkv_noalloc", "NOALLOC_SCRATCH_BYTES",
    "fa_fwd_splitkv_paged", "fa_fwd_splitkv_host", "fa_fwd_splitkv_host_buffer_size",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libfa_splitkv.so")
# the bounds-checking build (python -m split_kv_flashattention_gb300.build --debug),
# loaded instead when the environment variable FA_SPLITKV_DEBUG is 1
LIB_DEBUG_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib",
                              "libfa_splitkv_debug.so")

FA_KERNEL_AUTO, FA_KERNEL_SIMT, FA_KERNEL_UMMA, FA_KERNEL_UMMA2 = 0, 1, 2, 3
FA_RUN_PARTIAL_ONLY, FA_RUN_COMBINE_ONLY = 4, 8
FA_KID_NONE, FA_KID_SIMT, FA_KID_UMMA, FA_KID_UMMA2, FA_KID_UMMA2_PERSISTENT = 0, 1, 2, 3, 4
DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1, torch.float8_e4m3fn: 2}
EXPORTED = (
    "fa_fwd_splitkv_ex", "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_size", "fa_plan",
    "fa_debug_split_ranges", "fa_get_device_error", "fa_status_string", "fa_version",
    "fa_fwd_splitkv_noalloc", "fa_fwd_splitkv_paged", "fa_debug_wait_timeout",
    "fa_debug_last_kernel", "fa_fwd_splitkv_host", "fa_fwd_splitkv_host_buffer_size",
)
NOALLOC_SCRATCH_BYTES = 8 << 20


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {fa_status_string(status)} ({status})")
        self.status = status


class FaLibraryMissing(ImportError):
    pass


_lib = None

_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p


def library() -> ctypes.CDLL:
    """The loaded C library (loaded on first use)."""
    global _lib
    if _lib is not None:
        return _lib
    debug = os.environ.get("FA_SPLITKV_DEBUG") == "1"
    path = LIB_DEBUG_PATH if debug else LIB_PATH
    if not os.path.exists(path):
        raise FaLibraryMissing(
            f"{path} is missing; build it with python -m split_kv_flashattention_gb300.build"
            + (" --debug" if debug else ""))
    lib = ctypes.CDLL(path)
    lib.fa_fwd_splitkv_ex.restype = _c_int
    lib.fa_fwd_splitkv_ex.argtypes = [
        _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
        _c_float, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_size, _c_int, _c_int, _vp, _vp, _vp,
        _c_int, _vp]
    lib.fa_fwd_splitkv.restype = _c_int
    lib.fa_fwd_splitkv.argtypes = [
        _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
        _c_float, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp]
    lib.fa_fwd_splitkv_noalloc.restype = _c_int
    lib.fa_fwd_splitkv_noalloc.argtypes = [
        _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
        _c_float, _c_int, _c_int, _c_int, _vp, _vp, _c_int, _c_int, _vp, _vp, _vp, _c_int, _vp]
    lib.fa_fwd_splitkv_paged.restype = _c_int
    lib.fa_fwd_splitkv_paged.argtypes = [
        _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
        _c_int, _c_int, _c_int, _c_float, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_size, _c_int,
        _c_int, _vp, _vp, _vp, _c_int, _vp]
    lib.fa_fwd_splitkv_host.restype = _c_int
    lib.fa_fwd_splitkv_host.argtypes = [
        _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
        _c_float, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_size, _c_int, _c_int, _vp, _vp, _vp,
        _c_int, _vp]
    lib.fa_fwd_splitkv_host_buffer_size.restype = _c_size
    lib.fa_fwd_splitkv_host_buffer_size.argtypes = [_c_int] * 11
    lib.fa_fwd_splitkv_workspace_size.restype = _c_size
    lib.fa_fwd_splitkv_workspace_size.argtypes = [_c_int] * 6
    lib.fa_plan.restype = _c_int
    lib.fa_plan.argtypes = [_c_int] * 6 + [ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)]
    lib.fa_debug_split_ranges.restype = _c_int
    lib.fa_debug_split_ranges.argtypes = [_vp, _vp] + [_c_int] * 6 + [_vp, _vp]
    lib.fa_debug_wait_timeout.restype = _c_int
    lib.fa_debug_wait_timeout.argtypes = [ctypes.c_uint, _vp]
    lib.fa_debug_last_kernel.restype = _c_int
    lib.fa_debug_last_kernel.argtypes = []
    lib.fa_get_device_error.restype = _c_int
    lib.fa_get_device_error.argtypes = [_c_int]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [_c_int]
    lib.fa_version.restype = _c_int
    lib.fa_version.argtypes = []
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _tensor(t, name, shape=None, dtypes=None, optional=False):
    """Checks one argument before its pointer goes to the library, which only
    sees addresses: a strided view, a wrong dtype or shape, or host memory
    would otherwise be read as the packed device layout."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}; expected one of {sorted(map(str, dtypes))}")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}; expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on_device(ref, **tensors):
    """Every given tensor must live on the CUDA device of `ref`."""
    if not ref.is_cuda:
        raise ValueError("inputs must be CUDA tensors (device memory), got a "
                         f"{ref.device.type} tensor")
    dev = ref.get_device()
    for name, t in tensors.items():
        if t is not None and t.get_device() != dev:
            raise ValueError(f"{name} is on {t.device}, the inputs on {ref.device}")


_INPUT_DTYPES = tuple(DTYPE_CODES)
_I32 = (torch.int32,)
_F32 = (torch.float32,)


def _check_forward_args(q, k, v, cu_seqlens_q, seqlens_k_name, seqlens_k, out, lse, workspace,
                        descales, kv_ndim=3, on_host=False):
    """Shapes, dtypes, contiguity and device of a forward call's tensors (all
    in host memory when on_host)."""
    _tensor(q, "q", dtypes=_INPUT_DTYPES)
    _tensor(k, "k", dtypes=(q.dtype,))
    _tensor(v, "v", dtypes=(q.dtype,))
    if q.dim() != 3 or k.dim() != kv_ndim or v.dim() != kv_ndim:
        raise ValueError(f"q must be 3-D and k, v {kv_ndim}-D; got {q.dim()}, {k.dim()}, {v.dim()}")
    if tuple(k.shape[:-1]) != tuple(v.shape[:-1]):
        raise ValueError(f"k {tuple(k.shape)} and v {tuple(v.shape)} differ before the head dim")
    if k.shape[-1] != q.shape[2]:
        raise ValueError(f"q and k head dims differ ({q.shape[2]} vs {k.shape[-1]})")
    _tensor(cu_seqlens_q, "cu_seqlens_q", dtypes=_I32)
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q must be 1-D with batch+1 entries")
    batch = cu_seqlens_q.numel() - 1
    n_k = batch + 1 if seqlens_k_name == "cu_seqlens_k" else batch
    _tensor(seqlens_k, seqlens_k_name, shape=(n_k,), dtypes=_I32)
    total_q, h_q = q.shape[0], q.shape[1]
    _tensor(out, "out", shape=(total_q, h_q, v.shape[-1]), dtypes=_INPUT_DTYPES)
    _tensor(lse, "lse", shape=(h_q, total_q), dtypes=_F32, optional=True)
    _tensor(workspace, "workspace", optional=True)
    for name, d in descales.items():
        _tensor(d, name, dtypes=_F32, optional=True)
        if d is not None and d.numel() < 1:
            raise ValueError(f"{name} must hold one float32 value")
    if on_host:
        named = dict(q=q, k=k, v=v, cu_seqlens_q=cu_seqlens_q, **{seqlens_k_name: seqlens_k},
                     out=out, lse=lse, **descales)
        for name, t in named.items():
            if t is not None and t.is_cuda:
                raise ValueError(f"{name} must be a host (CPU) tensor, got {t.device}")
        return
    _on_device(q, k=k, v=v, cu_seqlens_q=cu_seqlens_q, **{seqlens_k_name: seqlens_k}, out=out,
               lse=lse, workspace=workspace, **descales)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise FaError(status, where)


def fa_status_string(status: int) -> str:
    return library().fa_status_string(int(status)).decode()


def fa_version() -> int:
    return library().fa_version()


def fa_plan(batch: int, max_seqlen_q: int, h_q: int, h_kv: int, num_splits: int = 0,
            num_sms: int = 0):
    """(num_splits, units) chosen by the planner; num_sms <= 0 queries the device."""
    ns, units = _c_int(0), _c_int(0)
    _check(library().fa_plan(batch, max_seqlen_q, h_q, h_kv, num_splits, num_sms,
                             ctypes.byref(ns), ctypes.byref(units)), "fa_plan")
    return ns.value, units.value


def fa_fwd_splitkv_workspace_size(batch: int, max_seqlen_q: int, h_q: int, h_kv: int, d_v: int,
                                  num_splits: int = 0) -> int:
    return int(library().fa_fwd_splitkv_workspace_size(batch, max_seqlen_q, h_q, h_kv, d_v,
                                                       num_splits))


def fa_debug_wait_timeout(timeout_ms: int, stream=None):
    """Test hook: a bounded device wait that runs out after timeout_ms and
    records FA_ERR_DEVICE_TIMEOUT (see the C header)."""
    _check(library().fa_debug_wait_timeout(int(timeout_ms), _stream(stream)), "fa_debug_wait_timeout")


def fa_debug_last_kernel() -> int:
    """Test hook: the partial kernel (FA_KID_*) that this thread's last forward
    call enqueued (see the C header)."""
    return int(library().fa_debug_last_kernel())


def fa_get_device_error(clear: bool = False) -> int:
    return library().fa_get_device_error(1 if clear else 0)


def fa_debug_split_ranges(cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, causal: bool,
                          window_left: int, num_splits: int, tile_queries: int, stream=None):
    """Device-computed key ranges, int32 [m_blocks, batch, num_splits, 2]."""
    _tensor(cu_seqlens_q, "cu_seqlens_q", dtypes=_I32)
    _tensor(cu_seqlens_k, "cu_seqlens_k", shape=tuple(cu_seqlens_q.shape), dtypes=_I32)
    _on_device(cu_seqlens_q, cu_seqlens_k=cu_seqlens_k)
    batch = cu_seqlens_q.numel() - 1
    m_blocks = -(-max_seqlen_q // tile_queries)
    out = torch.full((m_blocks, batch, num_splits, 2), -1, dtype=torch.int32,
                     device=cu_seqlens_q.device)
    _check(library().fa_debug_split_ranges(_ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch,
                                           max_seqlen_q, int(causal), window_left, num_splits,
                                           tile_queries, _ptr(out), _stream(stream)),
           "fa_debug_split_ranges")
    return out


def fa_fwd_splitkv_host_buffer_size(batch: int, total_q: int, total_k: int, max_seqlen_q: int,
                                    h_q: int, h_kv: int, d_qk: int, d_v: int, in_dtype,
                                    out_dtype, num_splits: int = 0) -> int:
    """Bytes of device buffer fa_fwd_splitkv_host needs (0: invalid sizes);
    in_dtype/out_dtype are torch dtypes."""
    return int(library().fa_fwd_splitkv_host_buffer_size(
        batch, total_q, total_k, max_seqlen_q, h_q, h_kv, d_qk, d_v, DTYPE_CODES[in_dtype],
        DTYPE_CODES[out_dtype], num_splits))


def fa_fwd_splitkv_host(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, out, lse,
                        device_buffer, scale: float = 0.0, causal: bool = False,
                        window_left: int = -1, num_splits: int = 0, descale_q=None,
                        descale_k=None, descale_v=None, flags: int = FA_KERNEL_AUTO,
                        stream=None):
    """Calls fa_fwd_splitkv_host: q, k, v, the offsets, out, lse and the
    descales are host (CPU) tensors, pinned for asynchronous copies;
    device_buffer is a CUDA tensor of at least
    fa_fwd_splitkv_host_buffer_size(...) bytes, 256-byte aligned.  The copies
    and the forward pass are enqueued on `stream`: synchronise it before
    reading out or lse."""
    _check_forward_args(q, k, v, cu_seqlens_q, "cu_seqlens_k", cu_seqlens_k, out, lse, None,
                        dict(descale_q=descale_q, descale_k=descale_k, descale_v=descale_v),
                        on_host=True)
    _tensor(device_buffer, "device_buffer")
    if not device_buffer.is_cuda:
        raise ValueError("device_buffer must be a CUDA tensor (device memory)")
    total_q, h_q, d_qk = q.shape
    total_k, h_kv, _ = k.shape
    d_v = v.shape[2]
    batch = cu_seqlens_q.numel() - 1
    nbytes = device_buffer.numel() * device_buffer.element_size()
    st = library().fa_fwd_splitkv_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, total_q,
        total_k, max_seqlen_q, h_q, h_kv, d_qk, d_v, float(scale), int(causal), int(window_left),
        int(num_splits), _ptr(out), _ptr(lse), _ptr(device_buffer), nbytes, DTYPE_CODES[q.dtype],
        DTYPE_CODES[out.dtype], _ptr(descale_q), _ptr(descale_k), _ptr(descale_v), int(flags),
        _stream(stream))
    _check(st, "fa_fwd_splitkv_host")


def fa_fwd_splitkv_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, out, lse=None,
                      workspace=None, scale: float = 0.0, causal: bool = False,
                      window_left: int = -1, num_splits: int = 0, descale_q=None,
                      descale_k=None, descale_v=None, flags: int = FA_KERNEL_AUTO,
                      stream=None):
    """Calls fa_fwd_splitkv_ex on torch CUDA tensors (shapes read from them).
    flags: FA_KERNEL_* optionally OR-ed with FA_RUN_PARTIAL_ONLY/COMBINE_ONLY."""
    _check_forward_args(q, k, v, cu_seqlens_q, "cu_seqlens_k", cu_seqlens_k, out, lse, workspace,
                        dict(descale_q=descale_q, descale_k=descale_k, descale_v=descale_v))
    total_q, h_q, d_qk = q.shape
    total_k, h_kv, _ = k.shape
    d_v = v.shape[2]
    batch = cu_seqlens_q.numel() - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = library().fa_fwd_splitkv_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, total_q,
        total_k, max_seqlen_q, h_q, h_kv, d_qk, d_v, float(scale), int(causal), int(window_left),
        int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, DTYPE_CODES[q.dtype],
        DTYPE_CODES[out.dtype], _ptr(descale_q), _ptr(descale_k), _ptr(descale_v), int(flags),
        _stream(stream))
    _check(st, "fa_fwd_splitkv_ex")


def fa_fwd_splitkv_noalloc(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, out,
                           lse=None, scale: float = 0.0, causal: bool = False,
                           window_left: int = -1, num_splits: int = 0, descale_q=None,
                           descale_k=None, descale_v=None, flags: int = FA_KERNEL_AUTO,
                           stream=None):
    """Calls fa_fwd_splitkv_noalloc: the forward pass without a caller
    workspace, for callers that cannot allocate device memory.  The split
    workspace is the library's fixed device array of NOALLOC_SCRATCH_BYTES;
    larger problems raise FaError(FA_ERR_WORKSPACE).  Calls that overlap on
    the GPU share that array and must be serialised by the caller."""
    _check_forward_args(q, k, v, cu_seqlens_q, "cu_seqlens_k", cu_seqlens_k, out, lse, None,
                        dict(descale_q=descale_q, descale_k=descale_k, descale_v=descale_v))
    total_q, h_q, d_qk = q.shape
    total_k, h_kv, _ = k.shape
    st = library().fa_fwd_splitkv_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        cu_seqlens_q.numel() - 1, total_q, total_k, max_seqlen_q, h_q, h_kv, d_qk, v.shape[2],
        float(scale), int(causal), int(window_left), int(num_splits), _ptr(out), _ptr(lse),
        DTYPE_CODES[q.dtype], DTYPE_CODES[out.dtype], _ptr(descale_q), _ptr(descale_k),
        _ptr(descale_v), int(flags), _stream(stream))
    _check(st, "fa_fwd_splitkv_noalloc")


def fa_fwd_splitkv_paged(q, k_cache, v_cache, cu_seqlens_q, seqlens_k, block_table,
                         max_seqlen_q: int, out, lse=None, workspace=None, scale: float = 0.0,
                         causal: bool = False, window_left: int = -1, num_splits: int = 0,
                         descale_q=None, descale_k=None, descale_v=None,
                         flags: int = FA_KERNEL_AUTO, stream=None):
    """Calls fa_fwd_splitkv_paged: K/V caches [num_pages, page_size, h_kv, d],
    block_table int32 [batch, max_pages], seqlens_k int32 [batch]."""
    _tensor(block_table, "block_table", dtypes=_I32)
    if block_table.dim() != 2 or block_table.shape[0] != cu_seqlens_q.numel() - 1:
        raise ValueError(f"block_table must be [batch, max_pages]; got {tuple(block_table.shape)}")
    _check_forward_args(q, k_cache, v_cache, cu_seqlens_q, "seqlens_k", seqlens_k, out, lse,
                        workspace,
                        dict(descale_q=descale_q, descale_k=descale_k, descale_v=descale_v),
                        kv_ndim=4)
    _on_device(q, block_table=block_table)
    total_q, h_q, d_qk = q.shape
    num_pages, page_size, h_kv, _ = k_cache.shape
    d_v = v_cache.shape[3]
    batch = cu_seqlens_q.numel() - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = library().fa_fwd_splitkv_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q), _ptr(seqlens_k),
        _ptr(block_table), batch, total_q, num_pages, page_size, block_table.shape[1],
        max_seqlen_q, h_q, h_kv, d_qk, d_v, float(scale), int(causal), int(window_left),
        int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, DTYPE_CODES[q.dtype],
        DTYPE_CODES[out.dtype], _ptr(descale_q), _ptr(descale_k), _ptr(descale_v), int(flags),
        _stream(stream))
    _check(st, "fa_fwd_splitkv_paged")


def fa_fwd_splitkv(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, out, lse=None,
                   workspace=None, scale: float = 0.0, causal: bool = False,
                   window_left: int = -1, num_splits: int = 0, stream=None):
    """Calls the bf16 shorthand entry point fa_fwd_splitkv."""
    _check_forward_args(q, k, v, cu_seqlens_q, "cu_seqlens_k", cu_seqlens_k, out, lse, workspace,
                        {})
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("fa_fwd_splitkv takes bf16 q, k, v and out; use fa_fwd_splitkv_ex")
    total_q, h_q, d_qk = q.shape
    total_k, h_kv, _ = k.shape
    st = library().fa_fwd_splitkv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        cu_seqlens_q.numel() - 1, total_q, total_k, max_seqlen_q, h_q, h_kv, d_qk, v.shape[2],
        float(scale), int(causal), int(window_left), int(num_splits), _ptr(out), _ptr(lse),
        _ptr(workspace), _stream(stream))
    _check(st, "fa_fwd_splitkv")


def forward(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, scale: float = 0.0,
            causal: bool = False, window_left: int = -1, num_splits: int = 0,
            descale_q=None, descale_k=None, descale_v=None, out_dtype=None,
            kernel: int = FA_KERNEL_AUTO, stream=None):
    """Allocates O, LSE and the workspace with torch, then calls
    fa_fwd_splitkv_ex.  Returns (out [total_q, h_q, d_v], lse [h_q, total_q])."""
    total_q, h_q, _ = q.shape
    h_kv, d_v = k.shape[1], v.shape[2]
    if out_dtype is None:
        out_dtype = torch.bfloat16 if q.dtype == torch.float8_e4m3fn else q.dtype
    out = torch.zeros((total_q, h_q, d_v), dtype=out_dtype, device=q.device)
    lse = torch.full((h_q, total_q), float("nan"), dtype=torch.float32, device=q.device)
    batch = cu_seqlens_q.numel() - 1
    ws_bytes = fa_fwd_splitkv_workspace_size(batch, max_seqlen_q, h_q, h_kv, d_v, num_splits)
    ws = torch.empty(max(ws_bytes, 16) // 4, dtype=torch.float32, device=q.device) if ws_bytes else None
    fa_fwd_splitkv_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, out, lse, ws, scale,
                      causal, window_left, num_splits, descale_q, descale_k, descale_v, kernel,
                      stream)
    return out, lse
