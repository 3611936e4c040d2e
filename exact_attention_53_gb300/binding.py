"""ctypes binding of libattn.so (declared in include/attn.h).

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream; every step of the attention forward runs in the library's
kernels.  There is no fallback: if the library cannot be loaded, or a call
returns an error status, :class:`AttnError` is raised.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_DTYPE_F16 = 0
ATTN_DTYPE_BF16 = 1

ATTN_MASK_NONE = 0
ATTN_MASK_CAUSAL = 1
ATTN_MASK_CAUSAL_BOTTOM_RIGHT = 2

EXPORTED = ("attn_fwd", "attn_fwd_general", "attn_fwd_host", "attn_fwd_plan", "attn_fwd_splitkv_plan",
            "attn_fwd_splitkv", "attn_fwd_splitkv_noalloc", "attn_bwd_workspace_size", "attn_bwd",
            "attn_bwd_general", "attn_fwd_splitkv_general_plan", "attn_fwd_splitkv_general",
            "attn_last_error", "attn_get_device_status", "attn_version")
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024    # ATTN_NOALLOC_SCRATCH_BYTES


class AttnPlan(ctypes.Structure):
    """Mirror of attn_plan_t (include/attn.h)."""
    _fields_ = [("block_m", ctypes.c_int64), ("block_n", ctypes.c_int64),
                ("q_tiles", ctypes.c_int64), ("kv_tiles", ctypes.c_int64),
                ("q_tiles_per_cta", ctypes.c_int64), ("bh", ctypes.c_int64),
                ("units", ctypes.c_int64), ("threads", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("tmem_cols", ctypes.c_int32),
                ("kv_stages", ctypes.c_int32)]

class AttnLayout(ctypes.Structure):
    """Mirror of attn_layout_t: element strides of batch, head and row."""
    _fields_ = [("batch", ctypes.c_int64), ("head", ctypes.c_int64), ("row", ctypes.c_int64)]


class AttnFwdParams(ctypes.Structure):
    """Mirror of attn_fwd_params_t (include/attn.h)."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("H_kv", ctypes.c_int64),
                ("S_q", ctypes.c_int64), ("S_k", ctypes.c_int64), ("d", ctypes.c_int64),
                ("q_layout", AttnLayout), ("k_layout", AttnLayout), ("v_layout", AttnLayout),
                ("o_layout", AttnLayout), ("mask", ctypes.c_int), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int)]


class AttnBwdParams(ctypes.Structure):
    """Mirror of attn_bwd_params_t (include/attn.h)."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("dout", ctypes.c_void_p),
                ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("H_kv", ctypes.c_int64),
                ("S_q", ctypes.c_int64), ("S_k", ctypes.c_int64), ("d", ctypes.c_int64),
                ("q_layout", AttnLayout), ("k_layout", AttnLayout), ("v_layout", AttnLayout),
                ("o_layout", AttnLayout), ("do_layout", AttnLayout), ("dq_layout", AttnLayout),
                ("dk_layout", AttnLayout), ("dv_layout", AttnLayout), ("mask", ctypes.c_int),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_int64)]


_DTYPE_CODE = {torch.float16: ATTN_DTYPE_F16, torch.bfloat16: ATTN_DTYPE_BF16}


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"attn status {status}: {message}")
        self.status = status
        self.message = message


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return os.environ.get("ATTN_LIBRARY", os.path.join(_PKG, "libattn.so"))


def load_library() -> ctypes.CDLL:
    """Open libattn.so (once) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise AttnError(ATTN_ERR_UNSUPPORTED,
                            f"{path} is missing; build it with exact_attention_53_gb300.build.build()")
        lib = ctypes.CDLL(path)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32,
                                 ctypes.c_float, i32, vp]
        lib.attn_fwd.restype = i32
        lib.attn_fwd_general.argtypes = [ctypes.POINTER(AttnFwdParams), vp]
        lib.attn_fwd_general.restype = i32
        lib.attn_fwd_splitkv_general_plan.argtypes = [ctypes.POINTER(AttnFwdParams), i64,
                                                      ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.attn_fwd_splitkv_general_plan.restype = i32
        lib.attn_fwd_splitkv_general.argtypes = [ctypes.POINTER(AttnFwdParams), i64, vp, i64, vp]
        lib.attn_fwd_splitkv_general.restype = i32
        lib.attn_bwd_general.argtypes = [ctypes.POINTER(AttnBwdParams), vp]
        lib.attn_bwd_general.restype = i32
        lib.attn_fwd_host.argtypes = [vp] * 10 + [i64, i64, i64, i64, i64, i32, ctypes.c_float,
                                                  i32, vp]
        lib.attn_fwd_host.restype = i32
        lib.attn_fwd_plan.argtypes = [i64, i64, i64, i64, i64, i32, i32, ctypes.POINTER(AttnPlan)]
        lib.attn_fwd_plan.restype = i32
        lib.attn_fwd_splitkv_plan.argtypes = [i64, i64, i64, i64, i64, i32, i64,
                                              ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.attn_fwd_splitkv_plan.restype = i32
        lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                         ctypes.c_float, i32, i64, vp, i64, vp]
        lib.attn_fwd_splitkv.restype = i32
        lib.attn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                                 ctypes.c_float, i32, i64, vp]
        lib.attn_fwd_splitkv_noalloc.restype = i32
        lib.attn_bwd_workspace_size.argtypes = [i64, i64, i64, i64, i64, i32, ctypes.POINTER(i64)]
        lib.attn_bwd_workspace_size.restype = i32
        lib.attn_bwd.argtypes = [vp] * 9 + [i64, i64, i64, i64, i64, i32, ctypes.c_float, i32, vp,
                                            i64, vp]
        lib.attn_bwd.restype = i32
        lib.attn_probe_ex2.argtypes = [vp, i32, i32, vp]
        lib.attn_probe_ex2.restype = i32
        lib.attn_last_error.argtypes = []
        lib.attn_last_error.restype = ctypes.c_char_p
        lib.attn_get_device_status.argtypes = [vp]
        lib.attn_get_device_status.restype = i32
        lib.attn_version.argtypes = []
        lib.attn_version.restype = i32
        _lib = lib
        return lib


DEBUG_EXPORTS = ("attn_debug_fwd", "attn_debug_bwd", "attn_debug_status")   # include/attn_debug.h
_debug_lib = None


def load_debug_library() -> ctypes.CDLL:
    """Open libattn_debug.so (once): the forward kernel built with 1 ms waits and a hook
    that makes one work unit's waits run out (include/attn_debug.h).  Tests only."""
    global _debug_lib
    with _lock:
        if _debug_lib is not None:
            return _debug_lib
        path = os.path.join(_PKG, "libattn_debug.so")
        if not os.path.exists(path):
            raise AttnError(ATTN_ERR_UNSUPPORTED,
                            f"{path} is missing; build it with exact_attention_53_gb300.build.build()")
        lib = ctypes.CDLL(path)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.attn_debug_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_float,
                                       ctypes.c_int, ctypes.c_uint64, vp]
        lib.attn_debug_fwd.restype = ctypes.c_int
        lib.attn_debug_bwd.argtypes = [vp] * 10 + [i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                                   ctypes.c_uint64, vp]
        lib.attn_debug_bwd.restype = ctypes.c_int
        lib.attn_debug_status.argtypes = [ctypes.POINTER(ctypes.c_uint), vp]
        lib.attn_debug_status.restype = ctypes.c_int
        _debug_lib = lib
        return lib


def attn_last_error() -> str:
    return load_library().attn_last_error().decode()


def _check(status: int) -> None:
    if status != ATTN_OK:
        raise AttnError(status, attn_last_error())


def _stream_handle(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def attn_fwd(q, k, v, o, lse, B, H, S_q, S_k, d, causal, scale, dtype, stream=None) -> None:
    """Enqueue the forward; q, k, v, o, lse are tensors or raw device pointers."""
    lib = load_library()
    ptr = lambda t: t.data_ptr() if isinstance(t, torch.Tensor) else t  # noqa: E731
    _check(lib.attn_fwd(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, S_q, S_k, d,
                        int(causal), float(scale), int(dtype), _stream_handle(stream)))


def attn_fwd_general(params: AttnFwdParams, stream=None) -> None:
    """Enqueue the general-layout forward described by ``params``."""
    _check(load_library().attn_fwd_general(ctypes.byref(params), _stream_handle(stream)))


def _layout(t: torch.Tensor) -> AttnLayout:
    if t.dim() != 4 or t.stride(3) != 1:
        raise AttnError(ATTN_ERR_INVALID_ARG, "tensors must be 4-D [B, heads, S, d] views with d contiguous")
    return AttnLayout(t.stride(0), t.stride(1), t.stride(2))


def fwd_general(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: int = ATTN_MASK_NONE,
                scale: float | None = None, out: torch.Tensor | None = None,
                lse: torch.Tensor | None = None):
    """Forward over strided views: q [B,H,S_q,d], k and v [B,H_kv,S_k,d] (any batch, head and
    row strides, d contiguous), H_kv dividing H.  ``out`` may be any strided [B,H,S_q,d] view
    (default: dense); ``lse`` is dense [B,H,S_q] fp32.  Returns ``(o, lse)``.
    """
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in _DTYPE_CODE:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "q, k, v must share dtype float16 or bfloat16")
    B, H, S_q, d = q.shape
    H_kv, S_k = k.shape[1], k.shape[2]
    if k.shape != (B, H_kv, S_k, d) or v.shape != k.shape:
        raise AttnError(ATTN_ERR_INVALID_ARG, f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, S_q, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
    p = AttnFwdParams(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      B, H, H_kv, S_q, S_k, d, _layout(q), _layout(k), _layout(v), _layout(out),
                      int(mask), float(scale), _DTYPE_CODE[q.dtype])
    attn_fwd_general(p)
    return out, lse


def _fwd_params(q, k, v, out, lse, mask, scale):
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in _DTYPE_CODE:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "q, k, v must share dtype float16 or bfloat16")
    B, H, S_q, d = q.shape
    H_kv, S_k = k.shape[1], k.shape[2]
    if k.shape != (B, H_kv, S_k, d) or v.shape != k.shape:
        raise AttnError(ATTN_ERR_INVALID_ARG, f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, S_q, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
    p = AttnFwdParams(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      B, H, H_kv, S_q, S_k, d, _layout(q), _layout(k), _layout(v), _layout(out),
                      int(mask), float(scale), _DTYPE_CODE[q.dtype])
    return p, out, lse


def attn_fwd_splitkv_general_plan(params: AttnFwdParams, n_split: int = 0) -> tuple[int, int]:
    """(ranges used, workspace bytes) of the general split-KV forward."""
    n_used, ws = ctypes.c_int64(), ctypes.c_int64()
    _check(load_library().attn_fwd_splitkv_general_plan(ctypes.byref(params), int(n_split),
                                                        ctypes.byref(n_used), ctypes.byref(ws)))
    return n_used.value, ws.value


def fwd_splitkv_general(q, k, v, n_split: int = 0, mask: int = ATTN_MASK_NONE,
                        scale: float | None = None, workspace=None, out=None, lse=None):
    """Split-KV forward over strided views with grouped key/value heads (see
    :func:`fwd_general`); returns ``(o, lse)``."""
    p, out, lse = _fwd_params(q, k, v, out, lse, mask, scale)
    _, ws = attn_fwd_splitkv_general_plan(p, n_split)
    if workspace is None:
        workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=q.device)
    _check(load_library().attn_fwd_splitkv_general(
        ctypes.byref(p), int(n_split), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(None)))
    return out, lse


def attn_fwd_host(q_host, k_host, v_host, o_host, lse_host, q_dev, k_dev, v_dev, o_dev, lse_dev,
                  B, H, S_q, S_k, d, causal, scale, dtype, stream=None) -> None:
    """Enqueue host→device copies, the forward, and device→host copies of O and LSE."""
    lib = load_library()
    ptr = lambda t: t.data_ptr() if isinstance(t, torch.Tensor) else t  # noqa: E731
    _check(lib.attn_fwd_host(ptr(q_host), ptr(k_host), ptr(v_host), ptr(o_host), ptr(lse_host),
                             ptr(q_dev), ptr(k_dev), ptr(v_dev), ptr(o_dev), ptr(lse_dev),
                             B, H, S_q, S_k, d, int(causal), float(scale), int(dtype),
                             _stream_handle(stream)))


def attn_fwd_plan(B, H, S_q, S_k, d, causal, dtype) -> AttnPlan:
    """The launch attn_fwd would use (host-only, no device needed)."""
    plan = AttnPlan()
    _check(load_library().attn_fwd_plan(B, H, S_q, S_k, d, int(causal), int(dtype),
                                        ctypes.byref(plan)))
    return plan


def attn_fwd_splitkv_plan(B, H, S_q, S_k, d, dtype, n_split=0) -> tuple[int, int]:
    """(ranges used, workspace bytes) for the split-KV forward; n_split 0 = automatic."""
    n_used, ws = ctypes.c_int64(), ctypes.c_int64()
    _check(load_library().attn_fwd_splitkv_plan(B, H, S_q, S_k, d, int(dtype), int(n_split),
                                                ctypes.byref(n_used), ctypes.byref(ws)))
    return n_used.value, ws.value


def attn_fwd_splitkv(q, k, v, o, lse, B, H, S_q, S_k, d, scale, dtype, n_split, workspace,
                     workspace_bytes, stream=None) -> None:
    """Enqueue the split-KV forward (full attention); tensors or raw device pointers."""
    lib = load_library()
    ptr = lambda t: t.data_ptr() if isinstance(t, torch.Tensor) else t  # noqa: E731
    _check(lib.attn_fwd_splitkv(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, S_q, S_k, d,
                                float(scale), int(dtype), int(n_split), ptr(workspace),
                                int(workspace_bytes), _stream_handle(stream)))


def attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, S_q, S_k, d, scale, dtype, n_split,
                             stream=None) -> None:
    """Enqueue the split-KV forward on the library's built-in scratch (no workspace)."""
    lib = load_library()
    ptr = lambda t: t.data_ptr() if isinstance(t, torch.Tensor) else t  # noqa: E731
    _check(lib.attn_fwd_splitkv_noalloc(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, S_q, S_k,
                                        d, float(scale), int(dtype), int(n_split),
                                        _stream_handle(stream)))


def attn_bwd_workspace_size(B, H, S_q, S_k, d, dtype) -> int:
    """Workspace bytes attn_bwd needs (host-only)."""
    ws = ctypes.c_int64()
    _check(load_library().attn_bwd_workspace_size(B, H, S_q, S_k, d, int(dtype), ctypes.byref(ws)))
    return ws.value


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, S_q, S_k, d, causal, scale, dtype,
             workspace, workspace_bytes, stream=None) -> None:
    """Enqueue the backward; tensors or raw device pointers."""
    lib = load_library()
    ptr = lambda t: t.data_ptr() if isinstance(t, torch.Tensor) else t  # noqa: E731
    _check(lib.attn_bwd(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(dout), ptr(dq), ptr(dk),
                        ptr(dv), B, H, S_q, S_k, d, int(causal), float(scale), int(dtype),
                        ptr(workspace), int(workspace_bytes), _stream_handle(stream)))


PROBES = ("attn_probe_ex2",)     # declared in include/attn_probe.h


def probe_ex2_rate(blocks: int = 0, iters: int = 4096) -> float:
    """ex2.approx evaluations per second on the current device (MUFU throughput)."""
    lib = load_library()
    if blocks <= 0:
        blocks = 8 * torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = torch.empty(blocks * 256, dtype=torch.float32, device="cuda")
    st = _stream_handle(None)
    for _ in range(2):
        if lib.attn_probe_ex2(out.data_ptr(), blocks, iters, st) != 0:
            raise AttnError(ATTN_ERR_CUDA, "attn_probe_ex2 failed")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    lib.attn_probe_ex2(out.data_ptr(), blocks, iters, st)
    b.record()
    torch.cuda.synchronize()
    return blocks * 256 * 8 * iters / (a.elapsed_time(b) * 1e-3)


def attn_get_device_status(stream=None) -> None:
    """Synchronise and raise AttnError(ATTN_ERR_TIMEOUT) if a kernel's wait ran out."""
    _check(load_library().attn_get_device_status(_stream_handle(stream)))


def _check_qkv(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise AttnError(ATTN_ERR_INVALID_ARG, "q, k, v must be 4-D [B,H,S,d]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise AttnError(ATTN_ERR_INVALID_ARG, "q, k, v must be contiguous")
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in _DTYPE_CODE:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "q, k, v must share dtype float16 or bfloat16")
    B, H, S_q, d = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape != k.shape:
        raise AttnError(ATTN_ERR_INVALID_ARG, f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    return B, H, S_q, k.shape[2], d


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: float | None = None, out: torch.Tensor | None = None,
        lse: torch.Tensor | None = None):
    """O, LSE for contiguous CUDA tensors q [B,H,S_q,d], k, v [B,H,S_k,d].

    ``scale`` defaults to 1/sqrt(d).  Outputs are allocated with torch unless
    given.  Returns ``(o, lse)``; work is enqueued on the current stream.
    """
    B, H, S_q, S_k, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, v, out, lse, B, H, S_q, S_k, d, causal, scale, _DTYPE_CODE[q.dtype])
    return out, lse


def fwd_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_split: int = 0,
                scale: float | None = None, workspace: torch.Tensor | None = None,
                out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """Split-KV forward (full attention) of contiguous CUDA tensors; see :func:`fwd`.

    ``n_split`` 0 lets the library choose.  The workspace is allocated with
    torch unless given (a uint8 tensor of at least the planned size).
    Returns ``(o, lse)``.
    """
    B, H, S_q, S_k, d = _check_qkv(q, k, v)
    dtype = _DTYPE_CODE[q.dtype]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _, ws = attn_fwd_splitkv_plan(B, H, S_q, S_k, d, dtype, n_split)
    if workspace is None:
        workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
    attn_fwd_splitkv(q, k, v, out, lse, B, H, S_q, S_k, d, scale, dtype, n_split, workspace,
                     workspace.numel() * workspace.element_size())
    return out, lse


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
        dout: torch.Tensor, causal: bool = False, scale: float | None = None,
        workspace: torch.Tensor | None = None):
    """dQ, dK, dV for contiguous CUDA tensors (the forward's q, k, v, o, lse and dO).

    Outputs and (unless given) the workspace are allocated with torch; work is
    enqueued on the current stream.  Returns ``(dq, dk, dv)``.
    """
    B, H, S_q, S_k, d = _check_qkv(q, k, v)
    if o.shape != q.shape or dout.shape != q.shape or o.dtype != q.dtype or dout.dtype != q.dtype:
        raise AttnError(ATTN_ERR_INVALID_ARG, "o and dout must match q in shape and dtype")
    if not (o.is_contiguous() and dout.is_contiguous() and lse.is_contiguous()):
        raise AttnError(ATTN_ERR_INVALID_ARG, "o, dout and lse must be contiguous")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, S_q):
        raise AttnError(ATTN_ERR_INVALID_ARG, "lse must be float32 [B, H, S_q]")
    dtype = _DTYPE_CODE[q.dtype]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws = attn_bwd_workspace_size(B, H, S_q, S_k, d, dtype)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, S_q, S_k, d, causal, scale, dtype,
             workspace, workspace.numel() * workspace.element_size())
    return dq, dk, dv


def attn_bwd_general(params: AttnBwdParams, stream=None) -> None:
    """Enqueue the general-layout backward described by ``params``."""
    _check(load_library().attn_bwd_general(ctypes.byref(params), _stream_handle(stream)))


def bwd_general(q, k, v, o, lse, dout, mask: int = ATTN_MASK_NONE, scale: float | None = None,
                dq=None, dk=None, dv=None, workspace=None):
    """Backward over strided views (shapes as :func:`fwd_general`).  Gradients are written into
    the given views (default: dense tensors).  Returns ``(dq, dk, dv)``.
    """
    B, H, S_q, d = q.shape
    H_kv, S_k = k.shape[1], k.shape[2]
    dtype = _DTYPE_CODE[q.dtype]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty((B, H, S_q, d), dtype=q.dtype, device=q.device) if dq is None else dq
    dk = torch.empty((B, H_kv, S_k, d), dtype=q.dtype, device=q.device) if dk is None else dk
    dv = torch.empty((B, H_kv, S_k, d), dtype=q.dtype, device=q.device) if dv is None else dv
    ws = attn_bwd_workspace_size(B, H, S_q, S_k, d, dtype)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=q.device)
    p = AttnBwdParams(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                      B, H, H_kv, S_q, S_k, d, _layout(q), _layout(k), _layout(v), _layout(o),
                      _layout(dout), _layout(dq), _layout(dk), _layout(dv), int(mask), float(scale),
                      dtype, workspace.data_ptr(), workspace.numel() * workspace.element_size())
    attn_bwd_general(p)
    return dq, dk, dv
