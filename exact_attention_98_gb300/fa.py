"""Python binding of libfa.so (include/fa.h), argument marshalling only.

The functions with the C names (``fa_fwd``, ``fa_bwd``, ...) take torch CUDA
tensors that the caller allocated and pass their device pointers, sizes and the
current CUDA stream straight to the C ABI; every step of the computation runs
in the library's kernels.  ``forward`` / ``backward`` are conveniences that
allocate the outputs with torch and then call those.

There is no fallback: if libfa.so is missing or cannot be loaded, importing
this module raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fa.h")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_WORKSPACE = 5
FA_ERR_TOO_LARGE = 6


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where} failed: {status_string(code)} ({code})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m exact_attention_98_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.fa_fwd_workspace_bytes.restype = sz
    lib.fa_set_exp2_poly_share.argtypes = [i]
    lib.fa_set_exp2_poly_share.restype = i
    lib.fa_get_exp2_poly_share.argtypes = []
    lib.fa_get_exp2_poly_share.restype = i
    lib.fa_fwd_2cta.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_fwd_2cta.restype = i
    lib.fa_fwd_splitkv_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.fa_fwd_splitkv_workspace_bytes.restype = sz
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_fwd_fp8_workspace_bytes.restype = sz
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_bytes.restype = sz
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd.restype = i
    lib.fa_last_device_status.argtypes = [vp]
    lib.fa_last_device_status.restype = i
    lib.fa_last_device_site.argtypes = []
    lib.fa_last_device_site.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_exp2_poly_eval.argtypes = [vp, vp, ctypes.c_longlong, vp]
    lib.fa_exp2_poly_eval.restype = i
    lib.fa_debug_bounded_wait.argtypes = [ctypes.c_ulonglong, vp]
    lib.fa_debug_bounded_wait.restype = i
    lib.fa_bwd_2cta.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd_2cta.restype = i
    lib.fa_bwd_deterministic_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_bwd_deterministic_workspace_bytes.restype = sz
    lib.fa_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp,
                                         sz, vp]
    lib.fa_bwd_deterministic.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_timing_enable.argtypes = [i]
    lib.fa_timing_enable.restype = i
    lib.fa_timing_last_ms.argtypes = [i, ctypes.POINTER(ctypes.c_float)]
    lib.fa_timing_last_ms.restype = i
    lib.fa_launch_count.argtypes = []
    lib.fa_launch_count.restype = ctypes.c_ulonglong
    return lib


lib = _load()


def declared_functions() -> list[str]:
    """Names of the functions include/fa.h declares."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^[ \t]*(?:const[ \t]+)?(?:\w+[ \t]+)*\w+[ \t]*\*?[ \t]*(fa_\w+)\s*\(",
                                 text, re.M)))


def status_string(code: int) -> str:
    return lib.fa_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != FA_OK:
        raise FAError(code, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d]")
    return tuple(int(x) for x in q.shape)


def _check_tensor(t, name, dtype, shape, device=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_attention(q, names_and_tensors, lse):
    """Shape, dtype, device and layout checks shared by the forward and
    backward calls; every operand lives on q's device."""
    B, H, N, d = _shape(q)
    if q.is_cuda and q.device.index != torch.cuda.current_device():
        raise ValueError(f"q is on {q.device}; the library launches on the current device "
                         f"cuda:{torch.cuda.current_device()}")
    for name, t in names_and_tensors:
        _check_tensor(t, name, torch.bfloat16, (B, H, N, d), q.device)
    _check_tensor(lse, "lse", torch.float32, (B, H, N), q.device)
    return B, H, N, d


def _workspace(ws, device):
    """(pointer, bytes) of a caller workspace: None, or a contiguous CUDA
    tensor on the operands' device (the library checks size and alignment)."""
    if ws is None:
        return None, 0
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or ws.device != device:
        raise ValueError(f"workspace must be a CUDA tensor on {device}")
    if not ws.is_contiguous():
        raise ValueError("workspace must be contiguous")
    return _ptr(ws), ws.numel() * ws.element_size()


# --- the C entry points --------------------------------------------------------


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool, workspace=None, stream=None) -> None:
    """workspace: None, or a CUDA tensor of at least fa_fwd_workspace_bytes()
    bytes that lets the call split its last partial round of work."""
    B, H, N, d = _check_attention(q, (("q", q), ("k", k), ("v", v), ("o", o)), lse)
    ws_ptr, ws_bytes = _workspace(workspace, q.device)
    _check(lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                      int(bool(causal)), ws_ptr, ws_bytes, _stream(stream)), "fa_fwd")


def fa_fwd_workspace_bytes(B: int, H: int, N: int, d: int, causal: bool) -> int:
    return int(lib.fa_fwd_workspace_bytes(B, H, N, d, int(bool(causal))))


def fa_set_exp2_poly_share(per_octet: int) -> None:
    _check(lib.fa_set_exp2_poly_share(int(per_octet)), "fa_set_exp2_poly_share")


def fa_get_exp2_poly_share() -> int:
    return int(lib.fa_get_exp2_poly_share())


def fa_fwd_2cta(q, k, v, o, lse, scale: float, causal: bool, stream=None) -> None:
    """fa_fwd computed by CTA pairs sharing each M = 256 product (d = 128)."""
    B, H, N, d = _check_attention(q, (("q", q), ("k", k), ("v", v), ("o", o)), lse)
    _check(lib.fa_fwd_2cta(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                           int(bool(causal)), _stream(stream)), "fa_fwd_2cta")


def fa_fwd_splitkv_workspace_bytes(B: int, H: int, N: int, d: int, num_splits: int) -> int:
    return int(lib.fa_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits))


def fa_fwd_splitkv(q, k, v, o, lse, scale: float, causal: bool, num_splits: int, workspace,
                   stream=None) -> None:
    B, H, N, d = _check_attention(q, (("q", q), ("k", k), ("v", v), ("o", o)), lse)
    ws_ptr, ws_bytes = _workspace(workspace, q.device)
    _check(lib.fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                              float(scale), int(bool(causal)), int(num_splits), ws_ptr,
                              ws_bytes, _stream(stream)), "fa_fwd_splitkv")


def fa_fwd_fp8_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib.fa_fwd_fp8_workspace_bytes(B, H, N, d))


def fa_fwd_fp8(q, k, v, o, lse, scale: float, causal: bool, rotate: bool, workspace,
               stream=None) -> None:
    B, H, N, d = _check_attention(q, (("q", q), ("k", k), ("v", v), ("o", o)), lse)
    ws_ptr, ws_bytes = _workspace(workspace, q.device)
    _check(lib.fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                          int(bool(causal)), int(bool(rotate)), ws_ptr, ws_bytes,
                          _stream(stream)), "fa_fwd_fp8")


def forward_fp8(q, k, v, causal: bool = False, scale: float | None = None, rotate: bool = True,
                stream=None):
    """FP8 forward (fa_fwd_fp8); returns (o, lse) freshly allocated."""
    B, H, N, d = _shape(q)
    scale = default_scale(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    ws = torch.empty(max(fa_fwd_fp8_workspace_bytes(B, H, N, d), 1), dtype=torch.uint8,
                     device=q.device)
    fa_fwd_fp8(q, k, v, o, lse, scale, causal, rotate, ws, stream)
    return o, lse


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib.fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, scale: float, causal: bool, workspace,
           stream=None) -> None:
    B, H, N, d = _check_attention(q, (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout),
                                      ("dq", dq), ("dk", dk), ("dv", dv)), lse)
    ws_ptr, ws_bytes = _workspace(workspace, q.device)
    _check(lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                      _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                      ws_ptr, ws_bytes, _stream(stream)), "fa_bwd")


def fa_bwd_2cta(q, k, v, o, lse, dout, dq, dk, dv, scale: float, causal: bool, workspace,
                stream=None) -> None:
    """fa_bwd computed by CTA pairs sharing each product (d = 128); same
    workspace as fa_bwd."""
    B, H, N, d = _check_attention(q, (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout),
                                      ("dq", dq), ("dk", dk), ("dv", dv)), lse)
    ws_ptr, ws_bytes = _workspace(workspace, q.device)
    _check(lib.fa_bwd_2cta(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                           _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                           ws_ptr, ws_bytes, _stream(stream)), "fa_bwd_2cta")


def fa_bwd_deterministic_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib.fa_bwd_deterministic_workspace_bytes(B, H, N, d))


def fa_bwd_deterministic(q, k, v, o, lse, dout, dq, dk, dv, scale: float, causal: bool,
                         workspace, stream=None) -> None:
    """fa_bwd with run-to-run bit-identical results (no dQ atomics)."""
    B, H, N, d = _check_attention(q, (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout),
                                      ("dq", dq), ("dk", dk), ("dv", dv)), lse)
    ws_ptr, ws_bytes = _workspace(workspace, q.device)
    _check(lib.fa_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                    _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                    int(bool(causal)), ws_ptr, ws_bytes,
                                    _stream(stream)), "fa_bwd_deterministic")


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, scale: float, causal: bool,
                   stream=None) -> None:
    """fa_bwd with the library's fixed scratch array instead of a caller
    workspace: for callers that cannot allocate device memory."""
    B, H, N, d = _check_attention(q, (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout),
                                      ("dq", dq), ("dk", dk), ("dv", dv)), lse)
    _check(lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                              _stream(stream)), "fa_bwd_noalloc")


def fa_last_device_status(stream=None) -> int:
    return int(lib.fa_last_device_status(_stream(stream)))


def fa_last_device_site() -> int:
    return int(lib.fa_last_device_site())


def fa_status_string(code: int) -> str:
    return status_string(code)


def fa_exp2_poly_eval(x, y, stream=None) -> None:
    _check_tensor(x, "x", torch.float32, x.shape)
    _check_tensor(y, "y", torch.float32, x.shape)
    _check(lib.fa_exp2_poly_eval(_ptr(x), _ptr(y), x.numel(), _stream(stream)),
           "fa_exp2_poly_eval")


def fa_debug_bounded_wait(limit_ns: int, stream=None) -> None:
    _check(lib.fa_debug_bounded_wait(int(limit_ns), _stream(stream)), "fa_debug_bounded_wait")


KERNEL_FWD = 0
KERNEL_BWD_MAIN = 1


def fa_timing_enable(enable: bool) -> None:
    _check(lib.fa_timing_enable(int(bool(enable))), "fa_timing_enable")


def fa_timing_last_ms(kernel: int) -> float:
    ms = ctypes.c_float(0.0)
    _check(lib.fa_timing_last_ms(int(kernel), ctypes.byref(ms)), "fa_timing_last_ms")
    return float(ms.value)


def fa_launch_count() -> int:
    return int(lib.fa_launch_count())


# --- conveniences ----------------------------------------------------------------


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None,
            num_splits: int = 1, two_cta: bool = False):
    """Returns (o, lse) freshly allocated on q's device.  num_splits > 1:
    split-KV forward (fa_fwd_splitkv) with a freshly allocated workspace;
    two_cta: the CTA-pair forward (fa_fwd_2cta)."""
    B, H, N, d = _shape(q)
    scale = default_scale(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if two_cta:
        if num_splits != 1:
            raise ValueError("the CTA-pair forward has no key-range split")
        fa_fwd_2cta(q, k, v, o, lse, scale, causal, stream)
    elif num_splits == 1:
        fa_fwd(q, k, v, o, lse, scale, causal, fwd_workspace_for(q, causal), stream)
    else:
        n = fa_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
        fa_fwd_splitkv(q, k, v, o, lse, scale, causal, num_splits, ws, stream)
    return o, lse


def fwd_workspace_for(q, causal: bool):
    """fa_fwd's optional workspace for q's shape on the current device (None
    when the call would not use one)."""
    B, H, N, d = _shape(q)
    n = fa_fwd_workspace_bytes(B, H, N, d, causal)
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n > 0 else None


def workspace_for(q, deterministic: bool = False):
    B, H, N, d = _shape(q)
    n = (fa_bwd_deterministic_workspace_bytes if deterministic else fa_bwd_workspace_bytes)(
        B, H, N, d)
    # torch's caching allocator hands out 512-byte aligned blocks
    return torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
             workspace=None, stream=None, deterministic: bool = False, two_cta: bool = False):
    """Returns (dq, dk, dv) freshly allocated on q's device.  deterministic:
    fa_bwd_deterministic (bit-identical from run to run) instead of fa_bwd;
    two_cta: the CTA-pair backward (fa_bwd_2cta)."""
    B, H, N, d = _shape(q)
    scale = default_scale(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    if deterministic and two_cta:
        raise ValueError("the CTA-pair backward adds dQ with atomics")
    if workspace is None:
        workspace = workspace_for(q, deterministic)
    run = fa_bwd_deterministic if deterministic else fa_bwd_2cta if two_cta else fa_bwd
    run(q, k, v, o, lse, dout, dq, dk, dv, scale, causal, workspace, stream)
    return dq, dk, dv
