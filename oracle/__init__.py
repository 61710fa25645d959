"""fp64 CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library in
``exact_attention_98_gb300`` never imports it, and the two share no code.

``attn_f64.c`` holds the plain definition (see its header for the formulas and
the passages they follow); this module only marshals numpy arrays into it.
``attn_np.py`` is a NumPy restatement of the same definition for tiny inputs.
``fp8.py`` restates the FP8 forward's recipe (rotation, e4m3 quantisation,
attention on the quantised operands) step by step, for the FP8 tests.

Arrays are float64, row-major.  Tensors of shape [B, H, N, d] are processed one
(batch, head) slice at a time.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_f64.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_f64.c into liboracle.so (gcc, OpenMP). Returns the path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            lib.oracle_fwd_rows.argtypes = [dp, ctypes.c_int, ip, dp, dp, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_double, ctypes.c_int, dp, dp]
            lib.oracle_fwd_rows.restype = ctypes.c_int
            lib.oracle_bwd_rows.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int, ip, ctypes.c_int, dp,
                                            ip, ctypes.c_int, dp, dp, ctypes.c_int]
            lib.oracle_bwd_rows.restype = ctypes.c_int
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16.restype = ctypes.c_double
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().oracle_num_threads())


def fwd_head(q, k, v, scale: float, causal: bool, rows=None):
    """Forward of one head.  q, k, v: [N, d].  rows: query positions to compute
    (default all).  Returns (o [R, d], lse [R]) for those rows."""
    lib = _load()
    k = _f64(k)
    v = _f64(v)
    q = _f64(q)
    N, d = k.shape
    if rows is None:
        rows = np.arange(N, dtype=np.int32)
    rows = _i32(rows)
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise ValueError("query row out of range")
    qs = _f64(q[rows])
    o = np.empty((len(rows), d), dtype=np.float64)
    lse = np.empty((len(rows),), dtype=np.float64)
    rc = lib.oracle_fwd_rows(_dp(qs), len(rows), _ip(rows), _dp(k), _dp(v), N, d,
                             float(scale), int(bool(causal)), _dp(o), _dp(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_fwd_rows failed with code {rc}")
    return o, lse


def round_bf16(x: float) -> float:
    """x rounded to the nearest bf16 value (ties to even), as the oracle does it."""
    return float(_load().oracle_round_bf16(float(x)))


def bwd_head(q, k, v, dout, scale: float, causal: bool, qrows=None, krows=None,
             o_bf16: bool = False):
    """Backward of one head with loss sum(O * dO).  q, k, v, dout: [N, d].
    qrows: rows of dQ to compute (default all); krows: rows of dK/dV (default
    all).  o_bf16: form D = rowsum(dO * O) from the oracle's own O rounded to
    bf16 -- the backward's O input as the library's API carries it -- instead
    of the exact fp64 O.  Returns (dq [len(qrows), d], dk [len(krows), d],
    dv [len(krows), d])."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    N, d = k.shape
    qrows = _i32(np.arange(N) if qrows is None else qrows)
    krows = _i32(np.arange(N) if krows is None else krows)
    dq = np.empty((len(qrows), d), dtype=np.float64)
    dk = np.empty((len(krows), d), dtype=np.float64)
    dv = np.empty((len(krows), d), dtype=np.float64)
    rc = lib.oracle_bwd_rows(_dp(q), _dp(k), _dp(v), _dp(dout), N, d, float(scale),
                             int(bool(causal)), _ip(qrows), len(qrows), _dp(dq),
                             _ip(krows), len(krows), _dp(dk), _dp(dv), int(bool(o_bf16)))
    if rc != 0:
        raise RuntimeError(f"oracle_bwd_rows failed with code {rc}")
    return dq, dk, dv


def fwd(q, k, v, scale: float, causal: bool):
    """Full forward over [B, H, N, d].  Returns (o [B,H,N,d], lse [B,H,N])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = fwd_head(q[b, h], k[b, h], v[b, h], scale, causal)
    return o, lse


def bwd(q, k, v, dout, scale: float, causal: bool, o_bf16: bool = False):
    """Full backward over [B, H, N, d].  Returns (dq, dk, dv), each [B,H,N,d]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = q.shape
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = bwd_head(q[b, h], k[b, h], v[b, h], dout[b, h],
                                                    scale, causal, o_bf16=o_bf16)
    return dq, dk, dv
