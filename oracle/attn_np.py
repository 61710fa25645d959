"""NumPy restatement of the exact-attention definition, for tiny inputs.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).  It states the
same definition as ``attn_f64.c`` with whole-matrix NumPy operations; the tests
use it to cross-check the C oracle and as the function whose finite
differences pin the backward formulas.

Forward (plain softmax attention, the mechanism the FlashAttention pages say is
left unchanged by their schedules): S = scale * Q K^T, masked to key <= query
when causal; P = softmax_rows(S); O = P V; LSE = ln sum_j exp(S_ij).
Backward of L = sum(O * dO) by the chain rule: dV = P^T dO, dP = dO V^T,
D = rowsum(dO * O), dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.
"""
from __future__ import annotations

import numpy as np


def _mask(N: int, causal: bool) -> np.ndarray:
    if not causal:
        return np.ones((N, N), dtype=bool)
    return np.tril(np.ones((N, N), dtype=bool))


def forward(q, k, v, scale: float, causal: bool):
    """q, k, v: [N, d] float64.  Returns (o [N, d], lse [N], p [N, N])."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    N = q.shape[0]
    s = scale * (q @ k.T)
    allowed = _mask(N, causal)
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.where(allowed, np.exp(s - m), 0.0)
    l = e.sum(axis=1, keepdims=True)
    p = e / l
    o = p @ v
    lse = (m + np.log(l))[:, 0]
    return o, lse, p


def round_bf16(x):
    """Nearest bf16 value of each element (8 significant bits, ties to even)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def backward(q, k, v, dout, scale: float, causal: bool, o_bf16: bool = False):
    """Gradients of sum(O * dO).  Returns (dq, dk, dv), each [N, d].  o_bf16:
    D = rowsum(dO * O) from O rounded to bf16 (the backward's O input as the
    library carries it) instead of the exact O."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    o, _, p = forward(q, k, v, scale, causal)
    dv = p.T @ dout
    dp = dout @ v.T
    D = (dout * (round_bf16(o) if o_bf16 else o)).sum(axis=1, keepdims=True)
    ds = p * (dp - D)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv
