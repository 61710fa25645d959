"""FP8 forward with incoherent processing, step by step on the CPU (numpy,
fp64 arithmetic on e4m3-rounded values).  Test infrastructure: only tests,
smoke() and the bench's CPU leg use it.

What the step computes ("FlashAttention-3 и FlashAttention-4", section
"Поддержка FP8 с контролем ошибок": before quantisation a cheap transform
spreads outliers over the coordinates):
  1. rotate Q and K along the head dimension with R = diag(sigma) H / sqrt(d),
     H the Sylvester-Hadamard matrix, sigma_i = -1 when bit 31 of
     (0x9E3779B1 * (i + 1)) mod 2^32 is set, else +1 (R is orthogonal, so
     (Q R)(K R)^T = Q K^T);
  2. quantise to e4m3 (round to nearest even, saturating at 448): Q with one
     scale per row, K and V with one scale per (batch, head), each scale
     448 / amax;
  3. S = scale * (Q8 K8^T) * descales, softmax with the row max, P * 64
     rounded to e4m3, O = (P8 V8) * V descale / (64 * sum of the unrounded P),
     LSE = max + ln(sum P).
Readings (the pages give no recipe beyond item 1): the scale granularity,
the factor 64 on P, and that the row sum uses the unrounded P.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def rot_signs(d: int) -> np.ndarray:
    i = np.arange(d, dtype=np.uint64)
    h = (np.uint64(0x9E3779B1) * (i + np.uint64(1))) & np.uint64(0xFFFFFFFF)
    return np.where((h >> np.uint64(31)) & np.uint64(1), -1.0, 1.0)


def hadamard(d: int) -> np.ndarray:
    """Sylvester-Hadamard matrix of order d (a power of two), entries +-1."""
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation(d: int) -> np.ndarray:
    return np.diag(rot_signs(d)) @ hadamard(d) / np.sqrt(d)


def round_e4m3(x) -> np.ndarray:
    """Nearest e4m3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits; subnormals below 2^-6 in steps of 2^-9; ties to even), saturating
    at +-448."""
    x = np.clip(np.asarray(x, dtype=np.float64), -E4M3_MAX, E4M3_MAX)
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -6)))  # exponent, floored at the subnormal range
    step = 2.0 ** (e - 3)
    return np.sign(x) * np.rint(ax / step) * step  # np.rint rounds ties to even


def quantise(x, axis=None):
    """e4m3 values and descale (amax / 448; 1 where amax is 0) with one scale
    per `axis` slice (None: one for the whole array)."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max(axis=axis, keepdims=axis is not None)
    s = np.where(amax > 0, E4M3_MAX / np.where(amax > 0, amax, 1.0), 1.0)
    return round_e4m3(x * s), 1.0 / s


def attention_quantised(q8, qd, k8, kd, v8, vd, scale: float, causal: bool):
    """Step 3 on given e4m3 operands: q8 [N, d] with row descales qd [N, 1],
    k8 [N, d] and v8 [N, d] with scalar descales kd, vd."""
    N = q8.shape[0]
    s = scale * (q8 @ k8.T) * qd * kd
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    p8 = round_e4m3(p * 64.0)
    o = (p8 @ v8) * vd / (64.0 * l)
    return o, (m + np.log(l))[:, 0]


def forward_head(q, k, v, scale: float, causal: bool, rotate: bool = True):
    """q, k, v: [N, d] (the bf16 inputs as fp64).  Returns (o, lse)."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    d = q.shape[1]
    if rotate:
        r = rotation(d)
        q, k = q @ r, k @ r
    q8, qd = quantise(q, axis=1)
    k8, kd = quantise(k)
    v8, vd = quantise(v)
    return attention_quantised(q8, qd, k8, kd, v8, vd, scale, causal)
