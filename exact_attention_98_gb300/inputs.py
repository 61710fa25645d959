"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle side.

This module holds none of the attention arithmetic: it only draws the bf16
tensors that both the CUDA path and the fp64 oracle receive, and picks the rows
that a sampled comparison looks at.

Recipe (all on the CPU with ``torch.Generator().manual_seed(seed)``):
  * Q, K, V, dO are drawn in that order as ``randn`` fp32 of shape [B, H, N, d]
    and rounded to bf16 (round-to-nearest-even).
  * The softmax-stress variant draws Q and K with standard deviation 3 and
    multiplies 1% of the key rows (the first floor(0.01 N) entries of
    ``randperm(N)`` under seed 2, the same rows for every head) by 8 before the
    bf16 rounding; V and dO stay N(0, 1).  Peaked rows exercise the running max
    and the conditional rescale.
  * Sampled rows of head (b, h): sorted(randperm(N, seed 1 + b*H + h)[:k])
    together with rows 0 and N-1.
  * Problems too large to draw on the host (tens of GB) are drawn one head at
    a time on the device: Q, K, V, dO of head h as ``randn`` fp32 [4, N, d]
    from a generator of that device seeded with seed * 1000003 + h, rounded
    to bf16 (same distribution, a different stream).
"""
from __future__ import annotations

import torch


def attention_inputs(B: int, H: int, N: int, d: int, seed: int = 0, stress: bool = False,
                     with_dout: bool = True):
    """Returns (q, k, v, dout) as contiguous CPU bf16 tensors [B, H, N, d]
    (dout is None when ``with_dout`` is False)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    dout = torch.randn(shape, generator=g, dtype=torch.float32) if with_dout else None
    if stress:
        q.mul_(3.0)
        k.mul_(3.0)
        n_hot = (N * 1) // 100
        if n_hot > 0:
            g2 = torch.Generator(device="cpu").manual_seed(2)
            hot = torch.randperm(N, generator=g2)[:n_hot]
            k[:, :, hot, :] *= 8.0
    to_bf16 = lambda t: None if t is None else t.to(torch.bfloat16).contiguous()
    return to_bf16(q), to_bf16(k), to_bf16(v), to_bf16(dout)


def sampled_rows(N: int, k: int, b: int, h: int, H: int):
    """Row indices compared for head (b, h) in a sampled check (sorted, unique)."""
    g = torch.Generator(device="cpu").manual_seed(1 + b * H + h)
    pick = torch.randperm(N, generator=g)[: min(k, N)]
    rows = set(int(x) for x in pick.tolist())
    rows.update({0, N - 1})
    return sorted(rows)


def device_head_inputs(N: int, d: int, seed: int, head: int, device):
    """Returns (q, k, v, dout) of one head, each a bf16 [N, d] tensor on
    ``device``, drawn there (see the module docstring)."""
    g = torch.Generator(device=device).manual_seed(int(seed) * 1000003 + int(head))
    x = torch.randn((4, N, d), generator=g, device=device, dtype=torch.float32)
    return tuple(x[i].to(torch.bfloat16) for i in range(4))
