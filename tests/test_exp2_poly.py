"""The software exp2 (polynomial on the FMA pipe) against fp64 exp2.

Bound: max relative error <= 2e-4 over the kernels' clamped domain.  The host
test evaluates the fitted constants with the kernel's algorithm in fp32
emulation; the GPU test runs the kernels' own device function.
"""
import os
import re

import numpy as np
import pytest
import torch

BOUND = 2e-4
COEFFS_H = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "exact_attention_98_gb300", "csrc", "exp2_poly_coeffs.h")


def coeffs():
    text = open(COEFFS_H).read()
    deg = int(re.search(r"FA_EXP2_POLY_DEGREE (\d+)", text).group(1))
    return [np.float32(float(re.search(rf"FA_EXP2_POLY_C{k} ([-0-9.eE+]+)f", text).group(1)))
            for k in range(1, deg + 1)]


def grid():
    # dense sweep of the clamped domain plus every integer and the edges
    x = np.concatenate([np.linspace(-125.0, 127.0, 2_000_001), np.arange(-125, 128),
                        np.linspace(-1.0, 1.0, 200_001)]).astype(np.float32)
    return x


def emulate(x: np.ndarray) -> np.ndarray:
    """The kernel's steps in fp32: t = x + 1.5*2^23 (rounds x to n), f = x - n,
    Horner with one rounding per FMA, then n added to the exponent bits."""
    c = coeffs()
    x = np.clip(x.astype(np.float32), -125.0, 127.0).astype(np.float32)
    t = (x + np.float32(12582912.0)).astype(np.float32)
    n = (t - np.float32(12582912.0)).astype(np.float32)
    f = (x - n).astype(np.float32)

    def fma(a, b, cc):
        return (a.astype(np.float64) * b.astype(np.float64) + np.float64(cc)).astype(np.float32)

    p = fma(np.full_like(f, c[2]), f, c[1])
    p = fma(p, f, c[0])
    p = fma(p, f, 1.0)
    bits = (p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23)) \
        & np.uint64(0xFFFFFFFF)
    return bits.astype(np.uint32).view(np.float32)


def test_fitted_constants_meet_bound_host():
    assert len(coeffs()) == 3
    x = grid()
    y = emulate(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y - ref) / ref
    assert rel.max() <= BOUND, rel.max()


def test_integers_are_exact_host():
    x = np.arange(-125, 128).astype(np.float32)
    assert np.array_equal(emulate(x).astype(np.float64), np.exp2(x.astype(np.float64)))


@pytest.mark.gpu
def test_device_exp2_poly_meets_bound():
    from exact_attention_98_gb300 import fa

    x = torch.from_numpy(grid())
    xd = x.cuda()
    yd = torch.empty_like(xd)
    fa.fa_exp2_poly_eval(xd, yd)
    y = yd.cpu().double().numpy()
    ref = np.exp2(x.double().numpy())
    rel = np.abs(y - ref) / ref
    assert rel.max() <= BOUND, rel.max()
    # integers exact, and the host emulation reproduces the device bit for bit
    ints = np.arange(-125, 128).astype(np.float32)
    yi = torch.empty(len(ints), dtype=torch.float32, device="cuda")
    fa.fa_exp2_poly_eval(torch.from_numpy(ints).cuda(), yi)
    assert np.array_equal(yi.cpu().double().numpy(), np.exp2(ints.astype(np.float64)))
    assert np.array_equal(y.astype(np.float32), emulate(x.numpy()))
