"""Fits the polynomial of the kernels' software exp2 and writes exp2_poly_coeffs.h.

The forward pass evaluates part of its exponentials as a polynomial on the FMA
pipe instead of the MUFU unit (the "software-emulated exponential" of the
FlashAttention-4 abstract, item 2; "Программная эмуляция экспоненты" in
"FlashAttention-3 и FlashAttention-4").  The pages give neither degree nor
coefficients, so they are fitted here:

  2^x = 2^n * 2^f,   n = round-to-nearest(x),  f = x - n in [-1/2, 1/2]
  2^f ~ p(f) = 1 + c1 f + c2 f^2 + ... + cK f^K

p(0) = 1 is imposed so that exact powers of two (x an integer) come out
exact.  The remaining coefficients minimise the maximum RELATIVE error
|p(f) - 2^f| / 2^f on a dense grid of [-1/2, 1/2] -- discrete Chebyshev
(minimax) approximation solved as a linear program (minimise E subject to
-E <= (p(f_i) - 2^f_i) / 2^f_i <= E).  The coefficients are then rounded to
fp32 and the error of the fp32 Horner evaluation (each step one rounded FMA)
is measured on the grid; the lowest degree whose fp32 error stays below the
2e-4 relative bound with a 40% margin is kept.

Run from the repository root:  python exact_attention_98_gb300/csrc/fit_exp2_poly.py
"""
from __future__ import annotations

import os

import numpy as np
from scipy.optimize import linprog

BOUND = 2e-4


def fit(degree: int, n_grid: int = 20001):
    f = np.linspace(-0.5, 0.5, n_grid)
    target = np.exp2(f)
    # unknowns: c1..cK, E.  residual r_i = (1 + sum_k c_k f^k - 2^f) / 2^f
    powers = np.stack([f ** k for k in range(1, degree + 1)], axis=1) / target[:, None]
    const = (1.0 - target) / target
    ones = np.ones((n_grid, 1))
    a_ub = np.vstack([np.hstack([powers, -ones]), np.hstack([-powers, -ones])])
    b_ub = np.concatenate([-const, const])
    cost = np.zeros(degree + 1)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * (degree + 1), method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    return res.x[:degree], res.x[degree]


def fp32_horner(coeffs_f32, f):
    """1 + f*(c1 + f*(c2 + ...)) with each multiply-add rounded once to fp32."""
    f = f.astype(np.float32)
    acc = np.full_like(f, coeffs_f32[-1], dtype=np.float32)
    for c in coeffs_f32[-2::-1]:
        acc = (acc.astype(np.float64) * f.astype(np.float64) + np.float64(c)).astype(np.float32)
    return (acc.astype(np.float64) * f.astype(np.float64) + 1.0).astype(np.float32)


def fp32_error(coeffs_f32, n_grid: int = 200001):
    f = np.linspace(-0.5, 0.5, n_grid).astype(np.float32)
    p = fp32_horner(coeffs_f32, f).astype(np.float64)
    t = np.exp2(f.astype(np.float64))
    return float(np.max(np.abs(p - t) / t))


def main():
    for degree in range(2, 7):
        c, e = fit(degree)
        c32 = np.asarray(c, dtype=np.float32)
        e32 = fp32_error(c32)
        print(f"degree {degree}: minimax rel err {e:.3e}, fp32 evaluation {e32:.3e}")
        if e32 <= 0.6 * BOUND:
            break
    lines = [
        "// Written by fit_exp2_poly.py -- do not edit by hand.",
        f"// 2^f ~ 1 + c1 f + ... + c{degree} f^{degree} on f in [-1/2, 1/2];",
        f"// minimax relative error {e:.3e} (exact arithmetic), {e32:.3e} (fp32 Horner).",
        "#pragma once",
        f"#define FA_EXP2_POLY_DEGREE {degree}",
    ]
    for k, ck in enumerate(c32, start=1):
        lines.append(f"#define FA_EXP2_POLY_C{k} {float(ck)!r}f")
    lines.append(f"#define FA_EXP2_POLY_MAX_REL_ERR {e32:.6e}")
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "exp2_poly_coeffs.h")
    with open(out, "w") as fh:
        fh.write("\n".join(lines) + "\n")
    print("wrote", out)


if __name__ == "__main__":
    main()
