"""The fixed-token sweep (B*N = 32768 tokens, H = 16, N = 1k .. 32k, d = 64 and
128, both masks) and its softmax-stress variant, against the fp64 oracle.

Every configuration runs forward and backward on the GPU at full size.  Four
heads are compared on 256 sampled rows: O and LSE element by element, dQ rows by
relative Frobenius error, and on the first of them dK and dV rows too (the
oracle then forms that head's full LSE and D, O(N^2 d): tens of seconds at
N = 32768).  On the full tensors, two properties
of the exact gradients are checked at every size: each head's dK rows sum to
zero (rows of dS sum to zero), and each head's dV rows sum to its dO rows
(rows of P sum to one).  The backward takes O as the forward returns it, in
bf16, so the oracle forms D from its own O rounded to bf16 (see parity.py)."""
import numpy as np
import pytest

import oracle
from exact_attention_98_gb300.inputs import sampled_rows
from parity import check_grad, check_lse, check_o, run_fwd_bwd

pytestmark = pytest.mark.gpu

SWEEP = [(N, d, c) for N in (1024, 2048, 4096, 8192, 16384, 32768) for d in (64, 128)
         for c in (False, True)]
STRESS = [(N, 128, c) for N in (1024, 8192) for c in (False, True)]


def heads_to_check(B, H):
    picks = [(0, 0), (B - 1, H - 1), (B // 2, 5 % H), (0, 9 % H)]
    return sorted(set(picks))


def check_config(N, d, causal, stress):
    B, H = 32768 // N, 16
    inputs, (o, lse), (dq, dk, dv), scale = run_fwd_bwd(B, H, N, d, causal, seed=N + d,
                                                        stress=stress)
    q64, k64, v64, do64 = (t.double().numpy() for t in inputs)
    for n, (b, h) in enumerate(heads_to_check(B, H)):
        rows = sampled_rows(N, 256, b, h, H)
        what = f"sweep B{B} H{H} N{N} d{d} causal={causal} stress={stress} head ({b},{h})"
        o_ref, l_ref = oracle.fwd_head(q64[b, h], k64[b, h], v64[b, h], scale, causal, rows=rows)
        check_o(o[b, h][rows], o_ref, what)
        check_lse(lse[b, h][rows], l_ref, what)
        krows = rows if n == 0 else []
        g = oracle.bwd_head(q64[b, h], k64[b, h], v64[b, h], do64[b, h], scale, causal,
                            qrows=rows, krows=krows, o_bf16=True)
        check_grad(dq[b, h][rows], g[0], what + " dQ")
        if krows:
            check_grad(dk[b, h][krows], g[1], what + " dK")
            check_grad(dv[b, h][krows], g[2], what + " dV")
    # properties of the full gradients, every head
    dk_sum = np.abs(dk.sum(axis=2)).max()
    assert dk_sum <= 2e-2 * np.abs(dk).sum(axis=2).max(), dk_sum
    dv_err = np.abs(dv.sum(axis=2) - do64.sum(axis=2)).max()
    assert dv_err <= 2e-2 * np.abs(do64).sum(axis=2).max(), dv_err


@pytest.mark.parametrize("N,d,causal", SWEEP)
def test_sweep(N, d, causal):
    check_config(N, d, causal, stress=False)


@pytest.mark.parametrize("N,d,causal", STRESS)
def test_sweep_stress(N, d, causal):
    check_config(N, d, causal, stress=True)
