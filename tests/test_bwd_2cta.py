"""The backward by CTA pairs (fa_bwd_2cta: two CTAs on consecutive key tiles
share every product as one tcgen05 cta_group::2 MMA; "Режим 2-CTA MMA" of
"FlashAttention-3 и FlashAttention-4") against the fp64 oracle with the
backward's bound (relative Frobenius error <= 2e-2 on dQ, dK, dV), on the
shapes of the single-CTA backward's tests: every element on small, ragged
and odd-key-tile shapes (a pair whose second key tile lies past N), the
softmax-stress inputs, and B2 H16 N8192 causal on sampled rows; plus its
agreement with fa_bwd on the same inputs."""
import math

import numpy as np
import pytest
import torch

from parity import compare_bwd, run_bwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 100, 128, 129, 200, 256, 383, 512, 640])
def test_ragged_and_multi_tile(N, causal):
    compare_bwd(2, 2, N, 128, causal, seed=7 * N + 128, two_cta=True)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_stress(causal):
    compare_bwd(1, 3, 768, 128, causal, stress=True, two_cta=True)


def test_b2_h16_n8192_causal():
    """B2 H16 N8192 d128 causal: head 0 on every row; 256 sampled dQ rows on
    every other head and sampled dK/dV rows on two more heads; then the
    properties of the full tensors (dK rows sum to zero, dV rows to dO's)."""
    worst, (dq, dk, dv), inputs = compare_bwd(2, 16, 8192, 128, True, full_heads=1,
                                             rows_per_head=256, kv_heads=(1, 17), two_cta=True)
    do = inputs[3].double().numpy()
    s = np.abs(dk.sum(axis=2)).max()
    assert s <= 2e-2 * np.abs(dk).sum(axis=2).max(), s
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), rtol=0, atol=0.5)


@pytest.mark.parametrize("causal", [False, True])
def test_agrees_with_single_cta_backward(causal):
    """Same inputs through fa_bwd and fa_bwd_2cta: dK and dV within bf16
    rounding of each other, dQ within the order of its fp32 additions."""
    _, (dq1, dk1, dv1), _ = run_bwd(2, 4, 1000, 128, causal, seed=5)
    _, (dq2, dk2, dv2), _ = run_bwd(2, 4, 1000, 128, causal, seed=5, two_cta=True)
    for a, b in ((dk1, dk2), (dv1, dv2), (dq1, dq2)):
        assert np.linalg.norm(a - b) <= 2e-3 * np.linalg.norm(a)


def test_unsupported_head_dim():
    from exact_attention_98_gb300 import fa

    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    ws = fa.workspace_for(q)
    with pytest.raises(fa.FAError) as e:
        fa.fa_bwd_2cta(q, q, q, q, lse, q, q, q, q, 0.125, False, ws)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
