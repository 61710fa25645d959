"""CTA-pair forward (fa_fwd_2cta): two CTAs share every product as one
M = 256 MMA, each loading half of every K and V tile.  Same bounds against
the fp64 oracle as fa_fwd."""
import numpy as np
import pytest
import torch

from parity import compare_fwd, run_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 256, 300, 512, 640, 1000, 1536])
def test_parity_every_element(N, causal):
    """Pair items of 512 rows: one, several and a ragged last one; query
    tiles of the pair past N (one CTA's, or both CTAs' second tile)."""
    compare_fwd(2, 3, N, 128, causal, seed=N + 7, two_cta=True)


@pytest.mark.parametrize("causal", [False, True])
def test_stress(causal):
    compare_fwd(2, 4, 1024, 128, causal, stress=True, two_cta=True)


@pytest.mark.parametrize("causal", [False, True])
def test_bench_shape_sampled(causal):
    """B2 H16 N4096: more items than pairs (persistent walk), 256 sampled rows
    per head after two full heads."""
    compare_fwd(2, 16, 4096, 128, causal, full_heads=2, rows_per_head=256, two_cta=True)


def test_long_causal_sampled():
    compare_fwd(1, 2, 16384, 128, True, full_heads=0, rows_per_head=256, two_cta=True)


def test_close_to_single_cta():
    """The pair and the single-CTA kernel round the same products in the same
    order per row, so they agree to far below the oracle bound."""
    _, o1, l1, _ = run_fwd(2, 4, 2048, 128, True, seed=4)
    _, o2, l2, _ = run_fwd(2, 4, 2048, 128, True, seed=4, two_cta=True)
    assert np.abs(o1 - o2).max() < 1e-2 and np.abs(l1 - l2).max() < 1e-4


def test_argument_errors():
    from exact_attention_98_gb300 import fa

    q = torch.zeros((1, 2, 300, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 300), dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError):  # d = 64 is not built for pairs
        fa.fa_fwd_2cta(q, q, q, o, lse, 0.125, False)
