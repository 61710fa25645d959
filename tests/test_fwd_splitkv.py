"""Split-KV forward (fa_fwd_splitkv): key tiles cut into num_splits ranges,
merged by log-sum-exp.  Same bounds against the fp64 oracle as fa_fwd."""
import numpy as np
import pytest
import torch

from parity import compare_fwd, run_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,splits", [(129, 2), (640, 2), (640, 3), (640, 5), (1000, 4), (1000, 8)])
def test_parity_every_element(N, splits, d, causal):
    """Ragged tails, uneven ranges, ranges past the causal diagonal (empty for
    the first query blocks), num_splits up to the number of key tiles."""
    compare_fwd(2, 3, N, d, causal, seed=N + splits, num_splits=splits)


@pytest.mark.parametrize("causal", [False, True])
def test_stress(causal):
    compare_fwd(2, 4, 1024, 128, causal, stress=True, num_splits=3)


def test_long_context_few_heads():
    """B1 H4 N16384 causal in 8 ranges: 256 sampled rows per head."""
    compare_fwd(1, 4, 16384, 128, True, full_heads=0, rows_per_head=256, num_splits=8)


def test_close_to_unsplit():
    _, o1, l1, _ = run_fwd(1, 4, 2048, 128, False, seed=4)
    _, o2, l2, _ = run_fwd(1, 4, 2048, 128, False, seed=4, num_splits=4)
    assert np.abs(o1 - o2).max() < 1e-2 and np.abs(l1 - l2).max() < 1e-4


def test_argument_errors():
    from exact_attention_98_gb300 import fa

    q = torch.zeros((1, 2, 300, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 300), dtype=torch.float32, device="cuda")
    need = fa.fa_fwd_splitkv_workspace_bytes(1, 2, 300, 64, 2)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for bad in (0, 4):  # 300 keys are 3 key tiles
        with pytest.raises(fa.FAError):
            fa.fa_fwd_splitkv(q, q, q, o, lse, 0.125, False, bad, ws)
    with pytest.raises(fa.FAError):
        fa.fa_fwd_splitkv(q, q, q, o, lse, 0.125, False, 2, ws[: need - 256])
