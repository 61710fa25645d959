"""The deterministic backward (fa_bwd_deterministic): dK and dV from the
key-stationary kernel without its dQ product and dQ from a query-stationary
kernel adding the key tiles in order in tensor memory, with no fp32 atomics.
Same bounds against the fp64 oracle as fa_bwd, and bit-identical results
from run to run."""
import numpy as np
import pytest
import torch

from parity import compare_bwd, run_bwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 383, 640])
def test_parity_every_element(N, d, causal):
    compare_bwd(2, 3, N, d, causal, seed=N + d + 7, deterministic=True)


@pytest.mark.parametrize("causal", [False, True])
def test_stress(causal):
    compare_bwd(2, 4, 1024, 128, causal, stress=True, deterministic=True)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bit_identical_runs(d, causal):
    """Two runs on the same inputs give the same bits for dQ, dK and dV."""
    _, g1, _ = run_bwd(2, 4, 1000, d, causal, seed=5, deterministic=True)
    _, g2, _ = run_bwd(2, 4, 1000, d, causal, seed=5, deterministic=True)
    for a, b, name in zip(g1, g2, ("dq", "dk", "dv")):
        assert np.array_equal(a, b), name


def test_matches_atomic_backward():
    """dK and dV do not depend on the dQ path; dQ differs from the atomic
    backward only by the order of fp32 additions."""
    _, ga, _ = run_bwd(1, 4, 2048, 128, False, seed=9)
    _, gd, _ = run_bwd(1, 4, 2048, 128, False, seed=9, deterministic=True)
    assert np.array_equal(ga[1], gd[1]) and np.array_equal(ga[2], gd[2])
    rel = np.linalg.norm(ga[0] - gd[0]) / np.linalg.norm(gd[0])
    assert rel < 1e-3, rel


def test_b2_h16_n4096_d128_causal_sampled():
    compare_bwd(2, 16, 4096, 128, True, full_heads=1, rows_per_head=256, kv_heads=(5, 17),
                deterministic=True)


def test_short_workspace_is_rejected():
    from exact_attention_98_gb300 import fa

    q = torch.zeros((1, 2, 256, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 256), dtype=torch.float32, device="cuda")
    need = fa.fa_bwd_deterministic_workspace_bytes(1, 2, 256, 64)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError):
        fa.fa_bwd_deterministic(q, q, q, q, lse, q, q.clone(), q.clone(), q.clone(), 0.125, False, ws)
