"""Pins of the FP8 reference steps (oracle/fp8.py) against things other than
itself: PyTorch's own e4m3 conversion, orthogonality of the rotation, the
exact-attention oracle, and hand-worked values."""
import math

import numpy as np
import pytest
import torch

import oracle.attn_np as exact
import oracle.fp8 as F


def test_round_e4m3_matches_torch_float8():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-4, 2.6, 20000),
                        np.arange(-470, 470, 0.25), [0.0, 2.0 ** -9, 3 * 2.0 ** -10, 2.0 ** -10]])
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(F.round_e4m3(x), ref)


def test_round_e4m3_by_hand():
    # 3 mantissa bits: 1.0625 lies between 1 and 1.125, nearer 1; 232 is the
    # tie between 224 and 240 (even mantissa: 224); 500 saturates to 448
    assert list(F.round_e4m3([1.0625, 1.07, 232.0, 500.0, -500.0])) == [1.0, 1.125, 224.0, 448.0, -448.0]


def test_rot_signs_by_hand():
    # (0x9E3779B1 * (i + 1)) mod 2^32 for i = 0, 1, 2: 0x9E3779B1 (bit 31 set),
    # 0x3C6EF362 (clear), 0xDAA66D13 (set)
    assert list(F.rot_signs(3)) == [-1.0, 1.0, -1.0]


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_is_orthogonal_and_keeps_scores(d):
    r = F.rotation(d)
    assert np.abs(r @ r.T - np.eye(d)).max() < 1e-12
    rng = np.random.default_rng(d)
    q, k = rng.standard_normal((16, d)), rng.standard_normal((16, d))
    assert np.abs((q @ r) @ (k @ r).T - q @ k.T).max() < 1e-10


def test_hadamard_rows_are_orthogonal_and_plus_minus_one():
    h = F.hadamard(128)
    assert set(np.unique(h)) == {-1.0, 1.0}
    assert np.array_equal(h @ h.T, 128 * np.eye(128))


def test_quantise_row_scales_by_hand():
    """One scale per row (axis=1) against one for the whole array: row 0 has
    amax 1 (scale 448), row 1 amax 8 (scale 56)."""
    x = np.array([[1.0, 0.5, 0.25, 0.0], [8.0, 4.0, 2.0, 1.0]])
    q8, desc = F.quantise(x, axis=1)
    assert np.array_equal(q8, [[448, 224, 112, 0], [448, 224, 112, 56]])
    assert np.array_equal(desc, [[1 / 448], [1 / 56]])
    q8, desc = F.quantise(x)
    assert np.array_equal(q8, [[56, 28, 14, 0], [448, 224, 112, 56]]) and desc == 1 / 56


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_by_hand(causal):
    """A 2 x 4 case worked by hand, without rotation, scale = ln 2 (so that
    exp(scale s) = 2^s).  Q rows have amax 1 and 3: row scales 448 and 448/3
    put both rows exactly on the e4m3 grid, while one scale for all of Q
    (448/3) would round row 0 (1 -> 144/(448/3), 0.5 -> 72/(448/3)) and change
    its scores.  K (amax 2) and V (amax 4) are exact with their scales.
      scores / ln 2 = Q K^T = [[2, 1], [3, -3]]
      row 0: p = [1, 1/2], l = 3/2, 64 p = [64, 32] (exact in e4m3)
             O = (v0 + v1 / 2) / (3/2) = [2, 2, 3, 17/6], LSE = 2 ln 2 + ln 3/2
             (causal: key 0 only, O = v0, LSE = 2 ln 2)
      row 1: p = [1, 1/64], l = 65/64, 64 p = [64, 1] (exact)
             O = (64 v0 + v1) / 65 = [68, 130, 257, 256.5] / 65,
             LSE = 3 ln 2 + ln 65/64"""
    q = np.array([[1.0, 0.5, 0.0, 0.0], [0.0, 0.0, 3.0, -1.5]])
    k = np.array([[2.0, 0.0, 1.0, 0.0], [0.0, 2.0, 0.0, 2.0]])
    v = np.array([[1.0, 2.0, 4.0, 4.0], [4.0, 2.0, 1.0, 0.5]])
    ln2 = math.log(2.0)
    o, lse = F.forward_head(q, k, v, ln2, causal, rotate=False)
    o0 = [1.0, 2.0, 4.0, 4.0] if causal else [2.0, 2.0, 3.0, 17.0 / 6.0]
    l0 = 2 * ln2 + (0.0 if causal else math.log(1.5))
    assert np.allclose(o, [o0, np.array([68.0, 130.0, 257.0, 256.5]) / 65.0], rtol=0, atol=1e-12)
    assert np.allclose(lse, [l0, 3 * ln2 + math.log(65.0 / 64.0)], rtol=0, atol=1e-12)


def test_quantise_is_lossless_on_the_e4m3_grid():
    grid = F.round_e4m3(np.linspace(-448, 448, 301))
    q8, desc = F.quantise(grid)
    assert desc == 1.0 and np.array_equal(q8, grid)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_close_to_exact_attention(causal):
    rng = np.random.default_rng(1)
    N, d = 256, 128
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    o_ref, lse_ref, _ = exact.forward(q, k, v, 1 / math.sqrt(d), causal)
    o, lse = F.forward_head(q, k, v, 1 / math.sqrt(d), causal)
    assert np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref) < 0.08
    assert np.abs(lse - lse_ref).max() < 0.1


def test_rotation_reduces_the_error_with_outlier_channels():
    """The pages' claim (a smaller FP8 error with incoherent processing) on
    inputs whose error the plain FP8 path concentrates: 4 of 128 channels of
    Q and K ten times larger."""
    rng = np.random.default_rng(2)
    N, d = 256, 128
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    ch = rng.permutation(d)[:4]
    q[:, ch] *= 10
    k[:, ch] *= 10
    scale = 1 / math.sqrt(d) / 10
    o_ref, _, _ = exact.forward(q, k, v, scale, False)
    err = lambda rot: np.linalg.norm(F.forward_head(q, k, v, scale, False, rot)[0] - o_ref)
    assert err(True) * 1.5 < err(False)
