"""Pins for the fp64 oracle, checked against facts that do not come from it.

Each test names the mistake it is there to catch.  The pages print no worked
example, so the pins are closed forms of special cases, invariants of the
definition, central finite differences of the forward, and a library routine
(PyTorch's fp64 CPU scaled-dot-product attention) on small inputs.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import attn_np

RNG = np.random.default_rng(1234)


def rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


def n_allowed(i, N, causal):
    return i + 1 if causal else N


# --- closed forms of special cases ----------------------------------------


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_allowed_values(causal):
    """Q = 0 makes every score 0: O_i is the plain mean of the allowed V rows
    and LSE_i = ln(#allowed).  Catches a causal off-by-one (j < i vs j <= i),
    a wrong log base, and a missing normalisation."""
    N, d = 23, 5
    q = np.zeros((N, d))
    k, v = rand(N, d), rand(N, d)
    o, lse = oracle.fwd_head(q, k, v, 0.37, causal)
    for i in range(N):
        n = n_allowed(i, N, causal)
        np.testing.assert_allclose(o[i], v[:n].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert abs(lse[i] - math.log(n)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_values(causal):
    """All keys equal to u: uniform P, O_i = mean of allowed V, and
    LSE_i = scale*q_i.u + ln(#allowed).  Catches a dropped or doubled scale in
    the scores or in LSE."""
    N, d, scale = 17, 6, 0.81
    u = rand(d)
    k = np.tile(u, (N, 1))
    q, v = rand(N, d), rand(N, d)
    o, lse = oracle.fwd_head(q, k, v, scale, causal)
    for i in range(N):
        n = n_allowed(i, N, causal)
        np.testing.assert_allclose(o[i], v[:n].mean(axis=0), rtol=1e-12, atol=1e-13)
        assert abs(lse[i] - (scale * float(q[i] @ u) + math.log(n))) < 1e-12


def test_causal_row_zero_is_value_row_zero():
    """Under the causal mask query 0 sees only key 0: O_0 = V_0 and
    LSE_0 = scale*q_0.k_0."""
    N, d, scale = 9, 4, 0.5
    q, k, v = rand(N, d), rand(N, d), rand(N, d)
    o, lse = oracle.fwd_head(q, k, v, scale, True)
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=1e-15)
    assert abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-14


def test_single_key():
    """N = 1: O = V and LSE = scale*q.k, masked or not."""
    q, k, v = rand(1, 7), rand(1, 7), rand(1, 7)
    for causal in (False, True):
        o, lse = oracle.fwd_head(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, v, atol=1e-15)
        assert abs(lse[0] - 0.3 * float(q[0] @ k[0])) < 1e-14


def test_two_keys_logistic_closed_form():
    """Two keys: P_i0 = 1/(1 + exp(s_i1 - s_i0)) (the logistic function),
    O_i = P_i0 v_0 + P_i1 v_1, LSE_i = s_i0 + ln(1 + exp(s_i1 - s_i0)).  With
    q, k chosen so that the scores are asymmetric, this catches a transposed
    Q K^T, a missing scale and a swapped value row."""
    scale = 0.7
    q = np.array([[1.0, 2.0], [-0.5, 0.25]])
    k = np.array([[0.3, -1.0], [2.0, 0.5]])
    v = np.array([[1.0, -3.0], [4.0, 0.5]])
    o, lse = oracle.fwd_head(q, k, v, scale, False)
    for i in range(2):
        s0 = scale * (q[i, 0] * k[0, 0] + q[i, 1] * k[0, 1])
        s1 = scale * (q[i, 0] * k[1, 0] + q[i, 1] * k[1, 1])
        p0 = 1.0 / (1.0 + math.exp(s1 - s0))
        p1 = 1.0 - p0
        np.testing.assert_allclose(o[i], p0 * v[0] + p1 * v[1], rtol=1e-14)
        assert abs(lse[i] - (s0 + math.log1p(math.exp(s1 - s0)))) < 1e-14
    # causal: row 1 is the same two-key softmax, row 0 sees key 0 only
    o, lse = oracle.fwd_head(q, k, v, scale, True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)


# --- invariants -----------------------------------------------------------


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    """V = all ones gives O_i = sum_j P_ij, which must be exactly 1."""
    N, d = 31, 8
    q, k = 2.0 * rand(N, d), 2.0 * rand(N, d)
    o, _ = oracle.fwd_head(q, k, np.ones((N, d)), 1.0, causal)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """Adding u to every key shifts row i's scores by the constant
    scale*q_i.u: O is unchanged and LSE_i moves by exactly that constant.
    Catches scores built from anything but q_i.k_j."""
    N, d, scale = 19, 6, 0.45
    q, k, v = rand(N, d), rand(N, d), rand(N, d)
    u = rand(d)
    o1, l1 = oracle.fwd_head(q, k, v, scale, causal)
    o2, l2 = oracle.fwd_head(q, k + u, v, scale, causal)
    np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, scale * (q @ u), rtol=1e-11, atol=1e-12)


def test_key_permutation_equivariance_noncausal():
    """Without a mask, reordering the (key, value) pairs leaves O and LSE
    unchanged; reordering the queries reorders O and LSE the same way."""
    N, d = 13, 5
    q, k, v = rand(N, d), rand(N, d), rand(N, d)
    perm = RNG.permutation(N)
    o1, l1 = oracle.fwd_head(q, k, v, 0.6, False)
    o2, l2 = oracle.fwd_head(q, k[perm], v[perm], 0.6, False)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=1e-13)
    o3, l3 = oracle.fwd_head(q[perm], k, v, 0.6, False)
    np.testing.assert_allclose(o3, o1[perm], rtol=1e-13)
    np.testing.assert_allclose(l3, l1[perm], rtol=1e-13)


def test_row_subset_matches_full():
    """Computing a subset of rows gives exactly those rows of the full result
    (the causal mask follows the row's position, not its index in the subset)."""
    N, d = 40, 8
    q, k, v, do = rand(N, d), rand(N, d), rand(N, d), rand(N, d)
    rows = [0, 3, 17, 39]
    for causal in (False, True):
        o, lse = oracle.fwd_head(q, k, v, 0.35, causal)
        os_, ls = oracle.fwd_head(q, k, v, 0.35, causal, rows=rows)
        np.testing.assert_array_equal(os_, o[rows])
        np.testing.assert_array_equal(ls, lse[rows])
        dq, dk, dv = oracle.bwd_head(q, k, v, do, 0.35, causal)
        dqs, dks, dvs = oracle.bwd_head(q, k, v, do, 0.35, causal, qrows=rows, krows=rows[::-1])
        np.testing.assert_allclose(dqs, dq[rows], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(dks, dk[rows[::-1]], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(dvs, dv[rows[::-1]], rtol=1e-13, atol=1e-15)


# --- backward ---------------------------------------------------------------


def _loss(q, k, v, do, scale, causal):
    o, _ = oracle.fwd_head(q, k, v, scale, causal)
    return float((o * do).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 3), (5, 4), (8, 8)])
def test_backward_matches_central_finite_differences(causal, N, d):
    """dQ, dK, dV equal the central differences of L = sum(O*dO) computed with
    the (separately pinned) forward alone; h = 1e-6 leaves ~1e-9 relative
    error.  Catches a sign, a missing D term, a missing scale, or dQ/dK swapped."""
    rng = np.random.default_rng(N * 100 + d + (7 if causal else 0))
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    scale = 0.9
    dq, dk, dv = oracle.bwd_head(q, k, v, do, scale, causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, scale, causal)
                       - _loss(args_m["q"], args_m["k"], args_m["v"], do, scale, causal)) / (2 * h)
        err = np.linalg.norm(g - fd) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-7, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    """sum_j dK_j = 0 (each row of dS sums to 0), sum_j dV_j = sum_i dO_i
    (each row of P sums to 1)."""
    N, d = 29, 7
    q, k, v, do = rand(N, d), rand(N, d), rand(N, d), rand(N, d)
    dq, dk, dv = oracle.bwd_head(q, k, v, do, 0.55, causal)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_identical_keys_give_zero_dq():
    """With identical keys every score in a row moves together, so the loss
    does not depend on Q: dQ = 0."""
    N, d = 12, 5
    u = rand(d)
    k = np.tile(u, (N, 1))
    q, v, do = rand(N, d), rand(N, d), rand(N, d)
    for causal in (False, True):
        dq, _, _ = oracle.bwd_head(q, k, v, do, 0.8, causal)
        np.testing.assert_allclose(dq, 0.0, atol=1e-13)


# --- library cross-check and the NumPy restatement ---------------------------


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_fp64(causal):
    """PyTorch's CPU scaled_dot_product_attention in fp64, with autograd, is a
    library implementation of the same definition: forward and all three
    gradients agree to ~1e-12."""
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 3, 21, 16
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator().manual_seed(5)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(4))
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    ot = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    (ot * do).sum().backward()
    o, _ = oracle.fwd(q.numpy(), k.numpy(), v.numpy(), scale, causal)
    dq, dk, dv = oracle.bwd(q.numpy(), k.numpy(), v.numpy(), do.numpy(), scale, causal)
    np.testing.assert_allclose(o, ot.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_c_oracle_matches_numpy_restatement(causal):
    N, d = 33, 9
    q, k, v, do = rand(N, d), rand(N, d), rand(N, d), rand(N, d)
    o, lse = oracle.fwd_head(q, k, v, 0.4, causal)
    o2, lse2, _ = attn_np.forward(q, k, v, 0.4, causal)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=1e-13, atol=1e-13)
    g1 = oracle.bwd_head(q, k, v, do, 0.4, causal)
    g2 = attn_np.backward(q, k, v, do, 0.4, causal)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_rejects_bad_rows():
    q = rand(4, 2)
    with pytest.raises(ValueError):
        oracle.fwd_head(q, q, q, 1.0, False, rows=[5])
    with pytest.raises(RuntimeError):
        oracle.bwd_head(q, q, q, q, 1.0, False, qrows=[-1])


def test_oracle_regression_fixture():
    """The oracle still reproduces the record that tests/golden/make_oracle_fixture.py
    wrote from it (guards against unnoticed changes to its arithmetic)."""
    import json
    import os

    from exact_attention_98_gb300.inputs import attention_inputs

    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny.json")
    rec = json.load(open(path))
    B, H, N, d = rec["shape"]
    q, k, v, do = (t.double().numpy()[0, 0] for t in attention_inputs(B, H, N, d, seed=rec["seed"]))
    for name, causal in (("full", False), ("causal", True)):
        want = rec["cases"][name]
        o, lse = oracle.fwd_head(q, k, v, rec["scale"], causal)
        dq, dk, dv = oracle.bwd_head(q, k, v, do, rec["scale"], causal)
        for got, key in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
            np.testing.assert_allclose(got, np.array(want[key]), rtol=1e-12, atol=1e-14)


# --- the backward's O input in bf16 -------------------------------------------


def test_round_bf16_against_torch_and_by_hand():
    """The oracle's bf16 rounding: exact values stay, halfway cases go to the
    even neighbour, and random doubles agree with PyTorch's bf16 conversion of
    their fp32 value where that fp32 value is itself exact."""
    torch = pytest.importorskip("torch")
    r = oracle.round_bf16
    assert r(1.0) == 1.0 and r(-0.15625) == -0.15625 and r(0.0) == 0.0
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to even -> 1
    assert r(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even -> 1 + 2^-6
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7
    xs = np.random.default_rng(3).standard_normal(2000).astype(np.float32).astype(np.float64)
    want = torch.from_numpy(xs.astype(np.float32)).to(torch.bfloat16).double().numpy()
    got = np.array([r(x) for x in xs])
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(attn_np.round_bf16(xs), want)


def test_backward_with_bf16_o_matches_numpy_and_differs_only_through_D():
    """o_bf16 changes only D: against the NumPy restatement with the same
    option, and exactly equal to the plain backward when O is already a bf16
    value (V rows bf16-exact and P one-hot: identical keys and N = 1)."""
    N, d = 24, 8
    q, k, v, do = rand(N, d), rand(N, d), rand(N, d), rand(N, d)
    for causal in (False, True):
        g1 = oracle.bwd_head(q, k, v, do, 0.5, causal, o_bf16=True)
        g2 = attn_np.backward(q, k, v, do, 0.5, causal, o_bf16=True)
        for a, b in zip(g1, g2):
            np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)
        g0 = oracle.bwd_head(q, k, v, do, 0.5, causal)
        assert not np.allclose(g1[0], g0[0], rtol=1e-14, atol=0)
        np.testing.assert_array_equal(g1[2], g0[2])  # dV does not involve D
    vb = attn_np.round_bf16(rand(1, d))
    q1, k1, do1 = rand(1, d), rand(1, d), rand(1, d)
    np.testing.assert_array_equal(oracle.bwd_head(q1, k1, vb, do1, 0.5, False)[0],
                                  oracle.bwd_head(q1, k1, vb, do1, 0.5, False, o_bf16=True)[0])
