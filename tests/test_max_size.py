"""The largest shapes: every tensor holds more than 2^31 elements, so any
32-bit element index in a kernel or its launch arithmetic would wrap.

B1 H136 N131072 d128 causal (2.28e9 elements, 4.6 GB per bf16 tensor; about
60 GB on the device in all), inputs drawn head by head on the device.  The
first and the last head (the largest offsets) are compared with the fp64
oracle on sampled rows: O and LSE element by element, dQ rows by relative
Frobenius error; dK and dV of those heads through the properties that hold
at any size (dK rows sum to zero, dV rows sum to the dO rows).  The 2-CTA
backward must stay within rounding of the backward on those heads, the
deterministic backward must equal it on dK and dV and stay within rounding
on dQ, the 2-CTA
forward must equal the forward bit for bit, and the FP8 forward must stay
within its bounds."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_98_gb300.inputs import device_head_inputs, sampled_rows
from parity import check_grad, check_lse, check_o, rel_fro, to64

pytestmark = pytest.mark.gpu

B, H, N, D = 1, 136, 131072, 128
SEED = 31


@pytest.fixture(scope="module")
def big():
    assert B * H * N * D > 2 ** 31
    dev = torch.device("cuda")
    q, k, v, do = (torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev) for _ in range(4))
    for h in range(H):
        for dst, src in zip((q, k, v, do), device_head_inputs(N, D, SEED, h, dev)):
            dst[0, h].copy_(src)
    yield q, k, v, do
    del q, k, v, do
    torch.cuda.empty_cache()


def head64(t, h):
    return t[0, h].to("cpu", torch.float64).numpy()


def test_forward_backward(big):
    from exact_attention_98_gb300 import fa

    q, k, v, do = big
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    assert fa.fa_last_device_status() == fa.FA_OK
    for h in (0, H - 1):
        qh, kh, vh, doh = (head64(t, h) for t in (q, k, v, do))
        rows = sampled_rows(N, 64, 0, h, H)
        what = f"B{B} H{H} N{N} causal head {h}"
        o_ref, l_ref = oracle.fwd_head(qh, kh, vh, scale, True, rows=rows)
        check_o(to64(o[0, h])[rows], o_ref, what)
        check_lse(to64(lse[0, h])[rows], l_ref, what)
        g = oracle.bwd_head(qh, kh, vh, doh, scale, True, qrows=rows, krows=[], o_bf16=True)
        check_grad(to64(dq[0, h])[rows], g[0], what + " dQ")
        dkh, dvh = head64(dk, h), head64(dv, h)
        assert np.abs(dkh.sum(axis=0)).max() <= 2e-2 * np.abs(dkh).sum(axis=0).max(), what
        dv_err = np.abs(dvh.sum(axis=0) - doh.sum(axis=0)).max()
        assert dv_err <= 2e-2 * np.abs(doh).sum(axis=0).max(), what
    # the 2-CTA backward on the same inputs: within rounding of fa_bwd on the
    # first and last heads (dK, dV in full; dQ on the sampled rows, which the
    # oracle bounds as above)
    dq2, dk2, dv2 = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, two_cta=True)
    assert fa.fa_last_device_status() == fa.FA_OK
    for h in (0, H - 1):
        rows = sampled_rows(N, 64, 0, h, H)
        for a, b in ((dk, dk2), (dv, dv2)):
            assert rel_fro(head64(b, h), head64(a, h)) <= 2e-3, h
        assert rel_fro(to64(dq2[0, h])[rows], to64(dq[0, h])[rows]) <= 2e-3, h
    del dq2, dk2, dv2
    # the deterministic backward (d = 128: dK/dV pass and query-stationary dQ
    # kernel, 139264 CTAs each): dK and dV equal fa_bwd's bit for bit, dQ
    # within rounding on the sampled rows
    dq3, dk3, dv3 = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, deterministic=True)
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.equal(dk3, dk) and torch.equal(dv3, dv)
    for h in (0, H - 1):
        rows = sampled_rows(N, 64, 0, h, H)
        assert rel_fro(to64(dq3[0, h])[rows], to64(dq[0, h])[rows]) <= 2e-3, h
    del dq, dk, dv, dq3, dk3, dv3
    # the 2-CTA forward: the same products and per-row arithmetic
    o2, lse2 = fa.forward(q, k, v, causal=True, scale=scale, two_cta=True)
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.equal(o2, o) and torch.equal(lse2, lse)
    del o2, lse2, o, lse
    torch.cuda.empty_cache()


def test_fp8_forward(big):
    from exact_attention_98_gb300 import fa

    q, k, v, _ = big
    scale = 1.0 / math.sqrt(D)
    o8, lse8 = fa.forward_fp8(q, k, v, causal=True, scale=scale)
    assert fa.fa_last_device_status() == fa.FA_OK
    for h in (0, H - 1):
        qh, kh, vh = (head64(t, h) for t in (q, k, v))
        rows = sampled_rows(N, 64, 0, h, H)
        o_ref, l_ref = oracle.fwd_head(qh, kh, vh, scale, True, rows=rows)
        assert rel_fro(to64(o8[0, h])[rows], o_ref) <= 0.08
        assert np.abs(to64(lse8[0, h])[rows] - l_ref).max() <= 0.25
    del o8, lse8
    torch.cuda.empty_cache()
