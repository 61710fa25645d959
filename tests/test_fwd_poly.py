"""The forward with part of its exponentials on the FMA pipe: 1, 2 or 3 of
every 8 exponentials of a row tile evaluated by the degree-3 polynomial exp2,
the rest by MUFU ("Программная эмуляция экспоненты" of "FlashAttention-3 и
FlashAttention-4"; FlashAttention-4 abstract, item 2), against the fp64
oracle with the forward's bounds.

Each share is a separate kernel instantiation, selected for later calls by
fa_set_exp2_poly_share; the tests cover ragged and one-key lengths, both head
dims, both masks (edge tiles -- the diagonal and a ragged last key tile --
fall back to MUFU so that masked -inf scores give exact zeros), the
softmax-stress inputs and an N >= 8k problem on sampled rows.  They also check
that the setting takes effect and selects what it says: the polynomial's
rounding differs from MUFU's, so outputs at different shares are never
bit-identical (a selection that evaluated the same set of exponentials for
two shares would fail this)."""
import math

import pytest
import torch

from parity import compare_fwd

pytestmark = pytest.mark.gpu

SHARES = (1, 2, 3)


@pytest.fixture
def share():
    from exact_attention_98_gb300 import fa

    before = fa.fa_get_exp2_poly_share()

    def set_share(n):
        fa.fa_set_exp2_poly_share(n)
        assert fa.fa_get_exp2_poly_share() == n

    yield set_share
    fa.fa_set_exp2_poly_share(before)


@pytest.mark.parametrize("poly", SHARES)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 383, 640])
def test_poly_small_and_ragged(share, poly, d, causal, N):
    share(poly)
    compare_fwd(1, 2, N, d, causal, seed=N + poly)


@pytest.mark.parametrize("poly", SHARES)
@pytest.mark.parametrize("causal", [False, True])
def test_poly_stress(share, poly, causal):
    share(poly)
    compare_fwd(1, 4, 1024, 128, causal, seed=7, stress=True, full_heads=1, rows_per_head=256)


@pytest.mark.parametrize("poly", SHARES)
def test_poly_long(share, poly):
    """B1 H4 N8192 d128 causal: head 0 in full, 256 sampled rows elsewhere."""
    share(poly)
    compare_fwd(1, 4, 8192, 128, True, seed=3, full_heads=1, rows_per_head=256)


@pytest.mark.parametrize("poly", SHARES)
def test_poly_b2h16n4096(share, poly):
    """The B2 H16 N4096 d128 non-causal forward (with its last-round split)."""
    share(poly)
    compare_fwd(2, 16, 4096, 128, False, full_heads=1, rows_per_head=128)


def test_share_takes_effect(share):
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    q, k, v, _ = (None if t is None else t.cuda()
                  for t in attention_inputs(1, 2, 640, 128, seed=1, with_dout=False))
    outs = {}
    for n in (0, 1, 2, 3):
        share(n)
        outs[n] = fa.forward(q, k, v, causal=False, scale=1 / math.sqrt(128))
    assert fa.fa_last_device_status() == fa.FA_OK
    # every share gives different bits: n of every 8 exponentials on the
    # polynomial, so no two shares evaluate the same set
    for a in (0, 1, 2, 3):
        for b in (0, 1, 2, 3):
            if a < b:
                assert not torch.equal(outs[a][0], outs[b][0]), (a, b)
    # the same share twice gives the same bits
    share(2)
    again = fa.forward(q, k, v, causal=False, scale=1 / math.sqrt(128))
    assert torch.equal(again[0], outs[2][0]) and torch.equal(again[1], outs[2][1])
