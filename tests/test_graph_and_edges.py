"""Robustness of the public calls: CUDA-graph capture and replay of a
training step, and edge shapes of the split and FP8 paths."""
import math

import numpy as np
import pytest
import torch

from parity import compare_fwd, run_fwd

pytestmark = pytest.mark.gpu


def test_cuda_graph_capture_of_a_step():
    """fwd + bwd captured once and replayed: the replay equals an eager step
    (O, LSE, dK, dV bit for bit; dQ up to the order of its fp32 additions).
    B2 H16 N4096 non-causal also takes the forward's last-round split, in
    the caller's workspace, inside the graph."""
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N, d = 2, 16, 4096, 128
    q, k, v, do = (t.cuda() for t in attention_inputs(B, H, N, d, seed=21))
    scale = 1 / math.sqrt(d)
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = fa.workspace_for(q)
    wsf = fa.fwd_workspace_for(q, False)
    assert wsf is not None  # 512 items on 152 SMs: the last round is split
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # eager reference
        fa.fa_fwd(q, k, v, o, lse, scale, False, wsf)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale, False, ws)
    s.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fa.fa_fwd(q, k, v, o, lse, scale, False, wsf)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale, False, ws)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for got, want, name in zip((o, lse, dk, dv), (ref[0], ref[1], ref[3], ref[4]), ("o", "lse", "dk", "dv")):
        assert torch.equal(got, want), name
    rel = (dq.float() - ref[2].float()).norm() / ref[2].float().norm()
    assert rel < 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_tail_split_with_ragged_keys(causal):
    """B2 H16 N4000: 512 work items, the last round's split in two key
    ranges, the last key tile ragged; head 1 full, sampled rows elsewhere."""
    compare_fwd(2, 16, 4000, 128, causal, full_heads=1, rows_per_head=128)


def test_forward_splits_only_in_a_given_workspace():
    """B2 H16 N4096 non-causal: 512 work items on the SMs leave a partial
    last round.  Without a workspace fa_fwd launches one kernel and
    allocates nothing; with one it splits that round (forward + merge).  Both
    meet the forward's bounds on head 0 and stay within rounding of each
    other."""
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs
    import oracle
    from parity import check_lse, check_o, to64

    B, H, N, d = 2, 16, 4096, 128
    q, k, v, _ = attention_inputs(B, H, N, d, seed=4, with_dout=False)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1 / math.sqrt(d)
    outs = []
    for ws in (None, fa.fwd_workspace_for(qd, False)):
        o, lse = torch.empty_like(qd), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free0, n0 = torch.cuda.mem_get_info()[0], fa.fa_launch_count()
        fa.fa_fwd(qd, kd, vd, o, lse, scale, False, ws)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert fa.fa_launch_count() - n0 == (1 if ws is None else 2)
        outs.append((to64(o), to64(lse)))
    assert fa.fa_last_device_status() == fa.FA_OK
    o_ref, l_ref = oracle.fwd_head(*(t[0, 0].double().numpy() for t in (q, k, v)), scale, False)
    for o, lse in outs:
        check_o(o[0, 0], o_ref, "head 0")
        check_lse(lse[0, 0], l_ref, "head 0")
    assert np.abs(outs[0][0] - outs[1][0]).max() <= 1e-2
    assert np.abs(outs[0][1] - outs[1][1]).max() <= 1e-4


@pytest.mark.parametrize("N", [1, 5, 129])
def test_fp8_degenerate_lengths(N):
    """FP8 forward on one key, a few keys and one key past a tile: V^T's
    padded pitch and zero keys, within the FP8 bounds of the exact oracle."""
    import oracle
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, d = 1, 2, 128
    q, k, v, _ = attention_inputs(B, H, N, d, seed=N, with_dout=False)
    o, lse = fa.forward_fp8(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert fa.fa_last_device_status() == fa.FA_OK
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    for h in range(H):
        q64, k64, v64 = (t[0, h].double().numpy() for t in (q, k, v))
        o_ref, l_ref = oracle.fwd_head(q64, k64, v64, 1 / math.sqrt(d), True)
        assert np.linalg.norm(o[0, h] - o_ref) / np.linalg.norm(o_ref) <= 0.08
        assert np.abs(lse[0, h] - l_ref).max() <= 0.25


def test_splitkv_single_key_tile():
    """num_splits = 1 on a one-tile problem runs the plain forward."""
    compare_fwd(1, 2, 100, 64, False, num_splits=1)


@pytest.mark.parametrize("d", [64, 128])
def test_output_only_16_byte_aligned(d):
    """The API asks 16-byte alignment of O; the forward writes O rows with
    32-byte stores when O allows them and with 16-byte stores otherwise.
    An O that starts 16 bytes past a 32-byte boundary gets bit-identical
    results to an aligned one."""
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N = 1, 2, 777
    q, k, v, _ = (None if t is None else t.cuda()
                  for t in attention_inputs(B, H, N, d, seed=5, with_dout=False))
    scale = 1 / math.sqrt(d)
    for causal in (False, True):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        assert o.data_ptr() % 32 == 0
        fa.fa_fwd(q, k, v, o, lse, scale, causal)
        buf = torch.empty(q.numel() + 8, dtype=q.dtype, device="cuda")
        o16 = buf[8:].view_as(q)
        assert o16.data_ptr() % 32 == 16
        lse16 = torch.empty_like(lse)
        fa.fa_fwd(q, k, v, o16, lse16, scale, causal)
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.equal(o16, o) and torch.equal(lse16, lse)


@pytest.mark.parametrize("d", [64, 128])
def test_gradients_only_16_byte_aligned(d):
    """The same for the backward's dK and dV rows: outputs 16 bytes past a
    32-byte boundary get the bits of aligned ones (dQ, summed with fp32
    atomics in a varying order, is compared within the gradient bound)."""
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N = 1, 2, 777
    q, k, v, do = (t.cuda() for t in attention_inputs(B, H, N, d, seed=6))
    scale = 1 / math.sqrt(d)
    ws = fa.workspace_for(q)
    for causal in (False, True):
        o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
        ref = [torch.empty_like(q) for _ in range(3)]
        fa.fa_bwd(q, k, v, o, lse, do, *ref, scale, causal, ws)
        bufs = [torch.empty(q.numel() + 8, dtype=q.dtype, device="cuda") for _ in range(3)]
        got = [b[8:].view_as(q) for b in bufs]
        assert all(g.data_ptr() % 32 == 16 for g in got)
        fa.fa_bwd(q, k, v, o, lse, do, *got, scale, causal, ws)
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
        rel = (got[0].float() - ref[0].float()).norm() / ref[0].float().norm()
        assert rel < 1e-3, float(rel)


def test_launch_counter_per_call():
    """fa_launch_count advances by the number of kernels each call launches
    (the figure the benchmark reports as its launch count)."""
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N, d = 1, 2, 384, 128
    q, k, v, do = (t.cuda() for t in attention_inputs(B, H, N, d, seed=5))
    scale = 1 / math.sqrt(d)
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))

    def count(call):
        before = fa.fa_launch_count()
        call()
        torch.cuda.synchronize()
        return fa.fa_launch_count() - before

    # 2 query blocks of 256 rows x 2 heads: fewer than the SMs, never split
    assert count(lambda: fa.fa_fwd(q, k, v, o, lse, scale, False)) == 1
    assert fa.fa_fwd_workspace_bytes(B, H, N, d, False) == 0
    ws = fa.workspace_for(q)
    assert count(lambda: fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale, False, ws)) == 3
    wsd = fa.workspace_for(q, deterministic=True)
    assert count(lambda: fa.fa_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv, scale, False,
                                                 wsd)) == 3
    ws2 = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(B, H, N, d, 2), dtype=torch.uint8,
                      device="cuda")
    assert count(lambda: fa.fa_fwd_splitkv(q, k, v, o, lse, scale, False, 2, ws2)) == 2
    ws8 = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    assert count(lambda: fa.fa_fwd_fp8(q, k, v, o, lse, scale, False, True, ws8)) == 3
    assert count(lambda: fa.fa_fwd_2cta(q, k, v, o, lse, scale, False)) == 1
    assert count(lambda: fa.fa_bwd_2cta(q, k, v, o, lse, do, dq, dk, dv, scale, False, ws)) == 3
    assert fa.fa_last_device_status() == fa.FA_OK
