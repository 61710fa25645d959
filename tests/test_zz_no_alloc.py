"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
(plugin hosts that give a library only its input and output buffers, and
latency-critical loops where cudaMalloc/cudaFree would synchronise the
device).  Its scratch is a fixed array inside the library, shared by every
call, so the tests check that

  * a call that follows a larger call with the other mask (which leaves more
    of the array written) gives the gradients of fa_bwd with a caller-owned
    workspace: dK and dV bit for bit, dQ up to the order of its fp32 atomic
    additions;
  * a second call in a row does the same and changes the device's free
    memory by nothing (no allocation);
  * the array is reserved only by a process that calls fa_bwd_noalloc
    (fa_fwd and fa_bwd in a fresh process leave it unloaded);
  * an oversized problem is refused.

This file is collected last, so a run that stops at its first failure has run
every other test before it."""
import ctypes
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def call_noalloc(fa, q, k, v, o, lse, do, grads, scale, causal):
    B, H, N, d = q.shape
    return fa.lib.fa_bwd_noalloc(
        *(ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, o, lse, do, *grads)),
        B, H, N, d, ctypes.c_float(scale), int(causal),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def check_dq(got, ref):
    """dQ is accumulated with fp32 atomics in an order that varies from call
    to call, then rounded to bf16.  The order changes the fp32 sum by a few
    fp32 ulps of its summands, which are of the size of the tensor's largest
    elements; rounded to bf16 that moves an element by one bf16 ulp where the
    sums straddle a rounding boundary, or, where cancellation leaves an
    element much smaller than its summands, by about the fp32 noise itself.
    So: every element within one bf16 ulp of fa_bwd's or within 1e-5 of the
    largest |dQ|, few elements different, and a relative Frobenius error of
    at most 1e-3 (one flipped bf16 element is 2^-8 relative)."""
    g = got.cpu().double().numpy()
    r = ref.cpu().double().numpy()
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 1e-30))) - 7)
    diff = np.abs(g - r)
    floor = 1e-5 * np.abs(r).max()
    assert (diff <= np.maximum(ulp * 1.0001, floor)).all(), float(diff.max())
    assert (diff > 0).mean() <= 1e-2, float((diff > 0).mean())
    rel = np.linalg.norm(g - r) / np.linalg.norm(r)
    assert rel <= 1e-3, rel


@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_matches_workspace_backward(causal):
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    # An earlier, larger call with the other mask leaves its D and dQ
    # accumulator in the shared array.
    Bb, Hb, Nb, d = 2, 8, 1500, 128
    qb, kb, vb, dob = (t.cuda() for t in attention_inputs(Bb, Hb, Nb, d, seed=12))
    scale = 1.0 / math.sqrt(d)
    ob, lseb = fa.forward(qb, kb, vb, causal=not causal, scale=scale)
    big = [torch.empty_like(qb) for _ in range(3)]
    assert call_noalloc(fa, qb, kb, vb, ob, lseb, dob, big, scale, not causal) == fa.FA_OK

    B, H, N = 2, 4, 1000
    q, k, v, do = (t.cuda() for t in attention_inputs(B, H, N, d, seed=11))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    ref = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    outs = [[torch.full_like(q, float("nan")) for _ in range(3)] for _ in range(2)]
    torch.cuda.synchronize()
    # free device memory around the two calls (nothing else runs in between:
    # the comparisons, which may make torch allocate, come afterwards)
    free = [torch.cuda.mem_get_info()[0]]
    for got in outs:
        rc = call_noalloc(fa, q, k, v, o, lse, do, got, scale, causal)
        assert rc == fa.FA_OK, fa.status_string(rc)
        assert fa.fa_last_device_status() == fa.FA_OK
        free.append(torch.cuda.mem_get_info()[0])
    # neither call (the first after the larger call, the second in a row)
    # allocated anything
    assert free[2] == free[1] == free[0]
    for got in outs:
        check_dq(got[0], ref[0])
        assert torch.equal(got[1].cpu(), ref[1].cpu()), "dK"
        assert torch.equal(got[2].cpu(), ref[2].cpu()), "dV"


PROBE = r"""
import math, sys, torch
sys.path.insert(0, sys.argv[1])
from exact_attention_98_gb300 import fa
from exact_attention_98_gb300.inputs import attention_inputs
q, k, v, do = (t.cuda() for t in attention_inputs(1, 2, 256, 64, seed=3))
o, lse = torch.empty_like(q), torch.empty((1, 2, 256), dtype=torch.float32, device="cuda")
g = [torch.empty_like(q) for _ in range(6)]
ws = fa.workspace_for(q)
torch.cuda.synchronize()
f0 = torch.cuda.mem_get_info()[0]
fa.fa_fwd(q, k, v, o, lse, 0.125, True)
fa.fa_bwd(q, k, v, o, lse, do, g[0], g[1], g[2], 0.125, True, ws)
torch.cuda.synchronize()
f1 = torch.cuda.mem_get_info()[0]
fa.fa_bwd_noalloc(q, k, v, o, lse, do, g[3], g[4], g[5], 0.125, True)
torch.cuda.synchronize()
f2 = torch.cuda.mem_get_info()[0]
assert fa.fa_last_device_status() == fa.FA_OK
assert all(torch.equal(g[i], g[i + 3]) for i in (1, 2))
print(f0 - f1, f1 - f2)
"""


def test_array_is_reserved_only_by_noalloc_callers():
    """In a fresh process, fa_fwd and fa_bwd leave the array unloaded; the
    first fa_bwd_noalloc call loads its module, reserving the array."""
    from exact_attention_98_gb300 import fa

    r = subprocess.run([sys.executable, "-c", PROBE, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    before, at_noalloc = (int(x) for x in r.stdout.split()[-2:])
    array = 96 << 20
    assert before < array // 2, before
    assert at_noalloc >= array, at_noalloc
    del fa


def test_noalloc_refuses_oversized_problem():
    from exact_attention_98_gb300 import fa

    fake = ctypes.c_void_p(0x1000)
    # 4 * 16 * 8192 rows at d = 128 need ~258 MiB of scratch, beyond the fixed array
    rc = fa.lib.fa_bwd_noalloc(*([fake] * 9), 4, 16, 8192, 128, ctypes.c_float(0.088), 0, None)
    assert rc == fa.FA_ERR_TOO_LARGE
    assert fa.status_string(rc) == "FA_ERR_TOO_LARGE"
    # shape errors keep their own codes
    rc = fa.lib.fa_bwd_noalloc(*([fake] * 9), 1, 1, 128, 96, ctypes.c_float(0.088), 0, None)
    assert rc == fa.FA_ERR_UNSUPPORTED
