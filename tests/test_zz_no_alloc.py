"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
(plugin hosts that give a library only its input and output buffers, and
latency-critical loops where cudaMalloc/cudaFree would synchronise the
device).  Its scratch is a fixed array inside the library, so the test checks
that two calls in a row -- the second one inheriting the first one's leftover
scratch contents -- give the same gradients as fa_bwd with a caller-owned
workspace, and that an oversized problem is refused."""
import ctypes
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

GRAD_RTOL = 2e-2  # the backward bound the parity tests use


def rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_matches_workspace_backward_twice(causal):
    from exact_attention_98_gb300 import fa
    from exact_attention_98_gb300.inputs import attention_inputs

    B, H, N, d = 2, 4, 1000, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t.cuda() for t in attention_inputs(B, H, N, d, seed=11))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    ref = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    for _ in range(2):
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = fa.lib.fa_bwd_noalloc(
            *(ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, o, lse, do, *got)),
            B, H, N, d, ctypes.c_float(scale), int(causal),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == fa.FA_OK, fa.status_string(rc)
        assert fa.fa_last_device_status() == fa.FA_OK
        for g, r in zip(got, ref):
            assert rel(g, r) <= GRAD_RTOL


def test_noalloc_refuses_oversized_problem():
    from exact_attention_98_gb300 import fa

    fake = ctypes.c_void_p(0x1000)
    # 4 * 16 * 8192 rows at d = 128 need ~258 MiB of scratch, beyond the fixed array
    rc = fa.lib.fa_bwd_noalloc(*([fake] * 9), 4, 16, 8192, 128, ctypes.c_float(0.088), 0, None)
    assert rc == fa.FA_ERR_TOO_LARGE
    assert fa.status_string(rc) == "FA_ERR_TOO_LARGE"
