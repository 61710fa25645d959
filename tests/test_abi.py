"""The C ABI: the library loads, exports every function include/fa.h declares,
and rejects bad arguments on the host (no GPU needed: these calls return
before any CUDA work)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_98_gb300 import build

    build.build()
    from exact_attention_98_gb300 import fa

    return fa


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared()
    for must in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_last_device_status",
                 "fa_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in declared():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    assert lib.status_string(0) == "FA_OK"
    assert lib.status_string(4) == "FA_ERR_TIMEOUT"
    assert lib.status_string(99) == "FA_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    ws = lib.fa_bwd_workspace_bytes
    B, H, N, d = 2, 16, 8192, 128
    rows = B * H * N
    up = lambda x: (x + 255) // 256 * 256
    assert ws(B, H, N, d) == up(4 * rows) + up(4 * rows * d)
    assert ws(1, 1, 1, 64) == 256 + 256
    assert ws(0, 1, 1, 64) == 0
    assert ws(1, 1, 1, 96) == 0  # unsupported head dim
    det = lib.fa_bwd_deterministic_workspace_bytes
    assert det(B, H, N, d) == up(4 * rows)  # D only: dQ accumulates in tensor memory
    assert det(1, 1, 129, 64) == up(4 * 129)
    assert det(0, 1, 1, 64) == 0


P = ctypes.c_void_p


def fwd(lib, q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, B=1, H=1, N=128, d=64,
        scale=0.125, causal=0, ws=0, ws_bytes=0):
    return lib.lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, scale, causal, P(ws),
                          ws_bytes, None)


def test_fwd_validation(lib):
    assert fwd(lib, B=-1) == lib.FA_ERR_INVALID_ARG
    assert fwd(lib, N=-5) == lib.FA_ERR_INVALID_ARG
    assert fwd(lib, d=96) == lib.FA_ERR_UNSUPPORTED
    assert fwd(lib, d=256) == lib.FA_ERR_UNSUPPORTED
    assert fwd(lib, scale=0.0) == lib.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("nan")) == lib.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("inf")) == lib.FA_ERR_INVALID_ARG
    assert fwd(lib, q=0) == lib.FA_ERR_INVALID_ARG
    assert fwd(lib, lse=0) == lib.FA_ERR_INVALID_ARG
    assert fwd(lib, k=0x1008) == lib.FA_ERR_INVALID_ARG  # not 16-byte aligned
    assert fwd(lib, lse=0x1002) == lib.FA_ERR_INVALID_ARG
    assert fwd(lib, causal=2) == lib.FA_ERR_INVALID_ARG
    # the optional workspace, when given, must be 256-byte aligned
    assert fwd(lib, ws=0x10010, ws_bytes=1 << 20) == lib.FA_ERR_WORKSPACE
    # empty problems are a no-op even with null pointers
    assert fwd(lib, q=0, k=0, v=0, o=0, lse=0, N=0) == lib.FA_OK
    assert fwd(lib, q=0, k=0, v=0, o=0, lse=0, B=0) == lib.FA_OK


def test_fwd_workspace_bytes(lib):
    """The last-round split needs scratch only where it applies: never for
    causal problems, empty or unsupported shapes, or work that fills whole
    rounds; here (no GPU, so no SM count) never at all."""
    ws = lib.fa_fwd_workspace_bytes
    assert ws(2, 16, 4096, 128, True) == 0
    assert ws(0, 16, 4096, 128, False) == 0
    assert ws(2, 16, 4096, 96, False) == 0
    assert ws(1, 1, 128, 64, False) == 0  # one work item: nothing to balance


def test_exp2_poly_share_setting(lib):
    before = lib.fa_get_exp2_poly_share()
    try:
        for n in (0, 1, 2, 3):
            lib.fa_set_exp2_poly_share(n)
            assert lib.fa_get_exp2_poly_share() == n
        for bad in (-1, 4, 8):
            assert lib.lib.fa_set_exp2_poly_share(bad) == lib.FA_ERR_INVALID_ARG
        assert lib.fa_get_exp2_poly_share() == 3
    finally:
        lib.fa_set_exp2_poly_share(before)


def test_fwd_2cta_validation(lib):
    def fwd2(d=128, N=128, causal=0, q=0x1000, scale=0.125):
        a = P(0x1000)
        return lib.lib.fa_fwd_2cta(P(q), a, a, a, a, 1, 1, N, d, scale, causal, None)

    assert fwd2(d=64) == lib.FA_ERR_UNSUPPORTED  # pairs are built for d = 128 only
    assert fwd2(N=-1) == lib.FA_ERR_INVALID_ARG
    assert fwd2(causal=3) == lib.FA_ERR_INVALID_ARG
    assert fwd2(q=0) == lib.FA_ERR_INVALID_ARG
    assert fwd2(scale=-1.0) == lib.FA_ERR_INVALID_ARG
    assert fwd2(q=0, N=0) == lib.FA_OK


def bwd(lib, ws=0x10000, ws_bytes=1 << 30, d=64, N=128, dq=0x1000, scale=0.125):
    a = P(0x1000)
    return lib.lib.fa_bwd(a, a, a, a, a, a, P(dq), a, a, 1, 1, N, d, scale, 0, P(ws), ws_bytes, None)


def test_bwd_validation(lib):
    need = lib.fa_bwd_workspace_bytes(1, 1, 128, 64)
    assert bwd(lib, ws=0) == lib.FA_ERR_WORKSPACE
    assert bwd(lib, ws_bytes=need - 1) == lib.FA_ERR_WORKSPACE
    assert bwd(lib, ws=0x10010) == lib.FA_ERR_WORKSPACE  # not 256-byte aligned
    assert bwd(lib, d=32) == lib.FA_ERR_UNSUPPORTED
    assert bwd(lib, dq=0) == lib.FA_ERR_INVALID_ARG
    assert bwd(lib, scale=-1.0) == lib.FA_ERR_INVALID_ARG
    assert bwd(lib, N=0, dq=0, ws=0) == lib.FA_OK


def test_bwd_deterministic_validation(lib):
    a = P(0x1000)
    need = lib.fa_bwd_deterministic_workspace_bytes(1, 1, 256, 64)
    call = lambda ws, nbytes, d=64: lib.lib.fa_bwd_deterministic(
        a, a, a, a, a, a, a, a, a, 1, 1, 256, d, 0.125, 0, P(ws), nbytes, None)
    assert call(0, need) == lib.FA_ERR_WORKSPACE
    assert call(0x10000, need - 1) == lib.FA_ERR_WORKSPACE
    assert call(0x10000, need, d=96) == lib.FA_ERR_UNSUPPORTED


def test_splitkv_workspace_bytes(lib):
    ws = lib.fa_fwd_splitkv_workspace_bytes
    up = lambda x: (x + 255) // 256 * 256
    B, H, N, d = 1, 4, 16300, 128
    slots = B * H * ((N + 255) // 256) * 8  # 256-row blocks x ranges
    assert ws(B, H, N, d, 8) == up(slots * 256 * d * 4) + up(slots * 256 * 4)
    assert ws(B, H, N, d, 1) == 0  # one range: fa_fwd, no workspace
    assert ws(B, H, N, d, 0) == 0
    assert ws(B, H, N, 96, 2) == 0


def test_splitkv_validation(lib):
    a = P(0x1000)
    call = lambda splits, ws, nbytes: lib.lib.fa_fwd_splitkv(
        a, a, a, a, a, 1, 1, 300, 64, 0.125, 0, splits, P(ws), nbytes, None)
    need = lib.fa_fwd_splitkv_workspace_bytes(1, 1, 300, 64, 2)
    assert call(0, 0x10000, need) == lib.FA_ERR_INVALID_ARG
    assert call(4, 0x10000, need) == lib.FA_ERR_INVALID_ARG  # 3 key tiles
    assert call(2, 0, need) == lib.FA_ERR_WORKSPACE
    assert call(2, 0x10000, need - 1) == lib.FA_ERR_WORKSPACE
    assert call(2, 0x10010, need) == lib.FA_ERR_WORKSPACE


def test_fp8_workspace_bytes(lib):
    ws = lib.fa_fwd_fp8_workspace_bytes
    up = lambda x: (x + 255) // 256 * 256
    B, H, N = 2, 3, 300
    rows, bh, np_ = B * H * N, B * H, 304
    blocks = (N + 127) // 128  # per-block amax slots of K and V
    # the FP8 operands and scales, then the forward's last-round split partials
    assert ws(B, H, N, 128) == (2 * up(rows * 128) + up(bh * 128 * np_) + up(rows * 4) +
                                up(2 * bh * 4) + up(2 * bh * blocks * 4) +
                                lib.fa_fwd_workspace_bytes(B, H, N, 128, False))
    assert ws(B, H, N, 64) == 0  # d = 128 only
    assert ws(0, H, N, 128) == 0


def test_fp8_validation(lib):
    a = P(0x1000)
    call = lambda d, ws, nbytes, rotate=1: lib.lib.fa_fwd_fp8(
        a, a, a, a, a, 1, 1, 256, d, 0.125, 0, rotate, P(ws), nbytes, None)
    need = lib.fa_fwd_fp8_workspace_bytes(1, 1, 256, 128)
    assert call(64, 0x10000, need) == lib.FA_ERR_UNSUPPORTED
    assert call(128, 0, need) == lib.FA_ERR_WORKSPACE
    assert call(128, 0x10000, need - 1) == lib.FA_ERR_WORKSPACE
    assert call(128, 0x10000, need, rotate=2) == lib.FA_ERR_INVALID_ARG


def test_diagnostics_validation(lib):
    assert lib.lib.fa_exp2_poly_eval(P(0), P(0), -1, None) == lib.FA_ERR_INVALID_ARG
    assert lib.lib.fa_exp2_poly_eval(P(0), P(0), 0, None) == lib.FA_OK
    assert lib.lib.fa_debug_bounded_wait(10, None) == lib.FA_ERR_INVALID_ARG


def test_binding_exposes_c_names(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_binding_rejects_host_operands(lib):
    """The binding refuses host tensors (operands or workspace) before any C
    call: the library takes device pointers only."""
    import torch

    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 1, 8, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lib.fa_fwd(q, q, q, q, lse, 0.125, False)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lib._workspace(torch.zeros(16, dtype=torch.uint8), torch.device("cuda", 0))
    assert lib._workspace(None, torch.device("cuda", 0)) == (None, 0)


def test_launch_counter_without_launches(lib):
    """Host-rejected calls launch nothing, so the counter does not move."""
    before = lib.fa_launch_count()
    assert lib.lib.fa_exp2_poly_eval(P(0), P(0), -1, None) == lib.FA_ERR_INVALID_ARG
    assert lib.lib.fa_debug_bounded_wait(10, None) == lib.FA_ERR_INVALID_ARG
    assert lib.fa_launch_count() == before
