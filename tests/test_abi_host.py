"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol include/gdn.h declares, sizes are consistent, and invalid arguments are
rejected with status codes before anything reaches a GPU. No kernel runs here."""
import ctypes
import os
import re

import pytest

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    return gdn.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert gdn.gdn_version() == 100
    assert lib.gdn_status_string(0).decode() == "ok"
    for s in range(6):
        assert lib.gdn_status_string(s)
    assert b"unknown" in lib.gdn_status_string(99)


def _dims(**kw):
    base = dict(B=2, T=128, H=3, Dk=128, Dv=128, g_per_channel=1, dtype=binding.GDN_BF16, flags=0)
    base.update(kw)
    return binding.GdnDims(**base)


def test_size_queries(lib):
    d = _dims()
    r = lib.gdn_chunk_residual_bytes(ctypes.byref(d))
    w = lib.gdn_chunk_bwd_workspace_bytes(ctypes.byref(d))
    n = 2 * 3 * 2  # chunk-heads
    C, D = 64, 128
    # Aqk, T, -W, U', Q-hat, K-tilde, state, U in bf16 plus gam in fp32 (each region 1 KiB aligned)
    want_r = n * (2 * C * C * 2 + 5 * C * D * 2 + D * D * 2 + D * 4)
    assert want_r <= r <= want_r + 9 * 1024
    assert r % 1024 == 0 and w % 1024 == 0
    d32 = _dims(dtype=binding.GDN_F32)
    assert lib.gdn_chunk_residual_bytes(ctypes.byref(d32)) > r
    assert lib.gdn_chunk_residual_bytes(ctypes.byref(_dims(T=100))) == 0  # T % 64 != 0
    assert lib.gdn_chunk_residual_bytes(ctypes.byref(_dims(Dk=96))) == 0
    assert lib.gdn_chunk_residual_bytes(None) == 0
    # linear in the number of chunk-heads
    r2 = lib.gdn_chunk_residual_bytes(ctypes.byref(_dims(T=256)))
    assert abs(r2 - 2 * r) <= 9 * 1024
    # the q/k L2 normalisation adds the normalised q, k rows (bf16) and their inverse norms
    rn = lib.gdn_chunk_residual_bytes(ctypes.byref(_dims(flags=binding.GDN_FLAG_QK_L2NORM)))
    rows = 2 * 128 * 3
    assert r + rows * (2 * D * 2 + 2 * 4) <= rn <= r + rows * (2 * D * 2 + 2 * 4) + 4 * 1024
    # 128-token chunks: the 64-token records (their states and U formed by the backward)
    # plus, per 128-token chunk-head, Aqk [128][128], -W, U', Q-hat, K-tilde [128][D], gam,
    # state and U
    f128 = binding.GDN_FLAG_CHUNK128
    r128 = lib.gdn_chunk_residual_bytes(ctypes.byref(_dims(flags=f128)))
    n2 = n // 2
    want128 = want_r + n2 * (128 * 128 * 2 + 5 * 128 * D * 2 + D * D * 2 + D * 4)
    assert want128 <= r128 <= want128 + 18 * 1024
    assert lib.gdn_chunk_residual_bytes(ctypes.byref(_dims(T=192, flags=f128))) == 0  # T % 128 != 0
    # the 128-token backward (bf16 operands only) passes the 64-token blocks' dU and dS1
    assert lib.gdn_chunk_bwd_workspace_bytes(ctypes.byref(_dims(flags=f128))) == w
    assert lib.gdn_chunk_bwd_workspace_bytes(ctypes.byref(_dims(flags=f128, dtype=binding.GDN_F32))) == 0


def _fake(addr=1 << 20):
    return ctypes.c_void_p(addr)


def test_invalid_arguments_are_rejected_on_the_host(lib):
    p = _fake()
    f = ctypes.c_float(0.1)
    fwd = lib.gdn_chunk_fwd
    # NULL dims
    assert fwd(None, p, p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_INVALID_ARG
    # unsupported widths / dtype / flags / shape
    assert fwd(ctypes.byref(_dims(Dk=96)), p, p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_UNSUPPORTED
    assert fwd(ctypes.byref(_dims(Dk=64, Dv=96)), p, p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_UNSUPPORTED
    assert fwd(ctypes.byref(_dims(dtype=7)), p, p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_UNSUPPORTED
    assert fwd(ctypes.byref(_dims(flags=8)), p, p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_dims(T=100)), p, p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_SHAPE
    f128 = binding.GDN_FLAG_CHUNK128
    assert fwd(ctypes.byref(_dims(T=192, flags=f128)), p, p, p, p, p, None, f, p, None, p,
               None) == binding.GDN_ERR_SHAPE
    assert fwd(ctypes.byref(_dims(flags=f128 | 8)), p, p, p, p, p, None, f, p, None, p,
               None) == binding.GDN_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_dims(B=-1)), p, p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_INVALID_ARG
    # NULL and misaligned required pointers, missing residuals, non-finite scale
    assert fwd(ctypes.byref(_dims()), None, p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_dims()), _fake((1 << 20) + 8), p, p, p, p, None, f, p, None, p, None) == binding.GDN_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_dims()), p, p, p, p, p, None, f, p, None, None, None) == binding.GDN_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_dims()), p, p, p, p, p, None, f, p, None, _fake((1 << 20) + 64), None) == binding.GDN_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_dims()), p, p, p, p, p, None, ctypes.c_float(float("nan")), p, None, p, None) == binding.GDN_ERR_INVALID_ARG
    # empty problems are accepted without touching the device
    assert fwd(ctypes.byref(_dims(B=0)), None, None, None, None, None, None, f, None, None, None, None) == binding.GDN_OK
    # backward: same widths and dtypes as the forward; workspace required
    bwd = lib.gdn_chunk_bwd
    args = [p, p, p, p, p, None, f, p, p, None, p, p, p, p, p, None, p, None]
    assert bwd(ctypes.byref(_dims(Dk=64, Dv=96)), *args) == binding.GDN_ERR_UNSUPPORTED
    assert bwd(ctypes.byref(_dims(dtype=7)), *args) == binding.GDN_ERR_UNSUPPORTED
    assert bwd(ctypes.byref(_dims(flags=binding.GDN_FLAG_CHUNK128, dtype=binding.GDN_F32)),
               *args) == binding.GDN_ERR_UNSUPPORTED
    bad = list(args)
    bad[16] = None  # workspace
    assert bwd(ctypes.byref(_dims()), *bad) == binding.GDN_ERR_INVALID_ARG
    bad = list(args)
    bad[8] = None  # dout
    assert bwd(ctypes.byref(_dims()), *bad) == binding.GDN_ERR_INVALID_ARG
    # recurrent: any T, mixed widths allowed; still validated
    rec = lib.gdn_recurrent
    assert rec(ctypes.byref(_dims(Dk=96)), p, p, p, p, p, None, f, p, p, None) == binding.GDN_ERR_UNSUPPORTED
    assert rec(ctypes.byref(_dims(T=13)), p, p, p, p, p, None, f, p, None, None) == binding.GDN_ERR_INVALID_ARG
    assert rec(ctypes.byref(_dims(B=0, T=5)), None, None, None, None, None, None, f, None, None, None) == binding.GDN_OK
    # scalar gates only need element alignment
    assert rec(ctypes.byref(_dims(T=13, g_per_channel=0)), p, p, p, _fake((1 << 20) + 3), p, None, f, p, p,
               None) == binding.GDN_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors():
    import torch

    q = torch.zeros(1, 64, 1, 64)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_chunk_fwd(q, q, q, q, torch.zeros(1, 64, 1))


def test_replay_sizes_and_validation(lib):
    d = _dims(T=1, dtype=binding.GDN_F32)
    # per (b, h): L slots of k, cumulative log-decay and delta, fp32
    assert lib.gdn_replay_buffer_bytes(ctypes.byref(d), 8) == 2 * 3 * 8 * (2 * 128 + 128) * 4
    assert lib.gdn_replay_buffer_bytes(ctypes.byref(_dims(T=1, Dk=64, Dv=128)), 1) == 2 * 3 * (2 * 64 + 128) * 4
    assert lib.gdn_replay_buffer_bytes(ctypes.byref(d), 0) == 0
    assert lib.gdn_replay_buffer_bytes(ctypes.byref(d), binding.GDN_REPLAY_MAX_TOKENS + 1) == 0
    assert lib.gdn_replay_buffer_bytes(ctypes.byref(_dims(T=1, Dk=96)), 4) == 0
    p, f = _fake(), ctypes.c_float(0.1)
    dec = lib.gdn_replay_decode
    ok_args = [p, p, p, p, p, f, p, p, p, p, None]
    assert dec(ctypes.byref(_dims(T=2)), 4, *ok_args) == binding.GDN_ERR_SHAPE
    assert dec(ctypes.byref(d), 0, *ok_args) == binding.GDN_ERR_INVALID_ARG
    assert dec(ctypes.byref(d), binding.GDN_REPLAY_MAX_TOKENS + 1, *ok_args) == binding.GDN_ERR_INVALID_ARG
    assert dec(ctypes.byref(_dims(T=1, Dk=96)), 4, *ok_args) == binding.GDN_ERR_UNSUPPORTED
    bad = list(ok_args)
    bad[6] = None  # ckpt
    assert dec(ctypes.byref(d), 4, *bad) == binding.GDN_ERR_INVALID_ARG
    bad = list(ok_args)
    bad[8] = _fake((1 << 20) + 2)  # fill not 4-byte aligned
    assert dec(ctypes.byref(d), 4, *bad) == binding.GDN_ERR_INVALID_ARG
    bad = list(ok_args)
    bad[5] = ctypes.c_float(float("inf"))
    assert dec(ctypes.byref(d), 4, *bad) == binding.GDN_ERR_INVALID_ARG
    assert dec(ctypes.byref(_dims(B=0, T=1)), 4, None, None, None, None, None, f, None, None, None, None,
               None) == binding.GDN_OK
    sta = lib.gdn_replay_state
    assert sta(ctypes.byref(d), 0, p, p, p, p, None) == binding.GDN_ERR_INVALID_ARG
    assert sta(ctypes.byref(d), 4, p, p, p, None, None) == binding.GDN_ERR_INVALID_ARG
    assert sta(ctypes.byref(_dims(B=0)), 4, None, None, None, None, None) == binding.GDN_OK


def test_selftest_rejects_bad_bounds_on_the_host(lib):
    # validated before anything touches a device
    assert lib.gdn_selftest_wait_timeout(0, None, None) == binding.GDN_ERR_INVALID_ARG
    assert lib.gdn_selftest_wait_timeout(1 << 20, None, None) == binding.GDN_ERR_INVALID_ARG
