"""Float64 CPU oracle for the gated delta rule (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The CUDA library and its Python binding never
touch it, and it shares no code with them: the only common module is the
seeded input generator, which holds none of the method's arithmetic.

Contents
- ``gdn_oracle.cpp``: the token-serial forward and its hand-derived reverse
  pass, in float64, threaded over (batch, head). Loaded here through ctypes.
- ``chunked_mirror.py``: a float64 numpy restatement of the chunked (WY/UT)
  form and of its backward, used to pin that derivation against the
  token-serial oracle. It is a second opinion on the algebra, never the
  reference values a GPU result is compared with.

Parity status: both entry points are pinned by tests in
``tests/test_oracle_pins.py`` (closed forms, gate semantics, the decay
factorisation worked example, finite differences, brute force), the optional
q/k L2 normalisation by finite differences and its scale invariance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (no GPU involved)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.oracle_fwd.argtypes = [i, i, i, i, i, i, dp, dp, dp, dp, dp, dp, ctypes.c_double,
                                       dp, dp, i]
            lib.oracle_fwd.restype = i
            lib.oracle_bwd.argtypes = [i, i, i, i, i, i, dp, dp, dp, dp, dp, dp, ctypes.c_double,
                                       dp, dp, dp, dp, dp, dp, dp, dp, i]
            lib.oracle_bwd.restype = i
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _c64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# The "gated-deltanet" kernel card (sections Usage and Correctness) offers an
# in-kernel L2 normalisation of q and k (use_qk_l2norm) without stating its
# guard for a zero vector; this oracle takes x / sqrt(sum_c x_c^2 + eps) per
# (token, head) with eps = 1e-6.
QK_L2NORM_EPS = 1e-6


def l2norm(x, eps: float = QK_L2NORM_EPS):
    """x / sqrt(sum over the last axis of x^2 + eps), float64."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def l2norm_backward(x, dxhat, eps: float = QK_L2NORM_EPS):
    """Gradient with respect to x of the normalisation above, given the gradient
    dxhat with respect to its output: with r = (|x|^2 + eps)^(-1/2) and
    xhat = r x, dx = r (dxhat - xhat <xhat, dxhat>)."""
    x = np.asarray(x, dtype=np.float64)
    dxhat = np.asarray(dxhat, dtype=np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    xhat = x * r
    return r * (dxhat - xhat * np.sum(xhat * dxhat, axis=-1, keepdims=True))


def fwd(q, k, v, g, beta, h0=None, scale: Optional[float] = None, nthreads: int = 0,
        qk_l2norm: bool = False):
    """Token-serial forward. Arrays as in the C ABI layouts, any float dtype
    (converted to float64). With qk_l2norm, q and k are first normalised per
    (token, head) by ``l2norm``. Returns (out [B,T,H,Dv], h_final [B,H,Dk,Dv])."""
    if qk_l2norm:
        q, k = l2norm(q), l2norm(k)
    q, k, v, g, beta, h0 = map(_c64, (q, k, v, g, beta, h0))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    per_channel = int(g.ndim == 4)
    if scale is None:
        scale = Dk ** -0.5
    out = np.zeros((B, T, H, Dv))
    h_final = np.zeros((B, H, Dk, Dv))
    rc = _load().oracle_fwd(B, T, H, Dk, Dv, per_channel, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), _ptr(h0), float(scale), _ptr(out), _ptr(h_final),
                            int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_fwd rejected its arguments (rc={rc})")
    return out, h_final


def bwd(q, k, v, g, beta, h0, dout, dh_final=None, scale: Optional[float] = None,
        nthreads: int = 0, qk_l2norm: bool = False) -> Dict[str, np.ndarray]:
    """Hand-derived reverse pass. Returns dq, dk, dv, dg, dbeta, dh0. With
    qk_l2norm the reverse pass runs on the normalised q, k and dq, dk are then
    taken back through ``l2norm_backward``."""
    if qk_l2norm:
        q_raw, k_raw = _c64(q), _c64(k)
        res = bwd(l2norm(q_raw), l2norm(k_raw), v, g, beta, h0, dout, dh_final, scale, nthreads)
        res["dq"] = l2norm_backward(q_raw, res["dq"])
        res["dk"] = l2norm_backward(k_raw, res["dk"])
        return res
    q, k, v, g, beta, h0, dout, dh_final = map(_c64, (q, k, v, g, beta, h0, dout, dh_final))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    per_channel = int(g.ndim == 4)
    if scale is None:
        scale = Dk ** -0.5
    res = {n: np.zeros(a.shape) for n, a in (("dq", q), ("dk", k), ("dv", v), ("dg", g),
                                                ("dbeta", beta))}
    res["dh0"] = np.zeros((B, H, Dk, Dv))
    rc = _load().oracle_bwd(B, T, H, Dk, Dv, per_channel, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), _ptr(h0), float(scale), _ptr(dout), _ptr(dh_final),
                            _ptr(res["dq"]), _ptr(res["dk"]), _ptr(res["dv"]), _ptr(res["dg"]),
                            _ptr(res["dbeta"]), _ptr(res["dh0"]), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_bwd rejected its arguments (rc={rc})")
    return res


def rel_l2(x, y) -> float:
    """||x - y||_2 / ||y||_2 over all elements (y = oracle); ||x||_2 if ||y|| = 0."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    ny = float(np.linalg.norm(y.ravel()))
    d = float(np.linalg.norm((x - y).ravel()))
    if ny == 0.0:
        return float(np.linalg.norm(x.ravel()))
    return d / ny
