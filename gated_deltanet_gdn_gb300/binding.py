"""ctypes binding of libgdn.so (include/gdn.h). Argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; PyTorch only
allocates device memory and supplies the current CUDA stream. There is no CPU
or framework fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, Optional, Tuple

import torch

from . import build as _build

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_SHAPE = 3
GDN_ERR_CUDA = 4
GDN_ERR_INTERNAL = 5
GDN_ERR_SCRATCH_LIMIT = 6
GDN_NOALLOC_SCRATCH_BYTES = 32 << 20
GDN_F32 = 0
GDN_BF16 = 1
GDN_FLAG_PAIRWISE_WITHIN_BLOCK = 1
GDN_FLAG_QK_L2NORM = 2
GDN_FLAG_CHUNK128 = 4
GDN_CHUNK = 64
GDN_CHUNK128 = 128

# every symbol include/gdn.h declares
EXPORTED = ("gdn_chunk_residual_bytes", "gdn_chunk_bwd_workspace_bytes", "gdn_chunk_fwd",
            "gdn_chunk_bwd", "gdn_recurrent", "gdn_check_device_error", "gdn_status_string",
            "gdn_version", "gdn_profile_enable", "gdn_profile_read", "gdn_kernel_name",
            "gdn_chunk_fwd_noalloc", "gdn_replay_buffer_bytes", "gdn_replay_decode",
            "gdn_replay_state", "gdn_selftest_wait_timeout")
KERNEL_COUNT = 21
GDN_REPLAY_MAX_TOKENS = 8


class GdnDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("Dk", ctypes.c_int), ("Dv", ctypes.c_int), ("g_per_channel", ctypes.c_int),
                ("dtype", ctypes.c_int), ("flags", ctypes.c_int)]


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load libgdn.so (building it first when missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_needed and _build.is_stale():
                _build.build()
            if not os.path.exists(_build.LIB_PATH):
                raise RuntimeError(f"libgdn.so not found at {_build.LIB_PATH}; run the package build first")
            lib = ctypes.CDLL(_build.LIB_PATH)
            vp, sz, i, f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
            pd = ctypes.POINTER(GdnDims)
            lib.gdn_chunk_residual_bytes.argtypes = [pd]
            lib.gdn_chunk_residual_bytes.restype = sz
            lib.gdn_chunk_bwd_workspace_bytes.argtypes = [pd]
            lib.gdn_chunk_bwd_workspace_bytes.restype = sz
            lib.gdn_chunk_fwd.argtypes = [pd, vp, vp, vp, vp, vp, vp, f, vp, vp, vp, vp]
            lib.gdn_chunk_fwd.restype = i
            lib.gdn_chunk_bwd.argtypes = [pd, vp, vp, vp, vp, vp, vp, f, vp, vp, vp, vp, vp, vp, vp,
                                          vp, vp, vp, vp]
            lib.gdn_chunk_bwd.restype = i
            lib.gdn_recurrent.argtypes = [pd, vp, vp, vp, vp, vp, vp, f, vp, vp, vp]
            lib.gdn_recurrent.restype = i
            lib.gdn_check_device_error.argtypes = []
            lib.gdn_check_device_error.restype = i
            lib.gdn_status_string.argtypes = [i]
            lib.gdn_status_string.restype = ctypes.c_char_p
            lib.gdn_version.argtypes = []
            lib.gdn_version.restype = i
            lib.gdn_profile_enable.argtypes = [i]
            lib.gdn_profile_enable.restype = i
            lib.gdn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i), i]
            lib.gdn_profile_read.restype = i
            lib.gdn_kernel_name.argtypes = [i]
            lib.gdn_kernel_name.restype = ctypes.c_char_p
            lib.gdn_chunk_fwd_noalloc.argtypes = [pd, vp, vp, vp, vp, vp, vp, f, vp, vp, vp]
            lib.gdn_chunk_fwd_noalloc.restype = i
            lib.gdn_replay_buffer_bytes.argtypes = [pd, i]
            lib.gdn_replay_buffer_bytes.restype = sz
            lib.gdn_replay_decode.argtypes = [pd, i, vp, vp, vp, vp, vp, f, vp, vp, vp, vp, vp]
            lib.gdn_replay_decode.restype = i
            lib.gdn_replay_state.argtypes = [pd, i, vp, vp, vp, vp, vp]
            lib.gdn_replay_state.restype = i
            lib.gdn_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp, vp]
            lib.gdn_selftest_wait_timeout.restype = i
            _lib = lib
    return _lib


def lib_path() -> str:
    return _build.LIB_PATH


def status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != GDN_OK:
        raise GdnError(fn, status, status_string(status))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return GDN_F32
    if dt == torch.bfloat16:
        return GDN_BF16
    raise GdnError("dtype", GDN_ERR_UNSUPPORTED, f"unsupported dtype {dt} (float32 or bfloat16)")


def make_dims(q: torch.Tensor, v: torch.Tensor, g: torch.Tensor, flags: int = 0) -> GdnDims:
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    return GdnDims(B, T, H, Dk, Dv, int(g.dim() == 4), _dtype_code(q.dtype), int(flags))


def _stream(dev: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _require(tensors: Dict[str, Optional[torch.Tensor]], device: torch.device):
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda or t.device != device:
            raise GdnError(name, GDN_ERR_INVALID_ARG, f"{name} must be a CUDA tensor on {device}")
        if not t.is_contiguous():
            raise GdnError(name, GDN_ERR_INVALID_ARG, f"{name} must be contiguous")


def gdn_chunk_residual_bytes(dims: GdnDims) -> int:
    return int(load().gdn_chunk_residual_bytes(ctypes.byref(dims)))


def gdn_chunk_bwd_workspace_bytes(dims: GdnDims) -> int:
    return int(load().gdn_chunk_bwd_workspace_bytes(ctypes.byref(dims)))


def gdn_chunk_fwd(q, k, v, g, beta, h0=None, scale: Optional[float] = None, *, out=None,
                  h_final=None, residuals=None, flags: int = 0):
    """Chunked forward. Returns (out [B,T,H,Dv], h_final fp32 [B,H,Dk,Dv], residuals)."""
    dev = q.device
    _require(dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, out=out, h_final=h_final,
                  residuals=residuals), dev)
    dims = make_dims(q, v, g, flags)
    if scale is None:
        scale = dims.Dk ** -0.5
    if out is None:
        out = torch.empty(v.shape, dtype=v.dtype, device=dev)
    if h_final is None:
        h_final = torch.empty((dims.B, dims.H, dims.Dk, dims.Dv), dtype=torch.float32, device=dev)
    if residuals is None:
        residuals = torch.empty(max(gdn_chunk_residual_bytes(dims), 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = load().gdn_chunk_fwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(h0), float(scale), _ptr(out), _ptr(h_final), _ptr(residuals),
                                  _stream(dev))
    _check("gdn_chunk_fwd", st)
    return out, h_final, residuals


def gdn_chunk_fwd_noalloc(q, k, v, g, beta, h0=None, scale: Optional[float] = None, *, out,
                          h_final, flags: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Chunked forward through the entry point that allocates nothing: the caller
    passes the outputs, the library keeps the residual records in its static
    device array (calls sharing it must not overlap on the GPU)."""
    dev = q.device
    _require(dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, out=out, h_final=h_final), dev)
    dims = make_dims(q, v, g, flags)
    if scale is None:
        scale = dims.Dk ** -0.5
    with torch.cuda.device(dev):
        st = load().gdn_chunk_fwd_noalloc(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                          _ptr(beta), _ptr(h0), float(scale), _ptr(out), _ptr(h_final),
                                          _stream(dev))
    _check("gdn_chunk_fwd_noalloc", st)
    return out, h_final


def gdn_chunk_bwd(q, k, v, g, beta, h0, residuals, dout, dh_final=None,
                  scale: Optional[float] = None, *, workspace=None, flags: int = 0,
                  need_dh0: bool = True, grads: Optional[Dict[str, torch.Tensor]] = None
                  ) -> Dict[str, torch.Tensor]:
    """Chunked backward (bf16 or fp32, the forward's dtype). Returns dq, dk, dv, dg, dbeta
    (input dtype) and dh0 (fp32).
    ``grads`` may supply preallocated output tensors under those names."""
    dev = q.device
    dims = make_dims(q, v, g, flags)
    if scale is None:
        scale = dims.Dk ** -0.5
    if grads is None:
        grads = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
                 "dg": torch.empty_like(g), "dbeta": torch.empty_like(beta)}
        grads["dh0"] = (torch.empty((dims.B, dims.H, dims.Dk, dims.Dv), dtype=torch.float32,
                                    device=dev) if need_dh0 else None)
    _require(dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, residuals=residuals, dout=dout,
                  dh_final=dh_final, workspace=workspace, **grads), dev)
    if workspace is None:
        workspace = torch.empty(max(gdn_chunk_bwd_workspace_bytes(dims), 1), dtype=torch.uint8,
                                device=dev)
    with torch.cuda.device(dev):
        st = load().gdn_chunk_bwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(h0), float(scale), _ptr(residuals), _ptr(dout),
                                  _ptr(dh_final), _ptr(grads["dq"]), _ptr(grads["dk"]),
                                  _ptr(grads["dv"]), _ptr(grads["dg"]), _ptr(grads["dbeta"]),
                                  _ptr(grads["dh0"]), _ptr(workspace), _stream(dev))
    _check("gdn_chunk_bwd", st)
    return grads


def gdn_recurrent(q, k, v, g, beta, h0=None, scale: Optional[float] = None, *, out=None,
                  h_final=None, flags: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Token-recurrent prefill / decode. h_final may be h0 (in-place carry)."""
    dev = q.device
    _require(dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, out=out, h_final=h_final), dev)
    dims = make_dims(q, v, g, flags)
    if scale is None:
        scale = dims.Dk ** -0.5
    if out is None:
        out = torch.empty(v.shape, dtype=v.dtype, device=dev)
    if h_final is None:
        h_final = torch.empty((dims.B, dims.H, dims.Dk, dims.Dv), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = load().gdn_recurrent(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(h0), float(scale), _ptr(out), _ptr(h_final), _stream(dev))
    _check("gdn_recurrent", st)
    return out, h_final


def gdn_replay_buffer_bytes(dims: GdnDims, L: int) -> int:
    return int(load().gdn_replay_buffer_bytes(ctypes.byref(dims), int(L)))


def replay_init(h0: torch.Tensor, L: int):
    """(ckpt, buffer, fill) for replay decode starting from state h0 [B,H,Dk,Dv] fp32:
    the checkpoint is a copy of h0, the buffer is empty (fill = 0)."""
    B, H, Dk, Dv = h0.shape
    dims = GdnDims(B, 1, H, Dk, Dv, 1, GDN_F32, 0)
    nbytes = gdn_replay_buffer_bytes(dims, L)
    if nbytes == 0 and B * H > 0:
        raise GdnError("gdn_replay_buffer_bytes", GDN_ERR_INVALID_ARG, f"bad dims or L={L}")
    ckpt = h0.detach().to(torch.float32).contiguous().clone()
    buffer = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=h0.device)
    fill = torch.zeros((B, H), dtype=torch.int32, device=h0.device)
    return ckpt, buffer, fill


def gdn_replay_decode(q, k, v, g, beta, ckpt, buffer, fill, L: int, scale: Optional[float] = None, *,
                      out=None, flags: int = 0) -> torch.Tensor:
    """One decode step (T = 1) against checkpoint + buffer; advances fill, folds the
    buffer into ckpt when it is full. Returns out [B,1,H,Dv]."""
    dev = q.device
    _require(dict(q=q, k=k, v=v, g=g, beta=beta, ckpt=ckpt, buffer=buffer, fill=fill, out=out), dev)
    dims = make_dims(q, v, g, flags)
    if scale is None:
        scale = dims.Dk ** -0.5
    if out is None:
        out = torch.empty(v.shape, dtype=v.dtype, device=dev)
    with torch.cuda.device(dev):
        st = load().gdn_replay_decode(ctypes.byref(dims), int(L), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                      _ptr(beta), float(scale), _ptr(ckpt), _ptr(buffer), _ptr(fill),
                                      _ptr(out), _stream(dev))
    _check("gdn_replay_decode", st)
    return out


def gdn_replay_state(ckpt, buffer, fill, L: int, *, h_out=None) -> torch.Tensor:
    """The full state [B,H,Dk,Dv] fp32 that checkpoint + buffer stand for."""
    dev = ckpt.device
    _require(dict(ckpt=ckpt, buffer=buffer, fill=fill, h_out=h_out), dev)
    B, H, Dk, Dv = ckpt.shape
    dims = GdnDims(B, 1, H, Dk, Dv, 1, GDN_F32, 0)
    if h_out is None:
        h_out = torch.empty_like(ckpt)
    with torch.cuda.device(dev):
        st = load().gdn_replay_state(ctypes.byref(dims), int(L), _ptr(ckpt), _ptr(buffer), _ptr(fill),
                                     _ptr(h_out), _stream(dev))
    _check("gdn_replay_state", st)
    return h_out


def gdn_selftest_wait_timeout(max_tries: int = 1024, device: Optional[torch.device] = None,
                              cycles: Optional[torch.Tensor] = None) -> None:
    """Launch the library's wait-timeout self-test kernel (see include/gdn.h). cycles: an
    optional int64 device tensor of three elements for the kernel's cycle counts."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    if cycles is not None:
        assert cycles.dtype == torch.int64 and cycles.numel() >= 3 and cycles.is_contiguous()
    with torch.cuda.device(dev):
        st = load().gdn_selftest_wait_timeout(int(max_tries), _ptr(cycles), _stream(dev))
    _check("gdn_selftest_wait_timeout", st)


def gdn_check_device_error() -> int:
    return int(load().gdn_check_device_error())


def gdn_version() -> int:
    return int(load().gdn_version())


def gdn_profile_enable(on: bool = True) -> None:
    _check("gdn_profile_enable", load().gdn_profile_enable(int(bool(on))))


def gdn_profile_read() -> Dict[str, Tuple[float, int]]:
    """{kernel name: (summed ms, launches)} since the last enable/read (kernels launched at least once)."""
    ms = (ctypes.c_double * KERNEL_COUNT)()
    n = (ctypes.c_int * KERNEL_COUNT)()
    _check("gdn_profile_read", load().gdn_profile_read(ms, n, KERNEL_COUNT))
    lib = load()
    return {lib.gdn_kernel_name(i).decode(): (float(ms[i]), int(n[i])) for i in range(KERNEL_COUNT) if n[i]}


def gdn_kernel_name(i: int) -> str:
    return load().gdn_kernel_name(int(i)).decode()


class GatedDeltaRule(torch.autograd.Function):
    """Chunked gated delta rule with the library's backward (bf16 or fp32)."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, h0, scale, flags):
        out, h_final, res = gdn_chunk_fwd(q, k, v, g, beta, h0, scale, flags=flags)
        ctx.save_for_backward(q, k, v, g, beta, h0, res)
        ctx.scale = scale
        ctx.flags = flags
        return out, h_final

    @staticmethod
    def backward(ctx, dout, dh_final):
        q, k, v, g, beta, h0, res = ctx.saved_tensors
        grads = gdn_chunk_bwd(q, k, v, g, beta, h0, res, dout.contiguous(),
                              None if dh_final is None else dh_final.contiguous(), ctx.scale,
                              flags=ctx.flags, need_dh0=h0 is not None)
        return (grads["dq"], grads["dk"], grads["dv"], grads["dg"], grads["dbeta"],
                grads["dh0"] if h0 is not None else None, None, None)


def gated_delta_rule(q, k, v, g, beta, h0=None, scale: Optional[float] = None, flags: int = 0):
    """(out, h_final) of the chunked gated delta rule, differentiable through autograd."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    return GatedDeltaRule.apply(q, k, v, g, beta, h0, float(scale), int(flags))
