"""gdn_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate.

Some callers cannot call cudaMalloc at all: an inference server or plugin host
that owns every byte of device memory through its own pool, or a real-time loop
that forbids allocation once it has started. This entry point takes only the
caller's inputs and outputs and keeps the forward's residual records in a static
device array inside the library. These tests call it through the C ABI twice in
a row (different inputs and shapes, so leftovers of the first call in the shared
array cannot leak into the second) and compare each result with gdn_chunk_fwd,
within the tolerance the parity tests use. The file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300 import binding
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

from helpers import TOL, cuda_inputs

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(d, out, h_final):
    lib = gdn.load()
    dims = gdn.make_dims(d["q"], d["v"], d["g"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gdn_chunk_fwd_noalloc(ctypes.byref(dims), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]),
                                     _ptr(d["g"]), _ptr(d["beta"]), _ptr(d["h0"]),
                                     float(dims.Dk ** -0.5), _ptr(out), _ptr(h_final), stream)


def _relerr(x, y):
    return float((x.double() - y.double()).norm() / y.double().norm())


def test_noalloc_forward_matches_the_allocating_entry_point_twice_in_a_row():
    cases = [
        ("bf16", WORKLOADS["train_fwd_bf16"].with_(B=1, T=4096, H=3), 0),  # 192 chunk-heads
        ("f32", WORKLOADS["train_fwd_f32"].with_(B=2, T=640, H=2, Dk=64, Dv=64), 1),
    ]
    for dtype, w, seed in cases:
        d = cuda_inputs(make_inputs(w, seed=seed))
        ref_out, ref_h, _ = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
        out = torch.full_like(ref_out, float("nan"))
        h_final = torch.full_like(ref_h, float("nan"))
        st = _call_noalloc(d, out, h_final)
        assert st == binding.GDN_OK, gdn.status_string(st)
        torch.cuda.synchronize()
        assert _relerr(out, ref_out) <= TOL[dtype]
        assert _relerr(h_final, ref_h) <= TOL[dtype]
    assert gdn.gdn_check_device_error() == 0


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    w = WORKLOADS["train_fwd_bf16"].with_(B=1, T=4096, H=4)  # 256 chunk-heads > 32 MiB of records
    d = cuda_inputs(make_inputs(w))
    dims = gdn.make_dims(d["q"], d["v"], d["g"])
    assert gdn.gdn_chunk_residual_bytes(dims) > binding.GDN_NOALLOC_SCRATCH_BYTES
    out = torch.empty_like(d["v"])
    h_final = torch.empty(1, 4, 128, 128, dtype=torch.float32, device="cuda")
    assert _call_noalloc(d, out, h_final) == binding.GDN_ERR_SCRATCH_LIMIT
    assert "scratch" in gdn.status_string(binding.GDN_ERR_SCRATCH_LIMIT)
