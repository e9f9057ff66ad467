"""Back-to-back training steps on one stream that reuse the residual and workspace
buffers, with different inputs each step. The chunk kernels are launched so that each
may be scheduled while the previous one finishes, and the backward runs part of its
work on the library's side stream: every step must still see only its own forward's
records (no kernel of step i + 1 may overwrite what step i's backward still reads)."""
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

from helpers import TOL, cuda_inputs, oracle_bwd, oracle_fwd, rel

pytestmark = pytest.mark.gpu


def test_back_to_back_steps_reusing_buffers():
    base = WORKLOADS["train_fwdbwd"].with_(B=2, T=256, H=2)
    hosts = [make_inputs(base.with_(g_mult=m, h0_std=s)) for m, s in ((0.1, 0.01), (1.0, 0.3), (0.3, 0.0))]
    devs = [cuda_inputs(h) for h in hosts]
    d0 = devs[0]
    dims = gdn.make_dims(d0["q"], d0["v"], d0["g"])
    res = torch.empty(gdn.gdn_chunk_residual_bytes(dims), dtype=torch.uint8, device="cuda")
    ws = torch.empty(gdn.gdn_chunk_bwd_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    results = []
    for d in devs:  # queued back to back, no synchronisation in between
        out, hT, _ = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], residuals=res)
        grads = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res, d["dout"],
                                  d["dh_final"], workspace=ws)
        results.append((out, hT, grads))
    torch.cuda.synchronize()
    for host, (out, hT, grads) in zip(hosts, results):
        o_ref, h_ref = oracle_fwd(host)
        ref = oracle_bwd(host)
        assert rel(out, o_ref) <= TOL["bf16"] and rel(hT, h_ref) <= TOL["bf16"]
        for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
            assert rel(grads[name], ref[name]) <= TOL["bf16"], name
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK
