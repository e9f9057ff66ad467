"""GPU parity of the token-recurrent kernel (gdn_recurrent) against the oracle.

Workloads: the tiny per-channel forward (B1 T128 H2 D64 fp32) and the
scalar-decay prefill+decode workload with periodic wipes (B2 H48 D128 T2048
fp32), whose required checks are one full call vs 128 calls of 16 tokens vs
2048 single-token decode calls, bitwise equal, each within 1e-4 of the oracle.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs, out_of_region_slice, to_f64
import oracle

from helpers import TOL, cuda_inputs, oracle_fwd, rel

pytestmark = pytest.mark.gpu


def _run(d, **kw):
    return gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], **kw)


@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_small_parity(per_channel, dims):
    w = WORKLOADS["tiny_fwd"].with_(T=77, H=3, B=2, Dk=dims[0], Dv=dims[1], h0_std=0.3,
                                    g_per_channel=per_channel)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _run(cuda_inputs(host))
    assert rel(out, o_ref) <= TOL["f32"]
    assert rel(hT, h_ref) <= TOL["f32"]


def test_tiny_forward_workload():
    w = WORKLOADS["tiny_fwd"]
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _run(cuda_inputs(host))
    assert rel(out, o_ref) <= TOL["f32"] and rel(hT, h_ref) <= TOL["f32"]


def test_bf16_inputs():
    w = WORKLOADS["tiny_fwd"].with_(dtype="bf16", T=200, H=4, Dk=128, Dv=128, h0_std=0.1)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _run(cuda_inputs(host))
    assert out.dtype == torch.bfloat16
    assert rel(out, o_ref) <= TOL["bf16"] and rel(hT, h_ref) <= 1e-4


def test_prefill_decode_workload_bitwise_and_parity():
    """One 2048-token call == 128 calls of 16 tokens == 2048 decode calls (bitwise),
    each within 1e-4 of the oracle."""
    w = WORKLOADS["recurrent"]
    host = make_inputs(w)
    d = cuda_inputs(host)
    out_full, h_full = _run(d)
    torch.cuda.synchronize()
    for step in (16, 1):
        state = None
        outs = []
        for t0 in range(0, w.T, step):
            sl = slice(t0, t0 + step)
            o, state = gdn.gdn_recurrent(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(),
                                         d["v"][:, sl].contiguous(), d["g"][:, sl].contiguous(),
                                         d["beta"][:, sl].contiguous(), state)
            outs.append(o)
        out_split = torch.cat(outs, 1)
        assert torch.equal(out_split, out_full), step
        assert torch.equal(state, h_full), step
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out_full, o_ref) <= TOL["f32"]
    assert rel(h_full, h_ref) <= TOL["f32"]


@pytest.mark.parametrize("H", [100, 3])
@pytest.mark.parametrize("dtype,dims,per_channel", [("bf16", (128, 128), True), ("f32", (64, 128), True),
                                                   ("f32", (128, 64), False), ("bf16", (64, 64), False)])
def test_single_token_calls_equal_one_call(dtype, dims, per_channel, H):
    """A sequence decoded one token per call (the single-token decode kernel, state
    carried in place) equals one prefill call bitwise, for every head geometry, both
    gate shapes and both input types. With H = 100 (200 heads, more than SMs) each
    decode CTA takes several whole heads; with H = 3 (fewer heads than SMs) each CTA
    takes a 32-column slice of one head."""
    w = WORKLOADS["tiny_fwd"].with_(B=2, T=24, H=H, Dk=dims[0], Dv=dims[1], dtype=dtype,
                                    g_per_channel=per_channel, h0_std=0.1)
    d = cuda_inputs(make_inputs(w))
    out_full, h_full = _run(d)
    state = d["h0"].clone()
    outs = []
    for t in range(w.T):
        sl = slice(t, t + 1)
        o, _ = gdn.gdn_recurrent(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(), d["v"][:, sl].contiguous(),
                                 d["g"][:, sl].contiguous(), d["beta"][:, sl].contiguous(), state, h_final=state)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, 1), out_full)
    assert torch.equal(state, h_full)
    assert gdn.gdn_check_device_error() == 0  # no bounded wait ran out


def test_in_place_state_carry_and_determinism():
    w = WORKLOADS["recurrent"].with_(B=1, T=100, H=4, h0_std=0.2)
    d = cuda_inputs(make_inputs(w))
    o1, h1 = _run(d)
    o2, h2 = _run(d)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    state = d["h0"].clone()
    o3, h3 = gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], state, h_final=state)
    assert h3.data_ptr() == state.data_ptr()
    assert torch.equal(o3, o1) and torch.equal(state, h1)


def test_gate_semantics():
    """beta = 0 and g = 0 is the exact identity; beta = 0 only decays."""
    w = WORKLOADS["tiny_fwd"].with_(T=50, H=2, B=2, Dk=128, Dv=128, h0_std=1.0)
    host = make_inputs(w)
    host["beta"] = torch.zeros_like(host["beta"])
    host["g"] = torch.zeros_like(host["g"])
    d = cuda_inputs(host)
    out, hT = _run(d)
    assert torch.equal(hT, d["h0"])
    host2 = make_inputs(w)
    host2["beta"] = torch.zeros_like(host2["beta"])
    d2 = cuda_inputs(host2)
    _, hT2 = _run(d2)
    fac = torch.exp(host2["g"].double().sum(1))  # [B,H,Dk]
    want = fac[..., None] * host2["h0"].double()
    assert rel(hT2, want.numpy()) <= 1e-5


def test_wipe_shrinks_state():
    w = WORKLOADS["recurrent"].with_(B=1, T=64, H=2, Dk=64, Dv=64, wipe_every=32, h0_std=1.0)
    host = make_inputs(w)
    d = cuda_inputs(host)
    big = dict(d, h0=d["h0"] * 1e3)
    zero = dict(d, h0=torch.zeros_like(d["h0"]))
    oa, _ = _run(big)
    ob, _ = _run(zero)
    after = (oa[:, 32:] - ob[:, 32:]).norm() / ob[:, 32:].norm()
    assert float(after) < 1e-4  # 1e3 * exp(-20) ~ 2e-6 plus decay


def test_edge_cases():
    w = WORKLOADS["tiny_fwd"].with_(T=1, H=2, B=1, Dk=64, Dv=64, h0_std=0.5)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _run(cuda_inputs(host))
    assert rel(out, o_ref) <= TOL["f32"] and rel(hT, h_ref) <= TOL["f32"]
    # T = 0 copies h0
    d = cuda_inputs(host)
    e = {k: (v[:, :0].contiguous() if k in ("q", "k", "v", "g", "beta", "dout") else v) for k, v in d.items()}
    out0, h0c = _run(e)
    assert out0.shape[1] == 0 and torch.equal(h0c, d["h0"])
    # no h0 given: zero state
    out1, h1 = gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], None)
    host["h0"] = None
    o_ref0, h_ref0 = oracle_fwd(host)
    assert rel(out1, o_ref0) <= TOL["f32"] and rel(h1, h_ref0) <= TOL["f32"]


def test_divergence_is_reproduced():
    """Out-of-region keys (beta |k|^2 >> 2): per-row agreement to 1e-4 while the
    oracle stays below 1e30; non-finite once the oracle leaves fp32 range."""
    w = WORKLOADS["long_context"].with_(B=1, T=64, H=2, dtype="f32")
    sl = out_of_region_slice(w, torch.randn(1, 2, 128, 128, generator=torch.Generator().manual_seed(3)) * 0.01)
    o_ref, _ = oracle.fwd(*[to_f64(sl[n]) for n in ("q", "k", "v", "g", "beta", "h0")])
    out, _ = gdn.gdn_recurrent(*[sl[n].cuda() if sl[n] is not None else None
                                 for n in ("q", "k", "v", "g", "beta", "h0")])
    o = out.double().cpu().numpy()
    norms = np.linalg.norm(o_ref, axis=-1)  # [1, T, H]
    assert norms.max() > 1e3 * norms.min()  # it does diverge
    checked = 0
    for t in range(o.shape[1]):
        for h in range(o.shape[2]):
            ref = o_ref[0, t, h]
            if np.linalg.norm(ref) < 1e30:
                err = np.linalg.norm(o[0, t, h] - ref) / max(np.linalg.norm(ref), 1e-30)
                assert err <= 1e-4, (t, h, err)
                checked += 1
            elif np.linalg.norm(ref) > 3.4e38 or not np.isfinite(np.linalg.norm(ref)):
                assert not np.all(np.isfinite(o[0, t, h])), (t, h)
    assert checked > 0


@pytest.mark.parametrize("dtype,per_channel", [("f32", False), ("bf16", True)])
def test_qk_l2norm_recurrent_and_decode(dtype, per_channel):
    """GDN_FLAG_QK_L2NORM in the recurrent kernel and the single-token decode kernel:
    within tolerance of the oracle's normalised rule, and one token per call (decode,
    state carried in place) equals one prefill call bitwise."""
    w = WORKLOADS["tiny_fwd"].with_(B=2, T=40, H=5, Dk=128, Dv=128, dtype=dtype, g_per_channel=per_channel,
                                    normalize_qk=False, h0_std=0.1)
    host = make_inputs(w)
    d = cuda_inputs(host)
    flags = gdn.GDN_FLAG_QK_L2NORM
    out_full, h_full = _run(d, flags=flags)
    o_ref, h_ref = oracle_fwd(host, qk_l2norm=True)
    assert rel(out_full, o_ref) <= TOL[dtype] and rel(h_full, h_ref) <= 1e-4
    state = d["h0"].clone()
    outs = []
    for t in range(w.T):
        sl = slice(t, t + 1)
        o, _ = gdn.gdn_recurrent(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(), d["v"][:, sl].contiguous(),
                                 d["g"][:, sl].contiguous(), d["beta"][:, sl].contiguous(), state, h_final=state,
                                 flags=flags)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, 1), out_full)
    assert torch.equal(state, h_full)
