"""GPU parity of the chunked backward (gdn_chunk_bwd) against the oracle's
hand-derived float64 reverse pass (rel-L2 <= 2e-2 per gradient, bf16 inputs).

Includes the training-shape fwd+bwd workload (B8 T4096 H6 D128 bf16) at full
size with the same launch the benchmark times; the oracle checks a sample of
(batch, head) pairs there (heads never interact, so a pair's gradients are those
of the pair alone).
"""
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

from helpers import TOL, cuda_inputs, head_slice, oracle_bwd, oracle_fwd, rel

pytestmark = pytest.mark.gpu
GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def _fwd_bwd(d, flags=0):
    out, hT, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=flags)
    grads = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res, d["dout"],
                              d["dh_final"], flags=flags)
    return out, hT, grads


@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("flags", [0, gdn.GDN_FLAG_PAIRWISE_WITHIN_BLOCK])
def test_small_parity(per_channel, D, flags):
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=192, H=2, Dk=D, Dv=D, g_per_channel=per_channel,
                                        g_mult=1.0 if per_channel else 0.1, h0_std=0.3)
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host), flags)
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


def test_extreme_decay_pairwise_backward():
    w = WORKLOADS["train_fwdbwd"].with_(B=1, T=128, H=2, Dk=64, Dv=64, g_mu=3.0, g_mult=1.0,
                                        h0_std=0.5)
    host = make_inputs(w)
    _, _, grads = _fwd_bwd(cuda_inputs(host))
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


def test_no_initial_state_and_no_final_gradient():
    w = WORKLOADS["train_fwdbwd"].with_(B=1, T=128, H=3, h0_std=0.0)
    host = make_inputs(w)
    host["dh_final"] = None
    d = cuda_inputs(host)
    out, hT, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None)
    grads = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, res, d["dout"], None)
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


def test_determinism():
    w = WORKLOADS["train_fwdbwd"].with_(B=1, T=256, H=2)
    d = cuda_inputs(make_inputs(w))
    _, _, g1 = _fwd_bwd(d)
    _, _, g2 = _fwd_bwd(d)
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


def test_autograd_wrapper():
    w = WORKLOADS["train_fwdbwd"].with_(B=1, T=128, H=2, h0_std=0.2)
    host = make_inputs(w)
    d = cuda_inputs(host)
    leaves = {n: d[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "h0")}
    out, hT = gdn.gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                   leaves["h0"])
    (out.float() * d["dout"].float()).sum().backward(retain_graph=True)
    hT.backward(d["dh_final"])
    ref = oracle_bwd(host)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    for n, gn in names.items():
        assert rel(leaves[n].grad, ref[gn]) <= TOL["bf16"], (n, rel(leaves[n].grad, ref[gn]))


def test_training_shape_fwd_bwd_workload():
    """B8 T4096 H6 D128 bf16: the benchmark's launch; oracle on sampled heads."""
    w = WORKLOADS["train_fwdbwd"]
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host))
    pairs = [(0, 0), (3, 5), (7, 2)]
    o_ref, h_ref = oracle_fwd(host, pairs)
    assert rel(head_slice(out.cpu(), pairs), o_ref) <= TOL["bf16"]
    assert rel(head_slice(hT.cpu(), pairs, state=True), h_ref) <= TOL["bf16"]
    ref = oracle_bwd(host, pairs)
    for n in GRADS:
        got = head_slice(grads[n].cpu(), pairs, state=(n == "dh0"))
        assert rel(got, ref[n]) <= TOL["bf16"], (n, rel(got, ref[n]))
    for n in GRADS:  # the heads not sampled are finite
        assert bool(torch.isfinite(grads[n].float()).all()), n


@pytest.mark.parametrize("D", [64, 128])
def test_qk_l2norm_forward_and_backward(D):
    """q and k drawn without normalisation (norms ~ sqrt(D)); with GDN_FLAG_QK_L2NORM the
    chunked forward and backward follow the oracle's normalised rule, and dq, dk are
    gradients with respect to the raw q, k."""
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=128, H=3, Dk=D, Dv=D, normalize_qk=False, h0_std=0.2)
    host = make_inputs(w)
    flags = gdn.GDN_FLAG_QK_L2NORM
    out, hT, grads = _fwd_bwd(cuda_inputs(host), flags)
    o_ref, h_ref = oracle_fwd(host, qk_l2norm=True)
    assert rel(out, o_ref) <= TOL["bf16"] and rel(hT, h_ref) <= TOL["bf16"]
    ref = oracle_bwd(host, qk_l2norm=True)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


@pytest.mark.parametrize("flags", [0, gdn.GDN_FLAG_PAIRWISE_WITHIN_BLOCK])
def test_scalar_decay_with_wipes(flags):
    """One decay per head with g = -20 wipes inside chunks (every 50 tokens): the scalar
    decay's mask form (decay as a C x C factor on the raw products) and the forced pairwise
    path both follow the oracle, forward and backward."""
    w = WORKLOADS["train_fwdbwd"].with_(B=1, T=256, H=3, g_per_channel=False, g_kind="logsigmoid",
                                        g_mu=2.0, wipe_every=50, h0_std=0.3)
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host), flags)
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out, o_ref) <= TOL["bf16"] and rel(hT, h_ref) <= TOL["bf16"]
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))
