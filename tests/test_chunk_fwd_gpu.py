"""GPU parity of the chunked forward (gdn_chunk_fwd) against the float64 oracle.

Cases span several chunks and both blocks of a chunk, per-channel and scalar
decay, fp32 (rel-L2 <= 1e-4) and bf16 inputs (<= 2e-2), both score paths
(row-scaled products and the pairwise in-block sums), decay strong enough to
force the pairwise path by itself, and the training-shape forward workload
(B4 T4096 H6 D128) in full.
"""
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

from helpers import TOL, cuda_inputs, head_slice, oracle_fwd, rel

pytestmark = pytest.mark.gpu


def _fwd(d, flags=0):
    out, hT, _ = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=flags)
    return out, hT


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("flags", [0, gdn.GDN_FLAG_PAIRWISE_WITHIN_BLOCK])
def test_small_parity(dtype, per_channel, D, flags):
    w = WORKLOADS["train_fwd_f32"].with_(B=2, T=192, H=3, Dk=D, Dv=D, dtype=dtype,
                                         g_per_channel=per_channel, g_mult=1.0, h0_std=0.3)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host), flags)
    assert rel(out, o_ref) <= TOL[dtype], rel(out, o_ref)
    assert rel(hT, h_ref) <= TOL[dtype], rel(hT, h_ref)


def test_tiny_forward_workload():
    w = WORKLOADS["tiny_fwd"]
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host))
    assert rel(out, o_ref) <= TOL["f32"] and rel(hT, h_ref) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_extreme_decay_takes_the_pairwise_path(dtype):
    """Per-token decay ~3 nats: a 32-token block spreads ~100 nats, beyond the
    row-scaling range, so in-block scores come from the pairwise sums."""
    w = WORKLOADS["train_fwd_f32"].with_(B=1, T=128, H=2, Dk=64, Dv=64, dtype=dtype,
                                         g_mu=3.0, g_mult=1.0, h0_std=0.5)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host))
    assert rel(out, o_ref) <= TOL[dtype] and rel(hT, h_ref) <= TOL[dtype]


def test_paths_agree_and_are_deterministic():
    w = WORKLOADS["train_fwd_bf16"].with_(B=2, T=256, H=2)
    d = cuda_inputs(make_inputs(w))
    a1, h1 = _fwd(d)
    a2, h2 = _fwd(d)
    assert torch.equal(a1, a2) and torch.equal(h1, h2)
    p1, ph = _fwd(d, gdn.GDN_FLAG_PAIRWISE_WITHIN_BLOCK)
    assert float((p1.float() - a1.float()).norm() / a1.float().norm()) < 2e-2


def test_chunked_equals_recurrent_fp32():
    w = WORKLOADS["train_fwd_f32"].with_(B=1, T=320, H=4)
    d = cuda_inputs(make_inputs(w))
    out, hT = _fwd(d)
    ro, rh = gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    assert float((out - ro).norm() / ro.norm()) < 1e-4
    assert float((hT - rh).norm() / rh.norm()) < 1e-4


def test_edge_cases():
    w = WORKLOADS["train_fwd_f32"].with_(B=1, T=64, H=1, h0_std=0.5)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host))
    assert rel(out, o_ref) <= TOL["f32"] and rel(hT, h_ref) <= TOL["f32"]
    d = cuda_inputs(host)
    e = {k: (v[:, :0].contiguous() if k in ("q", "k", "v", "g", "beta", "dout") else v) for k, v in d.items()}
    out0, h00 = _fwd(e)
    assert out0.shape[1] == 0 and torch.equal(h00, d["h0"])
    ragged = cuda_inputs(make_inputs(w.with_(T=100)))  # T not a multiple of 64
    with pytest.raises(gdn.GdnError) as ei:
        _fwd(ragged)
    assert ei.value.status == 3  # GDN_ERR_SHAPE


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_training_shape_forward_workload(dtype):
    """B4 T4096 H6 D128 at full size, every head against the oracle."""
    w = WORKLOADS["train_fwd_f32" if dtype == "f32" else "train_fwd_bf16"]
    host = make_inputs(w)
    out, hT = _fwd(cuda_inputs(host))
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out, o_ref) <= TOL[dtype], rel(out, o_ref)
    assert rel(hT, h_ref) <= TOL[dtype], rel(hT, h_ref)


def test_qk_l2norm_forward_fp32():
    """GDN_FLAG_QK_L2NORM with fp32 inputs: within the fp32 tolerance of the oracle's
    normalised forward; the residual buffer grows by the normalised rows."""
    w = WORKLOADS["train_fwd_f32"].with_(B=1, T=192, H=2, normalize_qk=False, h0_std=0.1)
    host = make_inputs(w)
    d = cuda_inputs(host)
    flags = gdn.GDN_FLAG_QK_L2NORM
    out, hT, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=flags)
    o_ref, h_ref = oracle_fwd(host, qk_l2norm=True)
    assert rel(out, o_ref) <= TOL["f32"] and rel(hT, h_ref) <= TOL["f32"]
    plain = gdn.gdn_chunk_residual_bytes(gdn.make_dims(d["q"], d["v"], d["g"]))
    assert res.numel() > plain


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("Dk,Dv", [(64, 128), (128, 64)])
def test_unequal_key_value_widths(dtype, per_channel, Dk, Dv):
    """Dk != Dv on the chunked forward (the gated-deltanet kernel card, Requirements and
    limits, allows unequal key and value widths), fp32 and bf16 inputs."""
    w = WORKLOADS["train_fwd_f32"].with_(B=2, T=192, H=3, Dk=Dk, Dv=Dv, dtype=dtype,
                                         g_per_channel=per_channel, g_mult=1.0, h0_std=0.3)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host))
    assert rel(out, o_ref) <= TOL[dtype], rel(out, o_ref)
    assert rel(hT, h_ref) <= TOL[dtype], rel(hT, h_ref)


def test_concurrent_forward_calls_on_two_streams():
    """Two forward calls on two streams at the same time (different problems, disjoint
    residual buffers). Each runs its scan and chunk outputs as one cooperative launch whose
    output CTAs wait on its scan CTAs; both must match the oracle and report no error."""
    ws_ = [WORKLOADS["train_fwdbwd"].with_(B=2, T=1024, H=6, h0_std=0.2),
           WORKLOADS["train_fwdbwd"].with_(B=3, T=512, H=4, h0_std=0.1)]
    hosts = [make_inputs(w, seed=i) for i, w in enumerate(ws_)]
    ds = [cuda_inputs(h) for h in hosts]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    main = torch.cuda.current_stream()
    results = []
    for d, s in zip(ds, streams):
        s.wait_stream(main)
        with torch.cuda.stream(s):
            results.append(gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"]))
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK
    for host, (out, hT, _) in zip(hosts, results):
        o_ref, h_ref = oracle_fwd(host)
        assert rel(out, o_ref) <= TOL["bf16"] and rel(hT, h_ref) <= TOL["bf16"]
