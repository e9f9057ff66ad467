"""GPU parity of the chunked forward over 128-token chunks (GDN_FLAG_CHUNK128: two
64-token blocks per chunk, merged by chunk_merge128_kernel) against the float64 oracle.

Cases span several 128-token chunks, fp32 (rel-L2 <= 1e-4) and bf16 (<= 2e-2), per-channel
and scalar decay, every width pair, both in-block score paths, decay strong enough that the
cross-block factors underflow, the q/k L2 normalisation, the allocation-free entry point,
the training-shape forward workload (B4 T4096 H6 D128) on every head, agreement with the
64-token chunking, determinism and the shape and backward refusals.
"""
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

from helpers import TOL, cuda_inputs, oracle_fwd, rel

pytestmark = pytest.mark.gpu

F128 = gdn.GDN_FLAG_CHUNK128


def _fwd(d, flags=F128):
    out, hT, _ = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=flags)
    return out, hT


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("Dk,Dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_small_parity(dtype, per_channel, Dk, Dv):
    w = WORKLOADS["train_fwd_f32"].with_(B=2, T=384, H=3, Dk=Dk, Dv=Dv, dtype=dtype,
                                         g_per_channel=per_channel, g_mult=1.0, h0_std=0.3)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host))
    print("C=128 %s pc=%d %dx%d: out %.3e h_final %.3e" % (dtype, per_channel, Dk, Dv, rel(out, o_ref),
                                                            rel(hT, h_ref)))
    assert rel(out, o_ref) <= TOL[dtype], rel(out, o_ref)
    assert rel(hT, h_ref) <= TOL[dtype], rel(hT, h_ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pairwise_in_block_scores(dtype):
    w = WORKLOADS["train_fwd_f32"].with_(B=1, T=256, H=2, dtype=dtype, g_mult=1.0, h0_std=0.3)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host), F128 | gdn.GDN_FLAG_PAIRWISE_WITHIN_BLOCK)
    assert rel(out, o_ref) <= TOL[dtype] and rel(hT, h_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_extreme_decay(dtype):
    """About 3 nats of decay per token: the 64-token blocks spread about 200 nats, so the
    cross-block factors exp(G_i - G_b), exp(G_b - G_j) underflow for far pairs (as the true
    weights do) and the in-block scores take the pairwise path."""
    w = WORKLOADS["train_fwd_f32"].with_(B=1, T=256, H=2, Dk=64, Dv=64, dtype=dtype,
                                         g_mu=3.0, g_mult=1.0, h0_std=0.5)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host))
    assert rel(out, o_ref) <= TOL[dtype] and rel(hT, h_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_training_shape_forward_workload(dtype):
    """B4 T4096 H6 D128 at full size over 128-token chunks, every head against the oracle."""
    w = WORKLOADS["train_fwd_f32" if dtype == "f32" else "train_fwd_bf16"]
    host = make_inputs(w)
    out, hT = _fwd(cuda_inputs(host))
    o_ref, h_ref = oracle_fwd(host)
    print("C=128 training-shape %s: out %.3e h_final %.3e" % (dtype, rel(out, o_ref), rel(hT, h_ref)))
    assert rel(out, o_ref) <= TOL[dtype], rel(out, o_ref)
    assert rel(hT, h_ref) <= TOL[dtype], rel(hT, h_ref)


def test_agrees_with_64_token_chunks_and_is_deterministic():
    for dtype, tol in (("f32", 2e-5), ("bf16", 1e-2)):
        w = WORKLOADS["train_fwd_f32"].with_(B=2, T=512, H=4, dtype=dtype, h0_std=0.2)
        d = cuda_inputs(make_inputs(w))
        a1, h1 = _fwd(d)
        a2, h2 = _fwd(d)
        assert torch.equal(a1, a2) and torch.equal(h1, h2)
        b1, g1 = _fwd(d, 0)
        assert float((a1.float() - b1.float()).norm() / b1.float().norm()) < tol
        assert float((h1 - g1).norm() / g1.norm()) < tol


def test_qk_l2norm_fp32():
    w = WORKLOADS["train_fwd_f32"].with_(B=1, T=256, H=2, normalize_qk=False, h0_std=0.1)
    host = make_inputs(w)
    d = cuda_inputs(host)
    flags = F128 | gdn.GDN_FLAG_QK_L2NORM
    out, hT, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=flags)
    o_ref, h_ref = oracle_fwd(host, qk_l2norm=True)
    assert rel(out, o_ref) <= TOL["f32"] and rel(hT, h_ref) <= TOL["f32"]


def test_allocation_free_entry_point():
    w = WORKLOADS["train_fwd_bf16"].with_(B=1, T=512, H=2, h0_std=0.2)
    host = make_inputs(w)
    d = cuda_inputs(host)
    out = torch.empty_like(d["v"])
    hT = torch.empty_like(d["h0"])
    gdn.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], out=out, h_final=hT,
                              flags=F128)
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out, o_ref) <= TOL["bf16"] and rel(hT, h_ref) <= TOL["bf16"]


def test_edge_cases():
    w = WORKLOADS["train_fwd_f32"].with_(B=1, T=128, H=1, h0_std=0.5)
    host = make_inputs(w)
    o_ref, h_ref = oracle_fwd(host)
    out, hT = _fwd(cuda_inputs(host))  # one chunk
    assert rel(out, o_ref) <= TOL["f32"] and rel(hT, h_ref) <= TOL["f32"]
    d = cuda_inputs(make_inputs(w.with_(T=256, h0_std=0.0)))
    d["h0"] = None  # zero initial state
    out, hT = _fwd(d)
    o_ref, h_ref = oracle_fwd({k: (v.cpu() if v is not None else None) for k, v in d.items()})
    assert rel(out, o_ref) <= TOL["f32"] and rel(hT, h_ref) <= TOL["f32"]
    e = {k: (v[:, :0].contiguous() if k in ("q", "k", "v", "g", "beta", "dout") else v)
         for k, v in cuda_inputs(host).items()}
    out0, h00 = _fwd(e)
    assert out0.shape[1] == 0 and torch.equal(h00, e["h0"])
    with pytest.raises(gdn.GdnError) as ei:  # 64-token multiple, not a 128-token one
        _fwd(cuda_inputs(make_inputs(w.with_(T=192))))
    assert ei.value.status == 3  # GDN_ERR_SHAPE
    d = cuda_inputs(make_inputs(WORKLOADS["train_fwdbwd"].with_(B=1, T=256, H=2)))
    _, _, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=F128)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res, d["dout"], flags=F128)
    assert ei.value.status == 2  # GDN_ERR_UNSUPPORTED: no backward over 128-token chunks
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK
