"""GPU parity of the chunked forward and backward over 128-token chunks
(GDN_FLAG_CHUNK128: two 64-token blocks per chunk, merged by chunk_merge128_kernel; the
backward's reverse scan over the 128-token chunks, then chunk_mid128_kernel and the
64-token chunk products) against the float64 oracle.

Forward cases span several 128-token chunks, fp32 (rel-L2 <= 1e-4) and bf16 (<= 2e-2),
per-channel and scalar decay, every width pair, both in-block score paths, decay strong
enough that the cross-block factors underflow, the q/k L2 normalisation, the
allocation-free entry point and the training-shape forward workload (B4 T4096 H6 D128) on
every head. Backward cases (bf16): every width pair, both decay forms, no h0 and no
dh_final, autograd, and the training-shape fwd+bwd workload (B8 T4096 H6 D128) on every
head. Plus agreement with the 64-token chunking, determinism and the shape and dtype
refusals.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

from helpers import TOL, cuda_inputs, head_slice, oracle_bwd, oracle_fwd, rel

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
    d = cuda_inputs(make_inputs(WORKLOADS["train_fwdbwd"].with_(B=1, T=256, H=2, dtype="f32")))
    _, _, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=F128)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res, d["dout"], flags=F128)
    assert ei.value.status == 2  # GDN_ERR_UNSUPPORTED: fp32 backward over 128-token chunks
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK


# ---------------------------------------------------------------- backward
GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def _fwd_bwd(d, flags=F128):
    out, hT, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=flags)
    grads = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res, d["dout"],
                              d["dh_final"], flags=flags)
    return out, hT, grads


@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("Dk,Dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_backward_parity(per_channel, Dk, Dv):
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=384, H=3, Dk=Dk, Dv=Dv, g_per_channel=per_channel,
                                        g_mult=1.0 if per_channel else 0.1, h0_std=0.3)
    host = make_inputs(w)
    _, _, grads = _fwd_bwd(cuda_inputs(host))
    ref = oracle_bwd(host)
    print("C=128 bwd pc=%d %dx%d: " % (per_channel, Dk, Dv) +
          " ".join("%s %.2e" % (n, rel(grads[n], ref[n])) for n in GRADS))
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


def test_backward_without_h0_or_final_gradient_and_autograd():
    w = WORKLOADS["train_fwdbwd"].with_(B=1, T=256, H=3, h0_std=0.0)
    host = make_inputs(w)
    host["dh_final"] = None
    d = cuda_inputs(host)
    out, hT, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, flags=F128)
    grads = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, res, d["dout"], None,
                              flags=F128)
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))
    host = make_inputs(w.with_(h0_std=0.2))
    d = cuda_inputs(host)
    leaves = {n: d[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "h0")}
    out, hT = gdn.gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                   leaves["h0"], flags=F128)
    (out.float() * d["dout"].float()).sum().backward(retain_graph=True)
    hT.backward(d["dh_final"])
    ref = oracle_bwd(host)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    for n, gn in names.items():
        assert rel(leaves[n].grad, ref[gn]) <= TOL["bf16"], (n, rel(leaves[n].grad, ref[gn]))


def test_many_heads_and_qk_l2norm_backward():
    """More (batch, head) pairs than SMs (the merge, mid-block and gradient grids span
    several waves, the gradients take their static stride), then the q/k L2
    normalisation through the backward (dq, dk with respect to the raw q, k)."""
    w = WORKLOADS["train_fwdbwd"].with_(B=4, T=256, H=48, h0_std=0.2)
    host = make_inputs(w)
    _, _, grads = _fwd_bwd(cuda_inputs(host))
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))
    w = WORKLOADS["train_fwdbwd"].with_(B=1, T=256, H=2, normalize_qk=False, h0_std=0.1)
    host = make_inputs(w)
    _, _, grads = _fwd_bwd(cuda_inputs(host), F128 | gdn.GDN_FLAG_QK_L2NORM)
    ref = oracle_bwd(host, qk_l2norm=True)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


def test_backward_agrees_with_64_token_chunks_and_is_deterministic():
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=512, H=4, h0_std=0.2)
    d = cuda_inputs(make_inputs(w))
    _, _, g1 = _fwd_bwd(d)
    _, _, g2 = _fwd_bwd(d)
    _, _, g0 = _fwd_bwd(d, 0)
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n
        x, y = g1[n].float(), g0[n].float()
        assert float((x - y).norm() / y.norm()) < 1e-2, n


def test_training_shape_fwd_bwd_workload():
    """B8 T4096 H6 D128 bf16 over 128-token chunks: every (batch, head) pair of out,
    h_final and every gradient against the oracle, per tensor and per pair (<= 2e-2)."""
    w = WORKLOADS["train_fwdbwd"]
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host))
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_fwd(host)
    ref = oracle_bwd(host)
    got = dict(grads, out=out, h_final=hT)
    refs = dict(ref, out=o_ref, h_final=h_ref)
    print("\nC=128 training shape B8 T4096 H6 D128 bf16, rel-L2 vs oracle (all 48 heads; worst pair):")
    for n in ("out", "h_final") + GRADS:
        state = n in ("h_final", "dh0")
        g = got[n].detach().double().cpu().numpy()
        y = refs[n]
        B, H = (g.shape[0], g.shape[1]) if state else (g.shape[0], g.shape[2])
        per = np.array([[np.linalg.norm((g[b, h] - y[b, h]) if state else (g[b, :, h] - y[b, :, h])) /
                         np.linalg.norm(y[b, h] if state else y[b, :, h]) for h in range(H)] for b in range(B)])
        whole = rel(got[n], refs[n])
        print(f"  {n:8s} {whole:.3e}  worst pair {per.max():.3e}")
        assert whole <= TOL["bf16"], (n, whole)
        assert per.max() <= TOL["bf16"], (n, per.max())


def test_cuda_graph_capture_of_a_training_step():
    """A fwd + bwd step over 128-token chunks captured in a CUDA graph replays to the same
    bits as the eager calls (every launch of the path on the caller's stream)."""
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=256, H=3, h0_std=0.2)
    d = cuda_inputs(make_inputs(w))
    dims = gdn.make_dims(d["q"], d["v"], d["g"], F128)
    res = torch.empty(gdn.gdn_chunk_residual_bytes(dims), dtype=torch.uint8, device="cuda")
    ws = torch.empty(gdn.gdn_chunk_bwd_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    out, hT = torch.empty_like(d["v"]), torch.empty_like(d["h0"])
    grads = {"dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"]),
             "dg": torch.empty_like(d["g"]), "dbeta": torch.empty_like(d["beta"]), "dh0": torch.empty_like(d["h0"])}

    def step():
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], out=out, h_final=hT, residuals=res,
                          flags=F128)
        gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res, d["dout"], d["dh_final"],
                          workspace=ws, grads=grads, flags=F128)

    step()
    torch.cuda.synchronize()
    eager = dict({n: t.clone() for n, t in grads.items()}, out=out.clone(), hT=hT.clone())
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in list(grads.values()) + [out, hT]:
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    got = dict(grads, out=out, hT=hT)
    for n, t in eager.items():
        assert torch.equal(got[n], t), n
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK


def test_long_context_shape():
    """B1 T32768 H16 D128 bf16 over 128-token chunks (256 steps per scan chain): out and
    h_final of every head, and every gradient of four heads, against the oracle."""
    w = WORKLOADS["long_context"]
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host))
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_fwd(host)
    print("\nC=128 long context: out %.3e h_final %.3e" % (rel(out, o_ref), rel(hT, h_ref)))
    assert rel(out, o_ref) <= TOL["bf16"] and rel(hT, h_ref) <= TOL["bf16"]
    pairs = [(0, 0), (0, 5), (0, 10), (0, 15)]
    ref = oracle_bwd(host, pairs)
    for n in GRADS:
        got = head_slice(grads[n].cpu(), pairs, state=(n == "dh0"))
        print("  %s %.3e" % (n, rel(got, ref[n])))
        assert rel(got, ref[n]) <= TOL["bf16"], (n, rel(got, ref[n]))
