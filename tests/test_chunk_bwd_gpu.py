"""GPU parity of the chunked backward (gdn_chunk_bwd) against the oracle's
hand-derived float64 reverse pass: rel-L2 <= 2e-2 per gradient with bf16 inputs,
1e-4 with fp32 inputs.

Also: a training step captured in a CUDA graph replays bitwise. Includes the
training-shape fwd+bwd workload (B8 T4096 H6 D128 bf16) at full
size with the same launch the benchmark times; the oracle checks every
(batch, head) pair there.
"""
import numpy as np
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


def _per_head_rel(got, ref, state=False):
    """rel-L2 of every (batch, head) pair: [B, T, H, ...] tensors ([B, H, ...] states)."""
    g = got.detach().double().cpu().numpy()
    B, H = (g.shape[0], g.shape[1]) if state else (g.shape[0], g.shape[2])
    out = np.zeros((B, H))
    for b in range(B):
        for h in range(H):
            x, y = (g[b, h], ref[b, h]) if state else (g[b, :, h], ref[b, :, h])
            out[b, h] = np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300)
    return out


def test_training_shape_fwd_bwd_workload():
    """B8 T4096 H6 D128 bf16: the benchmark's launch, every one of the 48 (batch, head)
    pairs against the oracle, element by element: rel-L2 <= 2e-2 per tensor over all
    elements and per pair. The measured margins are printed."""
    w = WORKLOADS["train_fwdbwd"]
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host))
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_fwd(host)
    ref = oracle_bwd(host)
    got = dict(grads, out=out, h_final=hT)
    refs = dict(ref, out=o_ref, h_final=h_ref)
    report = {}
    for n in ("out", "h_final") + GRADS:
        state = n in ("h_final", "dh0")
        whole = rel(got[n], refs[n])
        per = _per_head_rel(got[n], refs[n], state)
        report[n] = (whole, float(per.max()), tuple(int(i) for i in np.unravel_index(per.argmax(), per.shape)))
        assert whole <= TOL["bf16"], (n, whole)
        assert per.max() <= TOL["bf16"], (n, per.max(), report[n][2])
    print("\ntraining shape B8 T4096 H6 D128 bf16, rel-L2 vs oracle (all 48 heads; worst pair):")
    for n, (whole, worst, at) in report.items():
        print(f"  {n:8s} {whole:.3e}  worst pair {worst:.3e} at (b, h) = {at}")


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


def test_concurrent_backward_calls_on_two_streams():
    """The library owns no stream, event or lock: two backward calls on two streams at
    the same time (different problems, disjoint buffers) both match the oracle."""
    ws_ = [WORKLOADS["train_fwdbwd"].with_(B=2, T=1024, H=6, h0_std=0.2),
           WORKLOADS["train_fwdbwd"].with_(B=3, T=512, H=4, h0_std=0.1)]
    hosts = [make_inputs(w, seed=i) for i, w in enumerate(ws_)]
    ds = [cuda_inputs(h) for h in hosts]
    fwd = [gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"]) for d in ds]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    main = torch.cuda.current_stream()
    results = []
    for d, (out, hT, res), s in zip(ds, fwd, streams):
        s.wait_stream(main)
        with torch.cuda.stream(s):
            results.append(gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res,
                                             d["dout"], d["dh_final"]))
    torch.cuda.synchronize()
    for host, grads in zip(hosts, results):
        ref = oracle_bwd(host)
        for n in GRADS:
            assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("Dk,Dv", [(64, 128), (128, 64)])
def test_unequal_key_value_widths(per_channel, Dk, Dv):
    """Dk != Dv on the chunked path (the gated-deltanet kernel card, Requirements and
    limits, allows unequal key and value widths): forward and backward against the
    oracle, bf16 inputs."""
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=192, H=2, Dk=Dk, Dv=Dv, g_per_channel=per_channel,
                                        g_mult=1.0 if per_channel else 0.1, h0_std=0.3)
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host))
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out, o_ref) <= TOL["bf16"] and rel(hT, h_ref) <= TOL["bf16"]
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


def test_many_heads_two_launch_backward():
    """B*H = 160, at least the SM count: the reverse scan and the chunk-gradient kernel run
    as two launches (the single launch that runs them side by side needs SMs left over);
    every gradient of every head against the oracle."""
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=128, H=80, h0_std=0.2)
    host = make_inputs(w)
    _, _, grads = _fwd_bwd(cuda_inputs(host))
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["bf16"], (n, rel(grads[n], ref[n]))


def test_repeated_backward_reuses_workspace():
    """The single-launch backward's counters live in the workspace and start from zero on
    every call: three backward calls on one workspace give identical gradients."""
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=512, H=3, h0_std=0.2)
    d = cuda_inputs(make_inputs(w))
    out, hT, res = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    dims = gdn.make_dims(d["q"], d["v"], d["g"], 0)
    ws = torch.empty(gdn.gdn_chunk_bwd_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    runs = [gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], res, d["dout"],
                              d["dh_final"], workspace=ws) for _ in range(3)]
    for r in runs[1:]:
        for n in GRADS:
            assert torch.equal(r[n], runs[0][n]), n


# ------------------------------------------------------------------ fp32 operands
@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("Dk,Dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("flags", [0, gdn.GDN_FLAG_PAIRWISE_WITHIN_BLOCK])
def test_fp32_small_parity(per_channel, Dk, Dv, flags):
    """fp32 inputs through the CUDA-core backward chain (every width pair), rel-L2 <= 1e-4
    per gradient against the float64 oracle."""
    w = WORKLOADS["train_fwd_f32"].with_(B=2, T=192, H=2, Dk=Dk, Dv=Dv, g_per_channel=per_channel,
                                         g_mult=1.0 if per_channel else 0.1, h0_std=0.3)
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host), flags)
    assert grads["dq"].dtype == torch.float32
    ref = oracle_bwd(host)
    for n in GRADS:
        assert rel(grads[n], ref[n]) <= TOL["f32"], (n, rel(grads[n], ref[n]))


def test_fp32_extreme_decay_and_wipes():
    """fp32: strong per-channel decay (the pairwise in-block fallback) and a scalar decay
    with near-total wipes, each against the oracle at 1e-4."""
    for w in (WORKLOADS["train_fwd_f32"].with_(B=1, T=128, H=2, Dk=64, Dv=64, g_mu=3.0, g_mult=1.0,
                                               h0_std=0.5),
              WORKLOADS["recurrent"].with_(B=1, T=256, H=2, Dk=64, Dv=64, wipe_every=96)):
        host = make_inputs(w)
        _, _, grads = _fwd_bwd(cuda_inputs(host))
        ref = oracle_bwd(host)
        for n in GRADS:
            assert rel(grads[n], ref[n]) <= TOL["f32"], (w.name, n, rel(grads[n], ref[n]))


def test_fp32_autograd_and_qk_l2norm():
    """fp32 through the autograd wrapper, with and without the q/k L2 normalisation."""
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    for flags, norm in ((0, False), (gdn.GDN_FLAG_QK_L2NORM, True)):
        w = WORKLOADS["train_fwd_f32"].with_(B=1, T=128, H=2, h0_std=0.2, normalize_qk=not norm)
        host = make_inputs(w)
        d = cuda_inputs(host)
        leaves = {n: d[n].clone().requires_grad_(True) for n in names}
        out, hT = gdn.gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                       leaves["h0"], flags=flags)
        (out * d["dout"]).sum().backward(retain_graph=True)
        hT.backward(d["dh_final"])
        ref = oracle_bwd(host, qk_l2norm=norm)
        for n, gn in names.items():
            assert rel(leaves[n].grad, ref[gn]) <= TOL["f32"], (norm, n, rel(leaves[n].grad, ref[gn]))


def test_fp32_training_shape_slice():
    """B4 T4096 H6 D128 fp32 (the fp32 training shape): forward and backward at full size,
    every (batch, head) pair of the first two batches against the oracle at 1e-4."""
    w = WORKLOADS["train_fwd_f32"]
    host = make_inputs(w)
    out, hT, grads = _fwd_bwd(cuda_inputs(host))
    torch.cuda.synchronize()
    pairs = [(b, h) for b in range(2) for h in range(w.H)]
    ref = oracle_bwd(host, pairs)
    report = {}
    for n in GRADS:
        state = n == "dh0"
        got = head_slice(grads[n].cpu(), pairs, state=state)
        report[n] = rel(got, ref[n])
        assert report[n] <= TOL["f32"], (n, report[n])
    print("\nfp32 training shape B4 T4096 H6 D128, batches 0-1, rel-L2 vs oracle:")
    for n, r in report.items():
        print(f"  {n:8s} {r:.3e}")


def _graph_step_buffers(d):
    dims = gdn.make_dims(d["q"], d["v"], d["g"], 0)
    bufs = {
        "res": torch.empty(gdn.gdn_chunk_residual_bytes(dims), dtype=torch.uint8, device="cuda"),
        "ws": torch.empty(gdn.gdn_chunk_bwd_workspace_bytes(dims), dtype=torch.uint8, device="cuda"),
        "out": torch.empty_like(d["v"]),
        "hT": torch.empty((dims.B, dims.H, dims.Dk, dims.Dv), dtype=torch.float32, device="cuda"),
    }
    grads = {"dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"]),
             "dg": torch.empty_like(d["g"]), "dbeta": torch.empty_like(d["beta"]),
             "dh0": torch.empty((dims.B, dims.H, dims.Dk, dims.Dv), dtype=torch.float32, device="cuda")}
    return bufs, grads


@pytest.mark.parametrize("H", [3, 80])
def test_cuda_graph_capture_of_a_training_step(H):
    """A chunked fwd + bwd step captured in a CUDA graph replays to the same bits as the
    eager calls, twice: with B*H below the SM count (cooperative single launches,
    programmatic dependent launches and the counter-zeroing kernel inside the graph) and
    above it (split launches)."""
    w = WORKLOADS["train_fwdbwd"].with_(B=2, T=256, H=H, h0_std=0.2)
    d = cuda_inputs(make_inputs(w))
    bufs, grads = _graph_step_buffers(d)

    def step():
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], out=bufs["out"],
                          h_final=bufs["hT"], residuals=bufs["res"])
        gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], bufs["res"], d["dout"],
                          d["dh_final"], workspace=bufs["ws"], grads=grads)

    step()
    torch.cuda.synchronize()
    eager = {n: t.clone() for n, t in grads.items()}
    eager["out"], eager["hT"] = bufs["out"].clone(), bufs["hT"].clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        for t in list(grads.values()) + [bufs["out"], bufs["hT"]]:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        got = dict(grads, out=bufs["out"], hT=bufs["hT"])
        for n, t in eager.items():
            assert torch.equal(got[n], t), n
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK
