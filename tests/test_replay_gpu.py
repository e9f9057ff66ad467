"""GPU parity of replay decode (gdn_replay_decode / gdn_replay_state) against the oracle.

Replay decode keeps each head's state as a checkpoint plus a buffer of its last L
tokens (ReplaySSM summary, ai4snews "Gated DeltaNet" topic page). It computes the same
recurrence as the token-serial oracle, so every decoded output and the state the
buffer stands for are compared with the oracle's, over enough tokens to cross
several buffer folds. The fold shared by gdn_replay_state and a full step is checked
bitwise; so are a rollback of a rejected draft and the fill bookkeeping.
"""
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

from helpers import TOL, cuda_inputs, oracle_fwd, rel

pytestmark = pytest.mark.gpu


def _token(d, t, keys=("q", "k", "v", "g", "beta")):
    return [d[n][:, t:t + 1].contiguous() for n in keys]


def _decode(d, t0, t1, state, L, flags=0):
    ckpt, buffer, fill = state
    outs, fills = [], []
    for t in range(t0, t1):
        outs.append(gdn.gdn_replay_decode(*_token(d, t), ckpt, buffer, fill, L, flags=flags))
        fills.append(fill.clone())
    return torch.cat(outs, 1), fills


@pytest.mark.parametrize("L", [1, 5, 8])
@pytest.mark.parametrize("dtype,dims,per_channel", [("f32", (128, 128), True), ("f32", (64, 128), False),
                                                   ("bf16", (128, 64), True), ("bf16", (64, 64), False)])
def test_replay_decode_matches_oracle(L, dtype, dims, per_channel):
    T = 3 * L + 7 if L > 1 else 9
    w = WORKLOADS["tiny_fwd"].with_(B=2, T=T, H=3, Dk=dims[0], Dv=dims[1], dtype=dtype,
                                    g_per_channel=per_channel, h0_std=0.3)
    host = make_inputs(w)
    d = cuda_inputs(host)
    state = gdn.replay_init(d["h0"], L)
    out, fills = _decode(d, 0, T, state, L)
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out, o_ref) <= TOL[dtype]
    h = gdn.gdn_replay_state(*state, L)
    assert rel(h, h_ref) <= TOL["f32"]
    for t, f in enumerate(fills):  # the step that finds the buffer full folds it, then holds one token
        assert bool((f == (t % L) + 1).all()), t
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK


def test_replay_several_heads_per_cta():
    """B8 H48 (384 heads on at most 152 persistent CTAs, so each CTA runs its rings over
    two or three heads) over 20 tokens with L = 8: every head against the oracle."""
    L = 8
    w = WORKLOADS["recurrent"].with_(B=8, T=20, h0_std=0.01)
    host = make_inputs(w)
    d = cuda_inputs(host)
    state = gdn.replay_init(d["h0"], L)
    out, _ = _decode(d, 0, w.T, state, L)
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out, o_ref) <= TOL["f32"]
    assert rel(gdn.gdn_replay_state(*state, L), h_ref) <= TOL["f32"]
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK


def test_replay_state_is_the_next_checkpoint_bitwise():
    """gdn_replay_state of a full buffer == the checkpoint the next step folds and writes."""
    L = 8
    w = WORKLOADS["tiny_fwd"].with_(B=2, T=L + 1, H=4, Dk=128, Dv=128, h0_std=0.3)
    d = cuda_inputs(make_inputs(w))
    state = gdn.replay_init(d["h0"], L)
    _decode(d, 0, L, state, L)
    assert bool((state[2] == L).all())
    h = gdn.gdn_replay_state(*state, L)
    _decode(d, L, L + 1, state, L)
    assert torch.equal(state[0], h)
    # in place: the checkpoint becomes the full state when the caller then empties the buffer
    h2 = gdn.gdn_replay_state(*state, L)
    ck = state[0].clone()
    gdn.gdn_replay_state(*state, L, h_out=state[0])
    assert torch.equal(state[0], h2) and not torch.equal(ck, h2)


def test_replay_rollback_of_a_rejected_draft():
    """Decode 7 tokens, reject the last 3 (fill -= 3), decode 3 others: the outputs and the
    state are the oracle's for the accepted 4 tokens followed by the 3 new ones."""
    L = 8
    w = WORKLOADS["tiny_fwd"].with_(B=2, T=10, H=3, Dk=128, Dv=128, h0_std=0.3)
    host = make_inputs(w)
    d = cuda_inputs(host)
    state = gdn.replay_init(d["h0"], L)
    _decode(d, 0, 7, state, L)
    state[2].sub_(3)
    out_new, _ = _decode(d, 7, 10, state, L)
    keep = list(range(4)) + [7, 8, 9]
    host2 = {k: (v if v is None or k in ("h0", "dh_final") else v[:, keep].contiguous()) for k, v in host.items()}
    o_ref, h_ref = oracle_fwd(host2)
    assert rel(out_new, o_ref[:, 4:]) <= TOL["f32"]
    assert rel(gdn.gdn_replay_state(*state, L), h_ref) <= TOL["f32"]


def test_replay_scalar_decay_with_wipes_and_recurrent_agreement():
    """The scalar-decay decode geometry (B2 H48 Dk=Dv=128 fp32, g = logsigmoid(N(2,1)), a
    -20 wipe at token 255) over 300 tokens with L = 8: within 1e-4 of the oracle and of
    the token-recurrent decode of the same tokens."""
    L = 8
    w = WORKLOADS["recurrent"].with_(T=300, h0_std=0.01)
    host = make_inputs(w)
    d = cuda_inputs(host)
    state = gdn.replay_init(d["h0"], L)
    out, _ = _decode(d, 0, w.T, state, L)
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out, o_ref) <= TOL["f32"]
    h = gdn.gdn_replay_state(*state, L)
    assert rel(h, h_ref) <= TOL["f32"]
    o_rec, h_rec = gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    assert float((out - o_rec).norm() / o_rec.norm()) <= 1e-4
    assert float((h - h_rec).norm() / h_rec.norm()) <= 1e-4


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_replay_qk_l2norm(dtype):
    L = 6
    w = WORKLOADS["tiny_fwd"].with_(B=2, T=20, H=3, Dk=128, Dv=128, dtype=dtype, h0_std=0.3, normalize_qk=False)
    host = make_inputs(w)
    d = cuda_inputs(host)
    state = gdn.replay_init(d["h0"], L)
    out, _ = _decode(d, 0, w.T, state, L, flags=gdn.GDN_FLAG_QK_L2NORM)
    o_ref, h_ref = oracle_fwd(host, qk_l2norm=True)
    assert rel(out, o_ref) <= TOL[dtype]
    assert rel(gdn.gdn_replay_state(*state, L), h_ref) <= TOL["f32"]


def test_replay_fill_out_of_range_is_reported_and_clamped():
    """A fill above L is clamped by the kernel (the step folds L slots) and reported in the
    device error word; nothing outside the buffer is read."""
    L = 4
    w = WORKLOADS["tiny_fwd"].with_(B=1, T=L + 1, H=2, Dk=64, Dv=64, h0_std=0.3)
    d = cuda_inputs(make_inputs(w))
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK
    state = gdn.replay_init(d["h0"], L)
    _decode(d, 0, L, state, L)
    ref = [t.clone() for t in state]
    state[2].fill_(L + 5)
    out_bad, _ = _decode(d, L, L + 1, state, L)
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_ERR_INTERNAL
    out_ok, _ = _decode(d, L, L + 1, ref, L)
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK
    assert torch.equal(out_bad, out_ok) and torch.equal(state[0], ref[0])
