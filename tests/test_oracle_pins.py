"""Pins of the float64 oracle against facts the pages and the mathematics fix.

None of these compares the oracle with itself: each pin is a worked example
printed on the pages, a closed form, a gate-semantics fact, an independent
formulation, or finite differences.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import chunked_mirror as cm
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs, to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def _arrays(w, seed=0):
    d = make_inputs(w, seed)
    return {k: to_f64(v) for k, v in d.items()}


def _rand_problem(rng, B=1, T=8, H=1, Dk=4, Dv=3, per_channel=True, h0=True, norm=True):
    q = rng.standard_normal((B, T, H, Dk))
    k = rng.standard_normal((B, T, H, Dk))
    if norm:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, Dv))
    gs = (B, T, H, Dk) if per_channel else (B, T, H)
    g = -np.log1p(np.exp(rng.standard_normal(gs)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    S0 = 0.3 * rng.standard_normal((B, H, Dk, Dv)) if h0 else None
    return q, k, v, g, beta, S0


def _read_golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                name, val = line.split()
                vals[name] = float(val)
    return vals


# ---------------------------------------------------------------- worked example

def test_worked_example_factor_routine():
    """marin note, section Approach: key at -1, boundary -2, queries -3/-4."""
    gold = _read_golden()
    for qn, pn in (("query_a", "pair_factor_query_a_log"), ("query_b", "pair_factor_query_b_log")):
        kf, pf = cm.boundary_split_factor(gold["key"], gold["boundary"], gold[qn])
        assert kf == pytest.approx(np.exp(gold["key_to_boundary_factor_log"]), rel=1e-15)
        assert pf == pytest.approx(np.exp(gold[pn]), rel=1e-15)


def test_worked_example_through_the_oracle():
    """One key written at cumulative log-decay -1 and read back by queries at
    -2 (the boundary), -3 and -4: the oracle's outputs are the printed factors."""
    gold = _read_golden()
    T = 4
    g = np.full((1, T, 1, 1), -1.0)  # G = -1, -2, -3, -4
    q = np.ones((1, T, 1, 1))
    k = np.ones((1, T, 1, 1))
    v = np.zeros((1, T, 1, 1))
    v[0, 0, 0, 0] = 1.0
    beta = np.zeros((1, T, 1))
    beta[0, 0, 0] = 1.0  # the only write is the key at token 0
    out, _ = oracle.fwd(q, k, v, g, beta, None, scale=1.0)
    o = out[0, :, 0, 0]
    assert np.cumsum(g[0, :, 0, 0])[0] == gold["key"]
    assert o[0] == pytest.approx(1.0, rel=1e-15)
    assert o[1] == pytest.approx(np.exp(gold["key_to_boundary_factor_log"]), rel=1e-14)
    assert o[2] == pytest.approx(np.exp(gold["pair_factor_query_a_log"]), rel=1e-14)
    assert o[3] == pytest.approx(np.exp(gold["pair_factor_query_b_log"]), rel=1e-14)


def test_factored_scores_equal_pairwise():
    """Boundary-split (and in-block reference) scores equal the pairwise definition."""
    rng = np.random.default_rng(3)
    for decay in (0.05, 0.8, 2.0):
        x = rng.standard_normal((64, 16))
        y = rng.standard_normal((64, 16))
        G = np.cumsum(-decay * rng.random((64, 16)), axis=0)
        for incl in (True, False):
            a = cm.scores_factored(x, y, G, incl)
            b = cm.scores_pairwise(x, y, G, incl)
            assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b)))


# ---------------------------------------------------------------- gate semantics

def test_beta_zero_leaves_state_decayed_only():
    """'gated-deltanet' card, section Correctness: beta = 0 leaves the state
    untouched by writes, so h_final = diag(exp(sum_t g_t)) h0."""
    rng = np.random.default_rng(0)
    for per_channel in (True, False):
        q, k, v, g, beta, S0 = _rand_problem(rng, B=2, T=19, H=3, Dk=5, Dv=4,
                                             per_channel=per_channel)
        beta[:] = 0.0
        _, hT = oracle.fwd(q, k, v, g, beta, S0)
        tot = g.sum(axis=1)  # [B,H,(Dk)]
        fac = np.exp(tot if per_channel else tot[..., None] * np.ones(5))
        np.testing.assert_allclose(hT, fac[..., None] * S0, rtol=1e-13, atol=0)


def test_identity_gate_is_exact():
    """g = 0 and beta = 0 is the exact identity (bitwise), and every output is
    the plain read scale * h0^T q_t."""
    rng = np.random.default_rng(1)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=2, T=7, H=2, Dk=6, Dv=5)
    g[:] = 0.0
    beta[:] = 0.0
    out, hT = oracle.fwd(q, k, v, g, beta, S0, scale=0.7)
    assert np.array_equal(hT, S0)
    want = 0.7 * np.einsum("bhcv,bthc->bthv", S0, q)
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-15)


def test_large_negative_g_wipes_the_state():
    """Card, section Correctness: a large negative g shrinks the state by nine
    orders of magnitude (exp(-20) = 2.06e-9). Two runs whose initial states
    differ by 1e3 agree after the wipe token to ~1e-9 relative."""
    rng = np.random.default_rng(2)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=1, T=40, H=2, Dk=8, Dv=8, per_channel=False)
    g[:] = -0.05
    g[:, 20] = -20.0
    out_a, _ = oracle.fwd(q, k, v, g, beta, 1e3 * S0)
    out_b, _ = oracle.fwd(q, k, v, g, beta, np.zeros_like(S0))
    before = np.linalg.norm(out_a[:, :20] - out_b[:, :20]) / np.linalg.norm(out_b[:, :20])
    after = np.linalg.norm(out_a[:, 21:] - out_b[:, 21:]) / np.linalg.norm(out_b[:, 21:])
    assert before > 1.0
    assert after < 1e3 * np.exp(-20.0) * 5 and after > 1e3 * np.exp(-20.0) * 1e-3


# ---------------------------------------------------------------- delta-rule closed forms

def test_delta_rule_recalls_the_written_value():
    """Card, section Method: with |k| = 1 and beta = 1 the write makes the state
    return v for key k, so writing the same key twice does not double it."""
    rng = np.random.default_rng(4)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=1, T=6, H=1, Dk=6, Dv=4)
    beta[:] = 1.0
    k[:, 3] = k[:, 2]  # same key twice
    v[:, 3] = v[:, 2]
    _, hT2 = oracle.fwd(q[:, :3], k[:, :3], v[:, :3], g[:, :3], beta[:, :3], S0)
    _, hT3 = oracle.fwd(q[:, :4], k[:, :4], v[:, :4], g[:, :4], beta[:, :4], S0)
    kk = k[0, 2, 0]
    np.testing.assert_allclose(kk @ hT2[0, 0], v[0, 2, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(kk @ hT3[0, 0], v[0, 2, 0], rtol=1e-12, atol=1e-12)


def test_delta_identity_for_any_key_norm_and_gate():
    """Card, section Method, in general: after the write, k_t^T S_t = (1 - beta |k|^2) k_t^T S'
    + beta |k|^2 v_t, where S' is the decayed previous state (unnormalised keys)."""
    rng = np.random.default_rng(14)
    for per_channel in (True, False):
        q, k, v, g, beta, S0 = _rand_problem(rng, B=1, T=7, H=1, Dk=5, Dv=3, per_channel=per_channel,
                                             norm=False)
        t = 6
        _, h_prev = oracle.fwd(q[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t], S0)
        _, h_t = oracle.fwd(q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], g[:, :t + 1], beta[:, :t + 1], S0)
        a = np.exp(g[0, t, 0]) * np.ones(5)
        S_dec = a[:, None] * h_prev[0, 0]
        kt, bt = k[0, t, 0], beta[0, t, 0]
        nk = float(kt @ kt)
        want = (1.0 - bt * nk) * (kt @ S_dec) + bt * nk * v[0, t, 0]
        np.testing.assert_allclose(kt @ h_t[0, 0], want, rtol=1e-12, atol=1e-12)


def test_householder_product_form():
    """Independent formulation: S_t = (I - beta k k^T) diag(exp g) S_{t-1} + beta k v^T,
    o_t = scale S_t^T q_t, evaluated with plain matrix products."""
    rng = np.random.default_rng(5)
    for per_channel in (True, False):
        q, k, v, g, beta, S0 = _rand_problem(rng, B=2, T=9, H=2, Dk=5, Dv=3,
                                             per_channel=per_channel, norm=False)
        out, hT = oracle.fwd(q, k, v, g, beta, S0, scale=0.4)
        for b in range(2):
            for h in range(2):
                S = S0[b, h].copy()
                for t in range(9):
                    a = np.exp(g[b, t, h]) * np.ones(5)
                    kt = k[b, t, h]
                    P = np.eye(5) - beta[b, t, h] * np.outer(kt, kt)
                    S = P @ np.diag(a) @ S + beta[b, t, h] * np.outer(kt, v[b, t, h])
                    np.testing.assert_allclose(out[b, t, h], 0.4 * S.T @ q[b, t, h], rtol=1e-12,
                                               atol=1e-13)
                np.testing.assert_allclose(hT[b, h], S, rtol=1e-12, atol=1e-13)


def test_divergence_closed_form():
    """Card, section Correctness: the rule is stable only while beta |k|^2 <= 2.
    With one repeated key, v = 0 and g = 0, the prediction k^T S follows
    p_t = (1 - beta |k|^2)^t p_0 exactly: it grows when beta |k|^2 > 2."""
    Dk, Dv, T = 4, 3, 30
    k1 = np.array([1.0, 2.0, -1.0, 0.5])
    s = float(k1 @ k1)  # 6.25
    beta_v = 0.5  # beta |k|^2 = 3.125 > 2
    k = np.tile(k1, (1, T, 1, 1))
    q = np.tile(k1, (1, T, 1, 1))
    v = np.zeros((1, T, 1, Dv))
    g = np.zeros((1, T, 1, Dk))
    beta = np.full((1, T, 1), beta_v)
    S0 = np.arange(Dk * Dv, dtype=float).reshape(1, 1, Dk, Dv) / 10.0
    out, hT = oracle.fwd(q, k, v, g, beta, S0, scale=1.0)
    p0 = k1 @ S0[0, 0]
    fac = 1.0 - beta_v * s
    for t in range(T):
        np.testing.assert_allclose(out[0, t, 0], fac ** (t + 1) * p0, rtol=1e-10)
    assert abs(fac) > 1.0 and np.linalg.norm(out[0, -1]) > 1e9 * np.linalg.norm(p0)


# ---------------------------------------------------------------- chunking invariants

def test_chunked_calls_equal_one_call_bitwise():
    """Card, section Correctness: a sequence in 16-token calls carrying the state
    equals one call; token by token equals the batched pass (float64, bitwise)."""
    rng = np.random.default_rng(6)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=2, T=96, H=2, Dk=8, Dv=6)
    out, hT = oracle.fwd(q, k, v, g, beta, S0)
    for step in (16, 1):
        S = S0
        outs = []
        for t0 in range(0, 96, step):
            sl = slice(t0, t0 + step)
            o, S = oracle.fwd(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], S)
            outs.append(o)
        assert np.array_equal(np.concatenate(outs, axis=1), out)
        assert np.array_equal(S, hT)


def test_heads_are_independent():
    """Slicing one (batch, head) out of a problem gives the same result alone."""
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=3, T=12, H=4, Dk=5, Dv=3)
    out, hT = oracle.fwd(q, k, v, g, beta, S0)
    b, h = 2, 1
    o1, h1 = oracle.fwd(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, h:h + 1], v[b:b + 1, :, h:h + 1],
                        g[b:b + 1, :, h:h + 1], beta[b:b + 1, :, h:h + 1], S0[b:b + 1, h:h + 1])
    assert np.array_equal(o1[0, :, 0], out[b, :, h])
    assert np.array_equal(h1[0, 0], hT[b, h])


# ---------------------------------------------------------------- reverse pass

def _loss(q, k, v, g, beta, S0, dO, dhT, scale):
    out, hT = oracle.fwd(q, k, v, g, beta, S0, scale=scale)
    return float(np.sum(out * dO) + np.sum(hT * dhT))


@pytest.mark.parametrize("per_channel", [True, False])
def test_reverse_pass_matches_finite_differences(per_channel):
    """Central differences (step 1e-6) of the float64 forward, every input element."""
    rng = np.random.default_rng(8 + per_channel)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=1, T=8, H=1, Dk=4, Dv=3,
                                         per_channel=per_channel, norm=False)
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(S0.shape)
    scale = 0.6
    grads = oracle.bwd(q, k, v, g, beta, S0, dO, dhT, scale=scale)
    inputs = dict(q=q, k=k, v=v, g=g, beta=beta, h0=S0)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    eps = 1e-6
    for name, arr in inputs.items():
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            orig = arr[idx]
            arr[idx] = orig + eps
            lp = _loss(**{**dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0), "dO": dO, "dhT": dhT,
                          "scale": scale})
            arr[idx] = orig - eps
            lm = _loss(**{**dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0), "dO": dO, "dhT": dhT,
                          "scale": scale})
            arr[idx] = orig
            fd[idx] = (lp - lm) / (2 * eps)
        an = grads[names[name]]
        err = np.linalg.norm(an - fd) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, (name, err)


def test_qk_l2norm_reverse_pass_matches_finite_differences():
    """With the q/k L2 normalisation, the gradients of q and k (taken back through the
    normalisation) match central differences of the normalised forward."""
    rng = np.random.default_rng(21)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=1, T=6, H=1, Dk=4, Dv=3, per_channel=True, norm=False)
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(S0.shape)
    grads = oracle.bwd(q, k, v, g, beta, S0, dO, dhT, scale=0.7, qk_l2norm=True)

    def loss():
        out, hT = oracle.fwd(q, k, v, g, beta, S0, scale=0.7, qk_l2norm=True)
        return float(np.sum(out * dO) + np.sum(hT * dhT))

    eps = 1e-6
    for arr, name in ((q, "dq"), (k, "dk"), (v, "dv"), (g, "dg"), (beta, "dbeta")):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            orig = arr[idx]
            arr[idx] = orig + eps
            lp = loss()
            arr[idx] = orig - eps
            lm = loss()
            arr[idx] = orig
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(grads[name] - fd) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, (name, err)


def test_qk_l2norm_is_scale_invariant_and_unit_rows_pass_through():
    """Scaling each q and k row by a positive factor does not change the normalised
    forward (up to the eps guard); rows that already have unit norm give the same
    result with or without the normalisation; a zero row stays zero."""
    rng = np.random.default_rng(22)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=1, T=20, H=2, Dk=8, Dv=5, per_channel=False, norm=False)
    o1, h1 = oracle.fwd(q, k, v, g, beta, S0, qk_l2norm=True)
    cq = rng.uniform(0.5, 3.0, q.shape[:-1] + (1,))
    ck = rng.uniform(0.5, 3.0, k.shape[:-1] + (1,))
    o2, h2 = oracle.fwd(q * cq, k * ck, v, g, beta, S0, qk_l2norm=True)
    assert oracle.rel_l2(o2, o1) < 1e-5 and oracle.rel_l2(h2, h1) < 1e-5
    qu = q / np.linalg.norm(q, axis=-1, keepdims=True)
    ku = k / np.linalg.norm(k, axis=-1, keepdims=True)
    o3, h3 = oracle.fwd(qu, ku, v, g, beta, S0)
    o4, h4 = oracle.fwd(qu, ku, v, g, beta, S0, qk_l2norm=True)
    assert oracle.rel_l2(o4, o3) < 1e-5 and oracle.rel_l2(h4, h3) < 1e-5
    z = np.zeros((2, 8))
    assert np.array_equal(oracle.l2norm(z), z)


def test_reverse_pass_chunk_split_consistency():
    """The reverse pass of a sequence equals the reverse passes of its two halves
    chained through dh (the segment checkpointing must not leak)."""
    rng = np.random.default_rng(10)
    q, k, v, g, beta, S0 = _rand_problem(rng, B=1, T=150, H=2, Dk=4, Dv=3)
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(S0.shape)
    full = oracle.bwd(q, k, v, g, beta, S0, dO, dhT)
    m = 70
    _, Sm = oracle.fwd(q[:, :m], k[:, :m], v[:, :m], g[:, :m], beta[:, :m], S0)
    second = oracle.bwd(q[:, m:], k[:, m:], v[:, m:], g[:, m:], beta[:, m:], Sm, dO[:, m:], dhT)
    first = oracle.bwd(q[:, :m], k[:, :m], v[:, :m], g[:, :m], beta[:, :m], S0, dO[:, :m],
                       second["dh0"])
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(np.concatenate([first[n], second[n]], axis=1), full[n],
                                   rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(first["dh0"], full["dh0"], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- the chunked algebra

@pytest.mark.parametrize("per_channel", [True, False])
def test_chunked_form_equals_token_serial(per_channel):
    """The WY/UT chunked form the kernels follow (forward and backward) equals
    the token-serial oracle on a two-chunk problem."""
    w = WORKLOADS["tiny_fwd"].with_(T=128, H=2, Dk=16, Dv=8, h0_std=0.5,
                                    g_per_channel=per_channel)
    a = _arrays(w)
    out, hT = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"])
    o2, h2, _, _ = cm.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"])
    assert oracle.rel_l2(o2, out) < 1e-12 and oracle.rel_l2(h2, hT) < 1e-12
    gr = oracle.bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["dout"], a["dh_final"])
    gm = cm.bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["dout"], a["dh_final"])
    for n in gr:
        assert oracle.rel_l2(gm[n], gr[n]) < 1e-11, n


@pytest.mark.parametrize("per_channel", [True, False])
def test_chunked_form_with_128_token_chunks_equals_token_serial(per_channel):
    """The same chunked form with 128-token chunks cut into two 64-token blocks (the
    marin note's 64 x 64 score tile, atomic-ops' bt = 2 bc), forward and backward, equals
    the token-serial oracle: the algebra a C = 128 kernel would follow."""
    w = WORKLOADS["tiny_fwd"].with_(T=256, H=1, Dk=8, Dv=6, h0_std=0.5, g_per_channel=per_channel)
    a = _arrays(w)
    out, hT = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"])
    o2, h2, _, _ = cm.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], chunk=128)
    assert oracle.rel_l2(o2, out) < 1e-12 and oracle.rel_l2(h2, hT) < 1e-12
    gr = oracle.bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["dout"], a["dh_final"])
    gm = cm.bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["dout"], a["dh_final"], chunk=128)
    for n in gr:
        assert oracle.rel_l2(gm[n], gr[n]) < 1e-10, n


@pytest.mark.parametrize("per_channel", [True, False])
def test_two_64_token_blocks_merge_into_one_128_token_chunk(per_channel):
    """The merge the 128-token forward performs, in float64: from each 64-token block's
    own chunk quantities (relative to the block's start) the 128-token chunk's follow as
    M = -W2 Kt1^T (= -T22 A21), W = [W1; W2 diag(gam1) - M W1], U' = [U'1; U'2 + M U'1],
    Qh = [Qh1; Qh2 diag(gam1)], Kt = [Kt1 diag(gam2); Kt2], gam = gam1 gam2 and
    Aqk = [[Aqk1, 0], [Qh2 Kt1^T, Aqk2]], equal to the direct 128-token chunk."""
    w = WORKLOADS["tiny_fwd"].with_(T=128, H=1, Dk=8, Dv=6, h0_std=0.5, g_per_channel=per_channel)
    a = _arrays(w)
    g = cm._expand_g(a["g"], 8)
    args = [a["q"][0, :, 0], a["k"][0, :, 0], a["v"][0, :, 0], g[0, :, 0], a["beta"][0, :, 0]]
    full = cm.chunk_local(*args, factored=False)
    b1 = cm.chunk_local(*[x[:64] for x in args], factored=False)
    b2 = cm.chunk_local(*[x[64:] for x in args], factored=False)
    M = -b2["W"] @ b1["Kt"].T
    # M is -T22 A21, A21 the cross-block rows 64.. x columns ..63 of the 128-token Akk
    assert np.allclose(M, -b2["T"] @ full["Akk"][64:, :64], rtol=0, atol=1e-12)
    want = dict(W=np.vstack([b1["W"], b2["W"] * b1["gam"] - M @ b1["W"]]),
                Up=np.vstack([b1["Up"], b2["Up"] + M @ b1["Up"]]),
                Qh=np.vstack([b1["Qh"], b2["Qh"] * b1["gam"]]),
                Kt=np.vstack([b1["Kt"] * b2["gam"], b2["Kt"]]),
                gam=b1["gam"] * b2["gam"])
    aqk = np.zeros((128, 128))
    aqk[:64, :64] = b1["Aqk"]
    aqk[64:, 64:] = b2["Aqk"]
    aqk[64:, :64] = b2["Qh"] @ b1["Kt"].T
    want["Aqk"] = aqk
    for n, x in want.items():
        assert oracle.rel_l2(x, full[n]) < 1e-12, n


def test_transition_matrix_form_equals_token_serial():
    """The chunk recurrence as one affine map, S1 = diag(gam) S0 - K~^T W S0 + K~^T U',
    equals the token-serial oracle (the alternative scan form of the next-steps list)."""
    w = WORKLOADS["tiny_fwd"].with_(T=192, H=2, Dk=8, Dv=6, h0_std=0.5)
    a = _arrays(w)
    out, hT = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"])
    o2, h2 = cm.fwd_transition(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"])
    assert oracle.rel_l2(o2, out) < 1e-12 and oracle.rel_l2(h2, hT) < 1e-12


def test_input_generator_recipe():
    """The generator follows the workload recipes (no method arithmetic)."""
    w = WORKLOADS["recurrent"].with_(B=1, T=512, H=2, Dk=8, Dv=8)
    d = make_inputs(w)
    g = d["g"].double()
    assert g.shape == (1, 512, 2)
    assert bool((g[:, 255] == -20).all()) and bool((g[:, 511] == -20).all())
    assert bool((g[:, 254] > -20).all()) and float(g.max()) <= 0.0
    n = d["k"].double().norm(dim=-1)
    assert float((n - 1).abs().max()) < 1e-6
    b = d["beta"].double()
    assert 0.0 < float(b.min()) and float(b.max()) < 1.0
    assert d["h0"] is None
    w2 = WORKLOADS["train_fwd_bf16"].with_(B=1, T=64, H=1)
    d2 = make_inputs(w2)
    assert d2["q"].dtype.is_floating_point and str(d2["q"].dtype) == "torch.bfloat16"
    assert d2["h0"].dtype == d2["dh_final"].dtype
    assert float(d2["g"].double().max()) <= 0.0


@pytest.mark.parametrize("L,per_channel", [(1, True), (3, True), (8, True), (5, False)])
def test_replay_form_equals_token_serial(L, per_channel):
    """The checkpoint + buffer form the replay decode kernel follows (outputs from reads
    of the checkpoint, lazy fold when the buffer is full) equals the token-serial oracle,
    across several folds and with a -20 wipe inside the buffer."""
    from oracle import replay_mirror as rm

    w = WORKLOADS["tiny_fwd"].with_(T=23, H=2, Dk=8, Dv=6, h0_std=0.5, g_per_channel=per_channel)
    a = _arrays(w)
    a["g"][:, 11] = -20.0  # a wipe while tokens are buffered
    out, hT = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"])
    o2, h2, fills = rm.decode(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], L)
    assert oracle.rel_l2(o2, out) < 1e-12 and oracle.rel_l2(h2, hT) < 1e-12
    assert (fills == (w.T - 1) % L + 1).all()


def test_replay_rollback_forgets_the_rejected_tokens():
    """Lowering the fill count by r forgets exactly the last r tokens: decoding 7 tokens,
    rolling back 3 and decoding 3 others equals the oracle on the accepted sequence."""
    from oracle import replay_mirror as rm

    w = WORKLOADS["tiny_fwd"].with_(T=10, H=1, Dk=8, Dv=6, h0_std=0.5)
    a = _arrays(w)
    scale = w.Dk ** -0.5
    ckpt, slots, fill, outs = a["h0"][0, 0].copy(), [], 0, []
    for t in list(range(7)) + [7, 8, 9]:
        if t == 7:
            fill -= 3  # tokens 4, 5, 6 rejected
        o, ckpt, slots, fill = rm.step(ckpt, slots, fill, 8, a["q"][0, t, 0], a["k"][0, t, 0], a["v"][0, t, 0],
                                       a["g"][0, t, 0], float(a["beta"][0, t, 0]), scale)
        outs.append(o)
    keep = [0, 1, 2, 3, 7, 8, 9]
    sub = {n: (a[n][:, keep] if a[n] is not None and n not in ("h0", "dh_final") else a[n]) for n in a}
    out, hT = oracle.fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], sub["h0"])
    assert oracle.rel_l2(np.stack(outs[7:]), out[0, 4:, 0]) < 1e-12
    assert oracle.rel_l2(rm.fold(ckpt, slots, fill), hT[0, 0]) < 1e-12
