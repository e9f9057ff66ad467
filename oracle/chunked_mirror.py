"""Float64 restatement of the chunked (WY/UT) gated delta rule and its backward.

TEST INFRASTRUCTURE ONLY (see the package docstring). This is the algebra the
CUDA kernels follow, written plainly so that a test can pin it against the
token-serial oracle (``gdn_oracle.cpp``) to ~1e-12. It is never the reference
a GPU result is compared with.

Per chunk of C tokens (local index t = 0..C-1) with incoming state S0:

  G_t  = sum_{s<=t} g_s (per key channel)      Gam_t = exp(G_t),  gam = Gam_{C-1}
  Aqk[t,j] = sum_c q_tc k_jc exp(G_tc - G_jc)      j <= t
  Akk[t,j] = beta_t sum_c k_tc k_jc exp(G_tc - G_jc)   j < t
  T  = (I + Akk)^-1
  W  = T diag(beta) (Gam * k)       U' = T diag(beta) V
  U  = U' - W S0                    (the per-token deltas)
  O  = scale (Gam*q) S0 + scale Aqk U
  S1 = diag(gam) S0 + (exp(G_{C-1} - G) * k)^T U

Unrolling the token recurrence (decay, read, delta, write, read, as in the
"gated-deltanet" kernel card, section Method) gives exactly these equations.

Decay-weighted scores use the boundary-split factorisation of the
marin.community note "factoring GDN-2 decay on TPU", section Approach: the
chunk is cut into two consecutive blocks and the decay of a pair that spans
the cut is split at the last token of the first block, so each query row and
key row is scaled once and the cross-block tile is one product Q K^T.
``scores_factored`` uses that same split point as the reference for every row:
query rows are scaled by exp(G_t - G_b) and key rows by exp(G_b - G_j), so the
whole chunk is one masked product; factors across the cut are <= 1 and the
in-block factors are bounded by exp(decay spread of the block).
``scores_pairwise`` is the direct definition.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

CHUNK = 64
BLOCK = 32


def scores_pairwise(x: np.ndarray, y: np.ndarray, G: np.ndarray, inclusive: bool) -> np.ndarray:
    """P[t,j] = sum_c x_tc y_jc exp(G_tc - G_jc) for j <= t (j < t if not inclusive)."""
    C = x.shape[0]
    P = np.zeros((C, C))
    for t in range(C):
        for j in range(t + 1 if inclusive else t):
            P[t, j] = np.sum(x[t] * y[j] * np.exp(G[t] - G[j]))
    return P


def scores_factored(x: np.ndarray, y: np.ndarray, G: np.ndarray, inclusive: bool,
                    block: int = BLOCK) -> np.ndarray:
    """Same scores as ``scores_pairwise`` from one row-scaled product.

    b is the last token of the first block. Query rows are scaled by
    exp(G_t - G_b) (<= 1 in the second block, >= 1 in the first) and key rows by
    exp(G_b - G_j) (<= 1 in the first block, >= 1 in the second), so each pair
    gets exp(G_t - G_j); pairs across the cut use two factors <= 1."""
    C = x.shape[0]
    b = block - 1
    P = (x * np.exp(G - G[b])) @ (y * np.exp(G[b] - G)).T
    mask = np.tril(np.ones((C, C)), 0 if inclusive else -1)
    return P * mask


def boundary_split_factor(G_key: float, G_boundary: float, G_query: float) -> Tuple[float, float]:
    """(key-to-boundary factor, pair factor) for one channel of a cross-block pair."""
    key_factor = np.exp(G_boundary - G_key)
    return key_factor, np.exp(G_query - G_boundary) * key_factor


def score_backward(x, y, G, dP):
    """Gradients of P[t,j] = sum_c x_tc y_jc exp(G_tc - G_jc) (dP already masked).

    dx_t = sum_j dP[t,j] y_j E_tj,  dy_j = sum_t dP[t,j] x_t E_tj and, because
    each term depends on G through exp(G_t - G_j), dG = x*dx - y*dy."""
    C = x.shape[0]
    E = np.exp(G[:, None, :] - G[None, :, :])  # [t, j, c]
    Em = np.where(np.tril(np.ones((C, C)))[:, :, None] > 0, E, 0.0)
    dx = np.einsum("tj,jc,tjc->tc", dP, y, Em)
    dy = np.einsum("tj,tc,tjc->jc", dP, x, Em)
    return dx, dy, x * dx - y * dy


def chunk_local(q, k, v, g, beta, factored: bool = True, block: int = BLOCK) -> Dict[str, np.ndarray]:
    """Everything in one chunk that does not depend on the incoming state. ``block``
    is the length of the chunk's first block (the factored scores' split point)."""
    C = q.shape[0]
    G = np.cumsum(g, axis=0)
    Gam = np.exp(G)
    if factored:
        Pqk = scores_factored(q, k, G, True, block)
        Pkk = scores_factored(k, k, G, False, block)
    else:
        Pqk = scores_pairwise(q, k, G, True)
        Pkk = scores_pairwise(k, k, G, False)
    Akk = beta[:, None] * Pkk
    Tm = np.linalg.inv(np.eye(C) + Akk)
    Kh = Gam * k
    Bk = beta[:, None] * Kh
    Bv = beta[:, None] * v
    return dict(G=G, Gam=Gam, gam=Gam[-1], Qh=Gam * q, Kh=Kh, Kt=np.exp(G[-1] - G) * k,
                Aqk=Pqk, Pkk=Pkk, Akk=Akk, T=Tm, Bk=Bk, Bv=Bv, W=Tm @ Bk, Up=Tm @ Bv)


def _expand_g(g, Dk):
    return g if g.ndim == 4 else np.repeat(g[..., None], Dk, axis=-1)


def fwd(q, k, v, g, beta, h0=None, scale=None, chunk: int = CHUNK, factored: bool = True,
        block: Optional[int] = None):
    """Chunked forward. Returns (out, h_final, residual chunk-start states
    [B,H,N,Dk,Dv], per-chunk U [B,H,N,C,Dv])."""
    q, k, v, beta = (np.asarray(a, np.float64) for a in (q, k, v, beta))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    gx = _expand_g(np.asarray(g, np.float64), Dk)
    assert T % chunk == 0
    N = T // chunk
    scale = Dk ** -0.5 if scale is None else scale
    out = np.zeros((B, T, H, Dv))
    hT = np.zeros((B, H, Dk, Dv))
    states = np.zeros((B, H, N, Dk, Dv))
    Us = np.zeros((B, H, N, chunk, Dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((Dk, Dv)) if h0 is None else np.asarray(h0, np.float64)[b, h].copy()
            for n in range(N):
                sl = slice(n * chunk, (n + 1) * chunk)
                L = chunk_local(q[b, sl, h], k[b, sl, h], v[b, sl, h], gx[b, sl, h],
                                beta[b, sl, h], factored, chunk // 2 if block is None else block)
                states[b, h, n] = S
                U = L["Up"] - L["W"] @ S
                Us[b, h, n] = U
                out[b, sl, h] = scale * (L["Qh"] @ S + L["Aqk"] @ U)
                S = L["gam"][:, None] * S + L["Kt"].T @ U
            hT[b, h] = S
    return out, hT, states, Us


def fwd_transition(q, k, v, g, beta, h0=None, scale=None, chunk: int = CHUNK):
    """The same forward with the state recurrence written as one affine map per chunk,
        S1 = diag(gam) S0 + P S0 + C,   P = -K~^T W,   C = K~^T U',
    (substitute U = U' - W S0 into S1 = diag(gam) S0 + K~^T U), the outputs taken from the
    chunk-start states as before. A scan in this form has one product per chunk on its
    sequential chain instead of two. Returns (out, h_final)."""
    q, k, v, beta = (np.asarray(a, np.float64) for a in (q, k, v, beta))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    gx = _expand_g(np.asarray(g, np.float64), Dk)
    N = T // chunk
    scale = Dk ** -0.5 if scale is None else scale
    out = np.zeros((B, T, H, Dv))
    hT = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((Dk, Dv)) if h0 is None else np.asarray(h0, np.float64)[b, h].copy()
            for n in range(N):
                sl = slice(n * chunk, (n + 1) * chunk)
                L = chunk_local(q[b, sl, h], k[b, sl, h], v[b, sl, h], gx[b, sl, h], beta[b, sl, h], True,
                                chunk // 2)
                P = -L["Kt"].T @ L["W"]
                Cm = L["Kt"].T @ L["Up"]
                U = L["Up"] - L["W"] @ S
                out[b, sl, h] = scale * (L["Qh"] @ S + L["Aqk"] @ U)
                S = L["gam"][:, None] * S + P @ S + Cm
            hT[b, h] = S
    return out, hT


def chunk_grads(q, k, v, beta, L, S0, U, dO, dS1, dU, scale):
    """Chunk-parallel gradients of one chunk given the reverse scan's dU and the
    gradient dS1 of the state leaving the chunk. Returns dq, dk, dv, dG, dbeta
    (dG is the gradient of the chunk-local cumulative log-decay G).

    With Bk = diag(beta) K-hat, Bv = diag(beta) V, W = T Bk, U' = T Bv and
    U = U' - W S0 = T (Bv - Bk S0), the WY factors' gradients collapse:
      dT = dW Bk^T + dU Bv^T = dU ((I + Akk) U)^T, so with Y = T^T dU
      dBv = Y,  dBk = -Y S0^T,  dAkk = -(T^T dT T^T) = -Y U^T  (masked j < t).
    The score term of dbeta, sum_j dAkk[t,j] Pkk[t,j], equals sum_c k_tc dx'_tc
    where dx' is the x-side score gradient taken with dAkk itself."""
    C = q.shape[0]
    incl = np.tril(np.ones((C, C)))
    strict = np.tril(np.ones((C, C)), -1)
    G, Gam = L["G"], L["Gam"]
    dQh = scale * dO @ S0.T
    dAqk = scale * (dO @ U.T) * incl
    dKt = U @ dS1.T
    dgam = np.sum(dS1 * S0, axis=1)
    Y = L["T"].T @ dU
    dv = beta[:, None] * Y
    dBk = -Y @ S0.T
    dAkk = -(Y @ U.T) * strict
    dq_s, dk_s, dG_qk = score_backward(q, k, G, dAqk)
    dxb, dyb, _ = score_backward(k, k, G, dAkk)          # with dP = dAkk
    _, dyb_beta, _ = score_backward(beta[:, None] * k, k, G, dAkk)  # dy of dP = diag(beta) dAkk
    dKh = beta[:, None] * dBk
    dbeta = np.sum(Y * v, 1) + np.sum(dBk * L["Kh"], 1) + np.sum(k * dxb, 1)
    dx_kk = beta[:, None] * dxb
    dq = dQh * Gam + dq_s
    dk = dKh * Gam + dKt * np.exp(G[-1] - G) + dk_s + dx_kk + dyb_beta
    dG = (dQh * L["Qh"] + dKh * L["Kh"] - dKt * L["Kt"] + dG_qk
          + k * dx_kk - k * dyb_beta)
    dG[-1] += np.sum(dKt * L["Kt"], 0) + dgam * L["gam"]
    return dq, dk, dv, dG, dbeta


def bwd(q, k, v, g, beta, h0, dout, dh_final=None, scale=None, chunk: int = CHUNK, block: Optional[int] = None):
    """Chunked backward: reverse state scan plus chunk-parallel gradients."""
    q, k, v, beta, dout = (np.asarray(a, np.float64) for a in (q, k, v, beta, dout))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    per_channel = np.asarray(g).ndim == 4
    gx = _expand_g(np.asarray(g, np.float64), Dk)
    N = T // chunk
    scale = Dk ** -0.5 if scale is None else scale
    _, _, states, Us = fwd(q, k, v, g, beta, h0, scale, chunk)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dgx = np.zeros_like(gx)
    dbeta = np.zeros_like(beta)
    dh0 = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            dS = np.zeros((Dk, Dv)) if dh_final is None else np.asarray(dh_final, np.float64)[b, h].copy()
            for n in reversed(range(N)):
                sl = slice(n * chunk, (n + 1) * chunk)
                L = chunk_local(q[b, sl, h], k[b, sl, h], v[b, sl, h], gx[b, sl, h], beta[b, sl, h], True,
                                chunk // 2 if block is None else block)
                dO = dout[b, sl, h]
                dU = scale * L["Aqk"].T @ dO + L["Kt"] @ dS
                cq, ck, cv, cG, cb = chunk_grads(q[b, sl, h], k[b, sl, h], v[b, sl, h],
                                                 beta[b, sl, h], L, states[b, h, n], Us[b, h, n],
                                                 dO, dS, dU, scale)
                dq[b, sl, h], dk[b, sl, h], dv[b, sl, h], dbeta[b, sl, h] = cq, ck, cv, cb
                dgx[b, sl, h] = np.cumsum(cG[::-1], axis=0)[::-1]
                dS = L["gam"][:, None] * dS + scale * L["Qh"].T @ dO - L["W"].T @ dU
            dh0[b, h] = dS
    dg = dgx if per_channel else dgx.sum(-1)
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dh0=dh0)
