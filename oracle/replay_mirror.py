"""Float64 restatement of replay decode: the gated delta rule's state held as a checkpoint
plus a buffer of the last few tokens.

TEST INFRASTRUCTURE ONLY (see the package docstring). This is the algebra the replay
decode kernel follows, written plainly so that a test can pin it against the
token-serial oracle (``gdn_oracle.cpp``) to ~1e-12. It is never the reference a GPU
result is compared with: the GPU tests compare replay decode with the oracle itself.

The representation follows the ReplaySSM summary on the ai4snews "Gated DeltaNet" topic
page (item "SSM decoding stops writing state every step"): a checkpoint S_c, written
only when the buffer of recent tokens is full, and outputs computed directly from the
checkpoint and the buffer. Unrolling the recurrence of the "gated-deltanet" kernel card
(section Method) from S_c over the buffered tokens j = 0..n, with G_j the log-decay summed
since the checkpoint (per key channel) and d_j = beta_j (v_j - S'_j^T k_j) each token's
delta, gives

  S_n = diag(exp(G_n)) S_c + sum_{j<=n} diag(exp(G_n - G_j)) k_j d_j^T

so token n needs only S_c and the buffer:

  d_n = beta_n (v_n - S_c^T (exp(G_n) k_n) - sum_{j<n} a_j d_j)
  o_n = scale (S_c^T (exp(G_n) q_n) + sum_{j<n} b_j d_j + (q_n . k_n) d_n)
  a_j = sum_c k_nc k_jc exp(G_nc - G_jc),   b_j = sum_c q_nc k_jc exp(G_nc - G_jc).

A step that finds the buffer full (fill == L) first folds it into the checkpoint with the
first formula (n = L - 1) and then treats its token as the buffer's first. Lowering
fill by r <= fill forgets the last r tokens (a rejected speculative draft).
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import numpy as np

Slot = Tuple[np.ndarray, np.ndarray, np.ndarray]  # k [Dk], G [Dk], d [Dv]


def fold(ckpt: np.ndarray, slots: List[Slot], n: int) -> np.ndarray:
    """The state the checkpoint and the first n slots stand for."""
    if n == 0:
        return ckpt.copy()
    G_last = slots[n - 1][1]
    S = np.exp(G_last)[:, None] * ckpt
    for k_j, G_j, d_j in slots[:n]:
        S = S + (np.exp(G_last - G_j) * k_j)[:, None] * d_j[None, :]
    return S


def step(ckpt: np.ndarray, slots: List[Slot], fill: int, L: int, q, k, v, g, beta: float,
         scale: float) -> Tuple[np.ndarray, np.ndarray, List[Slot], int]:
    """One decode step for one (batch, head). g is the token's log-decay per key channel.
    Returns (output, checkpoint, slots, fill) after the step."""
    if fill == L:
        ckpt = fold(ckpt, slots, L)
        fill = 0
    G_prev = slots[fill - 1][1] if fill > 0 else np.zeros_like(k)
    G_n = G_prev + g
    e = np.exp(G_n)
    x = ckpt.T @ (e * k)
    y = ckpt.T @ (e * q)
    for k_j, G_j, d_j in slots[:fill]:
        w = k_j * np.exp(G_n - G_j)
        x = x + np.dot(k, w) * d_j
        y = y + np.dot(q, w) * d_j
    d = beta * (v - x)
    o = scale * (y + np.dot(q, k) * d)
    slots = list(slots[:fill]) + [(k.copy(), G_n, d)]
    return o, ckpt, slots, fill + 1


def decode(q, k, v, g, beta, h0, L: int, scale: Optional[float] = None):
    """Token-by-token replay decode of [B, T, H, D] inputs (g [B,T,H,Dk] or [B,T,H]).
    Returns (outputs [B,T,H,Dv], the final full state [B,H,Dk,Dv], final fills [B,H])."""
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    scale = Dk ** -0.5 if scale is None else scale
    out = np.zeros((B, T, H, Dv))
    hT = np.zeros((B, H, Dk, Dv))
    fills = np.zeros((B, H), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            ckpt = np.zeros((Dk, Dv)) if h0 is None else np.array(h0[b, h], dtype=np.float64)
            slots: List[Slot] = []
            fill = 0
            for t in range(T):
                gt = g[b, t, h] if g.ndim == 4 else np.full(Dk, g[b, t, h])
                out[b, t, h], ckpt, slots, fill = step(ckpt, slots, fill, L, q[b, t, h], k[b, t, h], v[b, t, h],
                                                       gt, float(beta[b, t, h]), scale)
            hT[b, h] = fold(ckpt, slots, fill)
            fills[b, h] = fill
    return out, hT, fills
