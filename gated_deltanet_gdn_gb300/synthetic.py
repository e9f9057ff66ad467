"""Seeded synthetic inputs for the gated delta rule workloads.

This module draws random tensors and applies the input transforms that define
each workload (L2 normalisation of q and k, the -softplus / logsigmoid gates,
the sigmoid write gate, dtype rounding). It contains none of the recurrence's
arithmetic, so both the CUDA path and the float64 oracle can take their inputs
from here without sharing any of the method.

Draw order (fixed, on a CPU ``torch.Generator`` in float64):
q, k, v, g, beta, h0, dout, dh_final. Every workload draws all eight so that
the seed fixes every tensor independently of which outputs a test checks.

Workloads follow the shapes and distributions of the pages' benchmarks:
- marin.community "factoring GDN-2 decay on TPU", section Single-device
  benchmark: batches 4 and 8, 4096 tokens, 6 heads of width 128, FP32/BF16.
- "gated-deltanet" kernel card, sections Measured and Correctness: 48 heads,
  128 x 128 state, 2,048 tokens with periodic retention-gate wipes.
- atomic-ops 0.1.0, section Quick start: gates via -softplus (g <= 0),
  scale = d_head ** -0.5.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch
import torch.nn.functional as F

__all__ = ["Workload", "WORKLOADS", "make_inputs", "out_of_region_slice"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    Dk: int
    Dv: int
    dtype: str  # "f32" or "bf16": the type of q, k, v, g, beta, out and grads
    g_per_channel: bool
    g_kind: str  # "softplus" (g = -softplus(N(mu,1)) * mult) or "logsigmoid"
    g_mu: float = 0.0
    g_mult: float = 1.0
    wipe_every: int = 0  # scalar g only: tokens t with (t+1) % wipe_every == 0 get g = -20
    h0_std: float = 0.0  # 0: zero initial state
    normalize_qk: bool = True

    @property
    def scale(self) -> float:
        return float(self.Dk) ** -0.5

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the measurement plan, plus small parity cases built
# from them with ``with_``.
WORKLOADS: Dict[str, Workload] = {
    "tiny_fwd": Workload("tiny_fwd", B=1, T=128, H=2, Dk=64, Dv=64, dtype="f32",
                         g_per_channel=True, g_kind="softplus"),
    "recurrent": Workload("recurrent", B=2, T=2048, H=48, Dk=128, Dv=128, dtype="f32",
                          g_per_channel=False, g_kind="logsigmoid", g_mu=2.0,
                          wipe_every=256),
    "train_fwd_f32": Workload("train_fwd_f32", B=4, T=4096, H=6, Dk=128, Dv=128,
                              dtype="f32", g_per_channel=True, g_kind="softplus",
                              g_mult=0.1, h0_std=0.01),
    "train_fwd_bf16": Workload("train_fwd_bf16", B=4, T=4096, H=6, Dk=128, Dv=128,
                               dtype="bf16", g_per_channel=True, g_kind="softplus",
                               g_mult=0.1, h0_std=0.01),
    "train_fwdbwd": Workload("train_fwdbwd", B=8, T=4096, H=6, Dk=128, Dv=128,
                             dtype="bf16", g_per_channel=True, g_kind="softplus",
                             g_mult=0.1, h0_std=0.01),
    "long_context": Workload("long_context", B=1, T=32768, H=16, Dk=128, Dv=128,
                             dtype="bf16", g_per_channel=True, g_kind="softplus",
                             g_mu=-1.0, h0_std=0.01),
}


def _torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_inputs(w: Workload, seed: int = 0) -> Dict[str, torch.Tensor]:
    """Draw one workload's inputs on the CPU.

    Returns CPU tensors: q, k [B,T,H,Dk]; v [B,T,H,Dv]; g [B,T,H,Dk] or
    [B,T,H]; beta [B,T,H]; dout [B,T,H,Dv] in the workload dtype, and h0,
    dh_final [B,H,Dk,Dv] in float32 (h0 is None for a zero initial state).
    The oracle receives exactly these values, upcast to float64.
    """
    gen = torch.Generator().manual_seed(seed)
    f64 = torch.float64
    B, T, H, Dk, Dv = w.B, w.T, w.H, w.Dk, w.Dv

    def normal(*shape, mean=0.0, std=1.0):
        return torch.randn(*shape, generator=gen, dtype=f64) * std + mean

    q = normal(B, T, H, Dk)
    k = normal(B, T, H, Dk)
    v = normal(B, T, H, Dv)
    g_shape = (B, T, H, Dk) if w.g_per_channel else (B, T, H)
    g_raw = normal(*g_shape, mean=w.g_mu)
    beta_raw = normal(B, T, H)
    h0_raw = normal(B, H, Dk, Dv)
    dout = normal(B, T, H, Dv)
    dh_raw = normal(B, H, Dk, Dv)

    if w.normalize_qk:
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    if w.g_kind == "softplus":
        g = -F.softplus(g_raw) * w.g_mult
    elif w.g_kind == "logsigmoid":
        g = F.logsigmoid(g_raw) * w.g_mult
    else:
        raise ValueError(f"unknown gate recipe {w.g_kind}")
    if w.wipe_every:
        t_idx = torch.arange(T)
        wipe = ((t_idx + 1) % w.wipe_every) == 0
        if w.g_per_channel:
            g[:, wipe, :, :] = -20.0
        else:
            g[:, wipe, :] = -20.0
    beta = torch.sigmoid(beta_raw)

    dt = _torch_dtype(w.dtype)
    out = {
        "q": q.to(dt).contiguous(),
        "k": k.to(dt).contiguous(),
        "v": v.to(dt).contiguous(),
        "g": g.to(dt).contiguous(),
        "beta": beta.to(dt).contiguous(),
        "h0": (h0_raw * w.h0_std).to(torch.float32).contiguous() if w.h0_std > 0 else None,
        "dout": dout.to(dt).contiguous(),
        "dh_final": (dh_raw * 0.01).to(torch.float32).contiguous(),
    }
    return out


def out_of_region_slice(w: Workload, h0: torch.Tensor, seed: int = 1) -> Dict[str, torch.Tensor]:
    """The long-context workload's out-of-region slice: one 64-token chunk whose
    keys are N(0,1) draws WITHOUT L2 normalisation, so beta * |k|^2 is about
    beta * Dk, far above 2 (the regime where the "gated-deltanet" card,
    section Correctness, says the rule diverges). ``h0`` carries the state
    reached by the in-region run."""
    sl = w.with_(name=w.name + "_oor", B=h0.shape[0], T=64, H=h0.shape[1], normalize_qk=False,
                 h0_std=0.0)
    d = make_inputs(sl, seed=seed)
    # q keeps its normalisation so only the key magnitude leaves the stable region
    d["q"] = (d["q"].double() / d["q"].double().norm(dim=-1, keepdim=True)).to(d["q"].dtype)
    d["h0"] = h0.to(torch.float32).contiguous()
    return d


def to_f64(t: Optional[torch.Tensor]):
    """float64 numpy copy of a CPU tensor (None stays None)."""
    if t is None:
        return None
    return t.detach().to(torch.float64).cpu().numpy()
