"""Shared test helpers: moving synthetic inputs to the GPU and to the oracle."""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Tuple

import numpy as np
import torch

import oracle
from gated_deltanet_gdn_gb300.synthetic import to_f64

TOL = {"f32": 1e-4, "bf16": 2e-2}


def cuda_inputs(d: Dict[str, Optional[torch.Tensor]]) -> Dict[str, Optional[torch.Tensor]]:
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


def head_slice(t: Optional[torch.Tensor], pairs: Iterable[Tuple[int, int]], state: bool = False):
    """Select (b, h) pairs as a [1, T, P, ...] problem ([1, P, ...] for states)."""
    if t is None:
        return None
    if state:
        return torch.stack([t[b, h] for b, h in pairs], 0)[None]
    return torch.stack([t[b, :, h] for b, h in pairs], 1)[None]


def oracle_fwd(d, pairs: Optional[List[Tuple[int, int]]] = None, scale=None, qk_l2norm: bool = False):
    """float64 oracle forward of the whole problem, or of the listed (b, h) pairs."""
    if pairs is None:
        args = [to_f64(d[n]) for n in ("q", "k", "v", "g", "beta", "h0")]
    else:
        args = [to_f64(head_slice(d[n], pairs, state=(n == "h0"))) for n in ("q", "k", "v", "g", "beta", "h0")]
    return oracle.fwd(*args, scale=scale, qk_l2norm=qk_l2norm)


def oracle_bwd(d, pairs: Optional[List[Tuple[int, int]]] = None, scale=None, qk_l2norm: bool = False):
    names = ("q", "k", "v", "g", "beta", "h0", "dout", "dh_final")
    if pairs is None:
        args = [to_f64(d[n]) for n in names]
    else:
        args = [to_f64(head_slice(d[n], pairs, state=(n in ("h0", "dh_final")))) for n in names]
    return oracle.bwd(*args, scale=scale, qk_l2norm=qk_l2norm)


def rel(x: torch.Tensor, y: np.ndarray) -> float:
    return oracle.rel_l2(x.detach().double().cpu().numpy(), y)
